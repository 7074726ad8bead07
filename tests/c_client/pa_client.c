/*
 * A plain C99 client of the library's C ABI (include/pa.h): no PyTorch, no
 * CUDA headers. It exercises the host-only entry points and the host-side
 * argument checks (which return before anything is enqueued), and prints one
 * "name value" line per check for the test that builds and runs it.
 */
#include <stdint.h>
#include <stdio.h>

#include "pa.h"

int main(void)
{
    int ns = 0, pps = 0;
    char fake[64];
    void* p = (void*)(((uintptr_t)fake + 15) & ~(uintptr_t)15); /* never dereferenced */

    printf("version %d\n", pa_version());
    printf("status_shape %s\n", pa_status_string(PA_ERR_SHAPE));
    printf("plan_rc %d\n", (int)pa_decode_plan(32, 32, 8, 128, 32, 128, 0, &ns, &pps));
    printf("plan_covers %d\n", ns * pps >= 128);
    printf("ws_g4_d128 %zu\n", pa_decode_workspace_size(32, 32, 8, 128, 32, 128, 0));
    printf("budget_mb %lld\n",
           (long long)pa_block_budget(PA_BUDGET_MB, 4096.0, 0, 32, 8, 128, 32, PA_BF16,
                                      PA_KV_AUTO));
    printf("budget_ctx %lld\n",
           (long long)pa_block_budget(PA_BUDGET_CONTEXT, 1024.0, 0, 32, 8, 128, 32, PA_BF16,
                                      PA_KV_AUTO));
    /* an empty batch is a no-op; bad sizes are refused on the host */
    printf("decode_empty %d\n",
           (int)pa_decode(NULL, NULL, NULL, NULL, NULL, NULL, 0, 32, 8, 128, 32, 10, 8, 0.1f, 0,
                          PA_BF16, PA_KV_AUTO, 1.f, 1.f, NULL, 0, NULL));
    printf("decode_head_dim %d\n",
           (int)pa_decode(p, p, p, p, (const int32_t*)p, (const int32_t*)p, 4, 32, 8, 80, 32, 10,
                          8, 0.1f, 0, PA_BF16, PA_KV_AUTO, 1.f, 1.f, NULL, 0, NULL));
    printf("decode_group %d\n",
           (int)pa_decode(p, p, p, p, (const int32_t*)p, (const int32_t*)p, 4, 30, 8, 128, 32, 10,
                          8, 0.1f, 0, PA_BF16, PA_KV_AUTO, 1.f, 1.f, NULL, 0, NULL));
    printf("write_null %d\n",
           (int)pa_reshape_and_cache(p, p, NULL, p, (const int64_t*)p, 4, 8, 128, 32, 10, PA_BF16,
                                     PA_KV_AUTO, 1.f, 1.f, NULL));
    printf("int8_f32_query %d\n",
           (int)pa_decode_int8(p, p, (const int8_t*)p, (const int8_t*)p, (const float*)p,
                               (const float*)p, (const int32_t*)p, (const int32_t*)p, 4, 8, 2,
                               128, 32, 10, 8, 0.1f, 0, PA_F32, NULL, 0, NULL));
    printf("prefill_fp8_scale %d\n",
           (int)pa_prefill_fp8(p, p, (const uint8_t*)p, (const uint8_t*)p, (const int32_t*)p,
                               (const int32_t*)p, (const int32_t*)p, 40, 4, 8, 2, 128, 32, 10, 8,
                               16, 0.1f, 0.f, 1.f, PA_BF16, NULL));
    printf("cascade_fp8_head_dim %d\n",
           (int)pa_decode_cascade_fp8(p, p, (const uint8_t*)p, (const uint8_t*)p,
                                      (const int32_t*)p, (const int32_t*)p, 4, 8, 2, 96, 32, 40,
                                      8, 0.1f, 1.f, 1.f, PA_BF16, 3, p, (size_t)1 << 30, NULL));
    printf("cascade_int8_null_scales %d\n",
           (int)pa_decode_cascade_int8(p, p, (const int8_t*)p, (const int8_t*)p, NULL, NULL,
                                       (const int32_t*)p, (const int32_t*)p, 4, 8, 2, 64, 16, 40,
                                       8, 0.1f, PA_F16, 3, p, (size_t)1 << 30, NULL));
    return 0;
}
