// pa_decode_static.cu -- pa_decode_static_scratch: paged decode for callers that
// cannot allocate device memory.
//
// pa_decode needs a caller-provided workspace for the partial results of the
// contexts its persistent CTAs share. Some callers have no way to provide one:
// code embedded in a host application that owns every device allocation and
// exposes no allocator, or code that must not call cudaMalloc at all (its
// implicit synchronisation and unbounded latency are not acceptable where it
// runs). For them this entry point keeps those partials in a fixed array that
// the library itself carries in device memory, and otherwise runs exactly the
// kernels pa_decode runs.
#include <cuda_runtime.h>

#include "../../include/pa.h"

#define PA_API extern "C" __attribute__((visibility("default")))

namespace {

// Split partials of pa_decode_static_scratch. The CUDA runtime reserves it on
// a GPU when the library's device code is loaded there: with lazy module
// loading (the default) that happens at the first use of this code on that
// device -- the first launch of one of its kernels, or the first address
// lookup below -- not when the library is loaded into the process. It then
// stays reserved until the process exits.
static __device__ __align__(256) unsigned char g_static_scratch[PA_STATIC_SCRATCH_BYTES];

// In host code the array's name is only a host-side stand-in; the kernels must
// be given its device address, looked up on the device that is current (the
// one the stream belongs to). The lookup is repeated on every call, so the
// address stays right after the device's primary context has been reset and
// recreated; after the first call on a device it is a table lookup inside the
// runtime.
cudaError_t scratch_on_current_device(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
  if (e != cudaSuccess) return e;
  *out = p;
  return cudaSuccess;
}

}  // namespace

PA_API pa_status pa_decode_static_scratch(void* out, const void* query, const void* k_cache,
                                          const void* v_cache, const int32_t* block_tables,
                                          const int32_t* context_lens, int num_seqs,
                                          int num_heads, int num_kv_heads, int head_dim,
                                          int block_size, int num_blocks, int max_blocks_per_seq,
                                          float scale, int window, pa_dtype q_dtype,
                                          pa_kv_dtype kv_dtype, float k_scale, float v_scale,
                                          pa_stream_t stream) {
  const size_t need = pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim,
                                               block_size, max_blocks_per_seq, window);
  if (need > PA_STATIC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
  void* scratch = nullptr;
  size_t scratch_bytes = 0;
  if (need > 0) {
    if (scratch_on_current_device(&scratch) != cudaSuccess) return PA_ERR_CUDA;
    scratch_bytes = PA_STATIC_SCRATCH_BYTES;
  }
  // Nothing in the array has to start at zero: pa_decode clears the arrival
  // counters before its decode launch, and a partial slot is only read after
  // the launch that reads it has written it.
  return pa_decode(out, query, k_cache, v_cache, block_tables, context_lens, num_seqs, num_heads,
                   num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, scale,
                   window, q_dtype, kv_dtype, k_scale, v_scale, scratch, scratch_bytes, stream);
}
