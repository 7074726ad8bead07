// pa_device.cuh -- device-side building blocks for the sm_103a paged-attention
// kernels: mbarrier + 1-D bulk-copy (TMA) wrappers with bounded waits, element
// loads/conversions, and the per-device error word protocol.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <type_traits>
#include <stdint.h>

#include <utility>

#include "../../include/pa.h"

namespace pa {

// ---------------------------------------------------------------- error word
__device__ __forceinline__ void raise_error(unsigned* err, unsigned bit) {
  if (err) atomicOr(err, bit);
}

// ------------------------------------------------- device-scope ordering
// Release/acquire fence at GPU scope: before a relaxed atomic it publishes
// the stores ordered before it (also other threads' stores this thread has
// synchronised with); after one it orders later loads after what it saw.
__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ---------------------------------------------------------------- timers
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// A bounded wait gives up after this long (normal waits last microseconds).
constexpr uint64_t kWaitLimitNs = 200ull * 1000ull * 1000ull;

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete; false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}

// 1-D bulk asynchronous copy global -> shared, completion counted in bytes on
// an mbarrier of this CTA. Addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 2-D tensor copy global -> shared (TMA) of the box at element coordinates
// (x, y) of the tensor map, completion counted in bytes on an mbarrier of
// this CTA. `tmap` is the generic address of a tensor map held in kernel
// parameter space. x * element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// 2^x by the special-function unit (ex2.approx, flushing subnormal results
// to zero; 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------- tcgen05
// Fifth-generation tensor-core MMAs with accumulators in tensor memory
// (TMEM: 128 lanes x 512 columns of 32 bits per SM), issued by one thread,
// operands read from shared memory through 64-bit matrix descriptors.

// Allocate `ncols` TMEM columns (a power of two >= 32); the whole warp
// executes it and the base address lands in *dst (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Ordering of tcgen05 operations across a thread synchronisation.
__device__ __forceinline__ void tc05_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc05_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Writes to shared memory by ordinary stores, made visible to the tensor
// cores (the async proxy) before they read them.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Instruction descriptor of kind::f16 (fp32 accumulator): A and B both bf16
// (or both f16), A K-major, B K-major or MN-major, shape M x N.
__host__ __device__ constexpr uint32_t umma_idesc_f16(bool bf16, int M, int N, bool b_mn_major) {
  return (1u << 4)                                   // D format: f32
         | ((bf16 ? 1u : 0u) << 7)                   // A format
         | ((bf16 ? 1u : 0u) << 10)                  // B format
         | ((b_mn_major ? 1u : 0u) << 16)            // B major (A stays K-major)
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}
// Shared-memory matrix descriptor, 128-byte swizzle (atoms of 8 rows x 128
// bytes, 1024-byte aligned): start address, leading and stride byte offsets.
__device__ __forceinline__ uint64_t umma_sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// D (TMEM) [+]= A (smem) x B (smem), one thread.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}
// One arrival on `bar` once every MMA this thread issued before has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
// 32 consecutive 32-bit columns of this thread's TMEM lane (32x32b shape:
// warp w of a warpgroup reaches lanes 32w .. 32w + 31).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- warp MMA
// ldmatrix: four 8x8 matrices of 16-bit elements; lanes 8i .. 8i+7 give the
// row addresses of matrix i, and lane l receives row l/4, elements 2(l%4) and
// 2(l%4)+1 of each (the .trans form: column l/4, rows 2(l%4) and 2(l%4)+1).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <typename T>
struct Mma;
template <>
struct Mma<__nv_bfloat16> {
  __device__ __forceinline__ static void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  // two floats -> packed pair, lo in the low half (round to nearest even)
  __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
  }
  // sum of the two elements of a packed pair, in fp32 (exact widening)
  __device__ __forceinline__ static float sum2(uint32_t r) {
    return __uint_as_float(r << 16) + __uint_as_float(r & 0xFFFF0000u);
  }
};
template <>
struct Mma<__half> {
  __device__ __forceinline__ static void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
  }
  __device__ __forceinline__ static float sum2(uint32_t r) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&r));
    return f.x + f.y;
  }
};

// Programmatic dependent launch. pdl_wait() blocks until the grids this one
// depends on have completed and their writes are visible (a no-op when the
// launch had no programmatic dependency); every kernel calls it before its
// first global-memory access. pdl_trigger() lets the next grid in the stream
// be scheduled early (its CTAs then wait in their own pdl_wait()).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Named barrier over a subset of warps (id 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---------------------------------------------------------------- elements
template <typename T>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int bytes = 4;
  __device__ __forceinline__ static float to_f32(float x) { return x; }
  __device__ __forceinline__ static float from_f32(float x) { return x; }
};
template <>
struct Elem<__nv_bfloat16> {
  static constexpr int bytes = 2;
  __device__ __forceinline__ static float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
  __device__ __forceinline__ static __nv_bfloat16 from_f32(float x) { return __float2bfloat16_rn(x); }
};
template <>
struct Elem<__half> {
  static constexpr int bytes = 2;
  __device__ __forceinline__ static float to_f32(__half x) { return __half2float(x); }
  __device__ __forceinline__ static __half from_f32(float x) { return __float2half_rn(x); }
};
// FP8 E4M3 cache element (one byte).
struct E4M3 {};
template <>
struct Elem<E4M3> {
  static constexpr int bytes = 1;
};

// INT8 cache element (one two's-complement byte) with one fp32 scale per
// cached row, held beside the pages.
struct I8 {};
template <>
struct Elem<I8> {
  static constexpr int bytes = 1;
};

// Four INT8 codes (low byte first) -> two float pairs, exactly. Flipping a
// code's sign bit gives u = c + 128 in [0, 255]; the binary32 with bit
// pattern 0x4B0000uu is 2^23 + u, and subtracting 2^23 + 128 leaves c.
__device__ __forceinline__ void i8x4_to_float2x2(uint32_t w, float2* out) {
  const uint32_t u = w ^ 0x80808080u;
  const float2 bias = make_float2(-8388736.f, -8388736.f);
  out[0] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540)),
                                  __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7541))),
                      bias);
  out[1] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7542)),
                                  __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7543))),
                      bias);
}

// Two E4M3 codes (low byte first) -> two floats, via the hardware
// e4m3x2 -> f16x2 conversion (exact: every E4M3 value is an f16 value).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(two));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

// Widen a 32-bit word holding 32/(8*bytes) elements of CT into floats.
template <typename CT>
__device__ __forceinline__ void widen_word(uint32_t w, float* out);

template <>
__device__ __forceinline__ void widen_word<float>(uint32_t w, float* out) {
  out[0] = __uint_as_float(w);
}
template <>
__device__ __forceinline__ void widen_word<__nv_bfloat16>(uint32_t w, float* out) {
  out[0] = __uint_as_float(w << 16);
  out[1] = __uint_as_float(w & 0xFFFF0000u);
}
template <>
__device__ __forceinline__ void widen_word<__half>(uint32_t w, float* out) {
  __half2 h = *reinterpret_cast<__half2*>(&w);
  float2 f = __half22float2(h);
  out[0] = f.x;
  out[1] = f.y;
}
template <>
__device__ __forceinline__ void widen_word<E4M3>(uint32_t w, float* out) {
  float2 a = e4m3x2_to_float2(static_cast<uint16_t>(w & 0xFFFFu));
  float2 b = e4m3x2_to_float2(static_cast<uint16_t>(w >> 16));
  out[0] = a.x;
  out[1] = a.y;
  out[2] = b.x;
  out[3] = b.y;
}

// Load PB bytes (one "piece") from shared memory and widen its PB/bytes(CT)
// elements into out[]. PB in {1, 2, 4, 8, 16}; the address is PB-aligned.
template <typename CT, int PB>
__device__ __forceinline__ void load_piece(const uint8_t* p, float* out) {
  constexpr int EB = Elem<CT>::bytes;
  if constexpr (PB == 16) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    constexpr int E = 4 / EB;
    widen_word<CT>(v.x, out);
    widen_word<CT>(v.y, out + E);
    widen_word<CT>(v.z, out + 2 * E);
    widen_word<CT>(v.w, out + 3 * E);
  } else if constexpr (PB == 8) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    constexpr int E = 4 / EB;
    widen_word<CT>(v.x, out);
    widen_word<CT>(v.y, out + E);
  } else if constexpr (PB == 4) {
    widen_word<CT>(*reinterpret_cast<const uint32_t*>(p), out);
  } else if constexpr (PB == 2) {
    const uint16_t v = *reinterpret_cast<const uint16_t*>(p);
    if constexpr (EB == 2) {
      float tmp[2];
      widen_word<CT>(static_cast<uint32_t>(v), tmp);
      out[0] = tmp[0];
    } else {  // two E4M3 codes
      float2 f = e4m3x2_to_float2(v);
      out[0] = f.x;
      out[1] = f.y;
    }
  } else {  // PB == 1: one E4M3 code
    float2 f = e4m3x2_to_float2(static_cast<uint16_t>(*p));
    out[0] = f.x;
  }
}

// Load PB bytes (one "piece") from shared memory and widen its PB/bytes(CT)
// elements into PB/(2*bytes(CT)) float2 pairs (consecutive elements).
// PB in {2, 4, 8, 16} and PB >= 2*bytes(CT); the address is PB-aligned.
template <typename CT>
__device__ __forceinline__ void widen_word2(uint32_t w, float2* out);
template <>
__device__ __forceinline__ void widen_word2<__nv_bfloat16>(uint32_t w, float2* out) {
  out[0] = make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
template <>
__device__ __forceinline__ void widen_word2<__half>(uint32_t w, float2* out) {
  out[0] = __half22float2(*reinterpret_cast<__half2*>(&w));
}
template <>
__device__ __forceinline__ void widen_word2<E4M3>(uint32_t w, float2* out) {
  out[0] = e4m3x2_to_float2(static_cast<uint16_t>(w & 0xFFFFu));
  out[1] = e4m3x2_to_float2(static_cast<uint16_t>(w >> 16));
}
template <>
__device__ __forceinline__ void widen_word2<I8>(uint32_t w, float2* out) {
  i8x4_to_float2x2(w, out);
}

template <typename CT, int PB>
__device__ __forceinline__ void load_piece2(const uint8_t* p, float2* out) {
  constexpr int EB = Elem<CT>::bytes;
  static_assert(PB >= 2 * EB, "a piece must hold whole pairs");
  if constexpr (EB == 4) {  // float: pairs are already laid out
    if constexpr (PB == 16) {
      const float4 v = *reinterpret_cast<const float4*>(p);
      out[0] = make_float2(v.x, v.y);
      out[1] = make_float2(v.z, v.w);
    } else {
      out[0] = *reinterpret_cast<const float2*>(p);
    }
  } else {
    constexpr int P2W = 4 / (2 * EB);  // pairs per 32-bit word
    if constexpr (PB == 16) {
      const uint4 v = *reinterpret_cast<const uint4*>(p);
      widen_word2<CT>(v.x, out);
      widen_word2<CT>(v.y, out + P2W);
      widen_word2<CT>(v.z, out + 2 * P2W);
      widen_word2<CT>(v.w, out + 3 * P2W);
    } else if constexpr (PB == 8) {
      const uint2 v = *reinterpret_cast<const uint2*>(p);
      widen_word2<CT>(v.x, out);
      widen_word2<CT>(v.y, out + P2W);
    } else if constexpr (PB == 4) {
      widen_word2<CT>(*reinterpret_cast<const uint32_t*>(p), out);
    } else if constexpr (std::is_same<CT, I8>::value) {  // PB == 2: two INT8 codes
      float2 both[2];
      i8x4_to_float2x2(*reinterpret_cast<const uint16_t*>(p), both);
      out[0] = both[0];
    } else {  // PB == 2: two E4M3 codes
      out[0] = e4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(p));
    }
  }
}

// Four codes of w as two f16x2 words (bytes 0, 1 -> lo; bytes 2, 3 -> hi).
template <typename CT>
__device__ __forceinline__ void widen8(uint32_t w, uint32_t& lo, uint32_t& hi);
template <>
__device__ __forceinline__ void widen8<E4M3>(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l16, h16;\n\tmov.b32 {l16, h16}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l16;\n\tcvt.rn.f16x2.e4m3x2 %1, h16;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}
template <>
__device__ __forceinline__ void widen8<I8>(uint32_t w, uint32_t& lo, uint32_t& hi) {
  // u = c + 128 per byte; 0x6400 | u is the f16 1024 + u, exactly
  const uint32_t u = w ^ 0x80808080u;
  const __half2 bias = __floats2half2_rn(1152.f, 1152.f);
  uint32_t a = __byte_perm(u, 0x64646464u, 0x5140), b = __byte_perm(u, 0x64646464u, 0x7362);
  const __half2 x = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
  const __half2 y = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
  lo = *reinterpret_cast<const uint32_t*>(&x);
  hi = *reinterpret_cast<const uint32_t*>(&y);
}

// ---------------------------------------------------------------- FP8 encode
// E4M3 code of x (round to nearest even, finite saturation at +-448; NaN keeps
// its sign as 0x7F | sign).
__device__ __forceinline__ uint32_t e4m3x2_from_float2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  uint32_t out = r;
  if (isnan(lo)) out = (out & 0xFF00u) | 0x7Fu | (__float_as_uint(lo) >> 24 & 0x80u);
  if (isnan(hi)) out = (out & 0x00FFu) | ((0x7Fu | (__float_as_uint(hi) >> 24 & 0x80u)) << 8);
  return out;
}

// Launch `kern` on `stream` with a programmatic dependency on the previous
// work in the stream (see pdl_wait / pdl_trigger).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace pa
