// pa_api.cu -- the C ABI of include/pa.h: host-side validation and planning,
// the small kernels (slot mapping, cache write, split reduction) and the
// per-device error word. The decode kernels live in pa_decode_<q>_<cache>.cu.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <cmath>
#include <mutex>

#include "pa_cascade.cuh"
#include "pa_decode.cuh"
#include "pa_device.cuh"

#define PA_API extern "C" __attribute__((visibility("default")))

namespace pa {

// ================================================================ error word
// One word per device; kernels OR PA_DEVERR_* bits into it, never trap.
__device__ unsigned g_error_word;

static std::mutex g_err_mu;
static unsigned* g_err_ptr[64];

// Device address of the current device's error word (NULL if unavailable).
static unsigned* error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (!g_err_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<unsigned*>(ptr);
  }
  return g_err_ptr[dev];
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int dtype_bytes(int dt) { return dt == PA_F32 ? 4 : 2; }

static bool valid_dtype(int dt) { return dt == PA_F32 || dt == PA_BF16 || dt == PA_F16; }

// GB300: the split plan is sized for its 152 SMs (fixed, so the plan is a
// pure function of the call's sizes and can be queried without a GPU).
constexpr int kPlanSMs = 152;
constexpr int kPlanCtasPerSM = 3;
constexpr int kPlanWaves = 4;
constexpr int kMinPagesPerSplit = 4;
constexpr int kMaxPagesPerSplit = 64;

static int group_bucket(int G) { return G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : 8; }

// ================================================================ kernels
// Zero fill of the balanced path's arrival counters. It waits for the
// previous kernel on the stream (which may be a decode still counting into
// them) and lets the next one launch early.
__global__ void clear_counters_kernel(int* counters, int n) {
  pdl_wait();
  pdl_trigger();
  for (int i = threadIdx.x; i < n; i += blockDim.x) counters[i] = 0;
}

// slot = block_tables[s][r / bs] * bs + r % bs, r = pos (mod W for a ring)
__global__ void slot_mapping_kernel(int64_t* out, const int32_t* block_tables,
                                    const int32_t* seq_idx, const int32_t* positions, int T,
                                    int S, int MB, int bs, int window, unsigned* err) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  const int pos = positions[t];
  const int s = seq_idx ? seq_idx[t] : t;
  if (pos < 0) {
    out[t] = -1;
    return;
  }
  const int r = window > 0 ? pos % window : pos;
  const int page = r / bs;
  if (s < 0 || s >= S || page >= MB) {
    out[t] = -1;
    raise_error(err, PA_DEVERR_SEQ);
    return;
  }
  out[t] = (int64_t)block_tables[(size_t)s * MB + page] * bs + r % bs;
}

// AUTO write: copy 16-byte chunks of each (token, kv head) row to its slot.
__global__ void cache_copy_kernel(const uint4* key, const uint4* value, uint4* k_cache,
                                  uint4* v_cache, const int64_t* slots, int T, int Hkv,
                                  int row_chunks, int bs, int64_t capacity, unsigned* err) {
  pdl_wait();
  pdl_trigger();
  const int64_t total = (int64_t)T * Hkv * row_chunks;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / row_chunks;  // t * Hkv + h
    const int ch = static_cast<int>(i - row * row_chunks);
    const int t = static_cast<int>(row / Hkv), h = static_cast<int>(row % Hkv);
    const int64_t slot = slots[t];
    if (slot < 0) continue;
    if (slot >= capacity) {
      if (h == 0 && ch == 0) raise_error(err, PA_DEVERR_SLOT);
      continue;
    }
    const int64_t blk = slot / bs, off = slot % bs;
    const int64_t dst = ((blk * Hkv + h) * bs + off) * row_chunks + ch;
    k_cache[dst] = key[i];
    v_cache[dst] = value[i];
  }
}

// FP8 write: 8 elements per thread, x / scale (IEEE binary32 division) then
// E4M3 round-to-nearest-even with finite saturation.
template <typename IT>
__global__ void cache_fp8_kernel(const IT* key, const IT* value, uint2* k_cache,
                                 uint2* v_cache, const int64_t* slots, int T, int Hkv,
                                 int row_chunks, int bs, int64_t capacity, float k_scale,
                                 float v_scale, unsigned* err) {
  pdl_wait();
  pdl_trigger();
  const int64_t total = (int64_t)T * Hkv * row_chunks;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / row_chunks;
    const int ch = static_cast<int>(i - row * row_chunks);
    const int t = static_cast<int>(row / Hkv), h = static_cast<int>(row % Hkv);
    const int64_t slot = slots[t];
    if (slot < 0) continue;
    if (slot >= capacity) {
      if (h == 0 && ch == 0) raise_error(err, PA_DEVERR_SLOT);
      continue;
    }
    const int64_t blk = slot / bs, off = slot % bs;
    const int64_t dst = ((blk * Hkv + h) * bs + off) * row_chunks + ch;
    float xk[8], xv[8];
    const IT* kp = key + i * 8;
    const IT* vp = value + i * 8;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      // a NaN input keeps its own sign (a NaN quotient's sign is unspecified)
      const float a = Elem<IT>::to_f32(kp[j]), b = Elem<IT>::to_f32(vp[j]);
      xk[j] = isnan(a) ? a : __fdiv_rn(a, k_scale);
      xv[j] = isnan(b) ? b : __fdiv_rn(b, v_scale);
    }
    uint2 ok, ov;
    ok.x = e4m3x2_from_float2(xk[0], xk[1]) | e4m3x2_from_float2(xk[2], xk[3]) << 16;
    ok.y = e4m3x2_from_float2(xk[4], xk[5]) | e4m3x2_from_float2(xk[6], xk[7]) << 16;
    ov.x = e4m3x2_from_float2(xv[0], xv[1]) | e4m3x2_from_float2(xv[2], xv[3]) << 16;
    ov.y = e4m3x2_from_float2(xv[4], xv[5]) | e4m3x2_from_float2(xv[6], xv[7]) << 16;
    k_cache[dst] = ok;
    v_cache[dst] = ov;
  }
}

// INT8 write: one warp per (token, kv head); lane i holds elements i, i + 32,
// ... of the row (at most E each). The row's max |x| is reduced across the
// warp, scale = max / 127 and code = rint(x / scale) clamped to +-127, both
// IEEE binary32 divisions; a zero scale stores zero codes.
template <typename IT, int E>
__device__ __forceinline__ void quantise_row_int8(const IT* x, int8_t* codes, float* scale_out,
                                                  int D, int lane) {
  float v[E];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const int d = lane + 32 * i;
    v[i] = d < D ? Elem<IT>::to_f32(x[d]) : 0.f;
    amax = fmaxf(amax, fabsf(v[i]));
  }
#pragma unroll
  for (int off = 16; off >= 1; off /= 2) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float scale = __fdiv_rn(amax, 127.f);
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const int d = lane + 32 * i;
    if (d < D) {
      const float r = scale == 0.f ? 0.f : fminf(fmaxf(rintf(__fdiv_rn(v[i], scale)), -127.f), 127.f);
      codes[d] = static_cast<int8_t>(__float2int_rz(r));
    }
  }
  if (lane == 0) *scale_out = scale;
}

template <typename IT, int E>
__global__ void cache_int8_kernel(const IT* key, const IT* value, int8_t* k_cache,
                                  int8_t* v_cache, float* k_scales, float* v_scales,
                                  const int64_t* slots, int T, int Hkv, int D, int bs,
                                  int64_t capacity, unsigned* err) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t wpb = blockDim.x >> 5;
  const int64_t total = (int64_t)T * Hkv;
  for (int64_t row = blockIdx.x * wpb + (threadIdx.x >> 5); row < total;
       row += (int64_t)gridDim.x * wpb) {
    const int t = static_cast<int>(row / Hkv), h = static_cast<int>(row % Hkv);
    const int64_t slot = slots[t];
    if (slot < 0) continue;
    if (slot >= capacity) {
      if (h == 0 && lane == 0) raise_error(err, PA_DEVERR_SLOT);
      continue;
    }
    const int64_t dst = (slot / bs * Hkv + h) * bs + slot % bs;  // row of the cache
    quantise_row_int8<IT, E>(key + row * D, k_cache + dst * D, k_scales + dst, D, lane);
    quantise_row_int8<IT, E>(value + row * D, v_cache + dst * D, v_scales + dst, D, lane);
  }
}

// LSE combination of split partials: one warp per (sequence, head) row; a
// lane owns the 4-float chunks lane, lane + 32, ... of the row. With at most
// kFewSplits splits every load of the row (each split's maximum, sum and
// chunks) is issued in one round; more splits take rounds of 8, lane j
// computing the weight of split j.
constexpr int kFewSplits = 8;
template <typename OT, int MAXC>
__global__ void __launch_bounds__(128)
    reduce_kernel(OT* out, const float* tmp_out, const float* max_logits, const float* exp_sums,
                  int64_t rows, int D, int NS) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t row = blockIdx.x * 4ll + (threadIdx.x >> 5);
  if (row >= rows) return;
  const float* ml = max_logits + row * NS;
  const float* es = exp_sums + row * NS;
  if (NS <= kFewSplits) {
    const int nchunk = D / 4;
    const float4* base = reinterpret_cast<const float4*>(tmp_out + row * NS * (int64_t)D);
    float mj[kFewSplits], lj[kFewSplits];
    float4 v[kFewSplits][MAXC];
#pragma unroll
    for (int j = 0; j < kFewSplits; ++j) {
      mj[j] = j < NS ? ml[j] : -INFINITY;
      lj[j] = j < NS ? es[j] : 0.f;
#pragma unroll
      for (int c = 0; c < MAXC; ++c) {
        const int d4 = lane + 32 * c;
        // an empty split's chunks may hold anything: loaded, never used
        v[j][c] = (j < NS && d4 < nchunk) ? base[(int64_t)j * nchunk + d4]
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int j = 0; j < kFewSplits; ++j)
      if (lj[j] > 0.f) M = fmaxf(M, mj[j]);
    OT* o = out + row * D;
    if (M == -INFINITY) {
      for (int d = lane; d < D; d += 32) o[d] = Elem<OT>::from_f32(0.f);
      return;
    }
    float4 acc[MAXC];
#pragma unroll
    for (int c = 0; c < MAXC; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
#pragma unroll
    for (int j = 0; j < kFewSplits; ++j) {
      if (lj[j] > 0.f) {
        const float w = lj[j] * expf(mj[j] - M);
        wsum += w;
#pragma unroll
        for (int c = 0; c < MAXC; ++c) {
          acc[c].x = fmaf(w, v[j][c].x, acc[c].x);
          acc[c].y = fmaf(w, v[j][c].y, acc[c].y);
          acc[c].z = fmaf(w, v[j][c].z, acc[c].z);
          acc[c].w = fmaf(w, v[j][c].w, acc[c].w);
        }
      }
    }
    const float inv = 1.f / wsum;
#pragma unroll
    for (int c = 0; c < MAXC; ++c) {
      const int d4 = lane + 32 * c;
      if (d4 < nchunk) {
        o[4 * d4 + 0] = Elem<OT>::from_f32(acc[c].x * inv);
        o[4 * d4 + 1] = Elem<OT>::from_f32(acc[c].y * inv);
        o[4 * d4 + 2] = Elem<OT>::from_f32(acc[c].z * inv);
        o[4 * d4 + 3] = Elem<OT>::from_f32(acc[c].w * inv);
      }
    }
    return;
  }
  float M = -INFINITY;
  for (int j = lane; j < NS; j += 32)
    if (es[j] > 0.f) M = fmaxf(M, ml[j]);
#pragma unroll
  for (int off = 16; off >= 1; off /= 2) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  OT* o = out + row * D;
  if (M == -INFINITY) {
    for (int d = lane; d < D; d += 32) o[d] = Elem<OT>::from_f32(0.f);
    return;
  }
  const int nchunk = D / 4;  // lane owns 4-float chunks lane, lane + 32, ...
  const float4* base = reinterpret_cast<const float4*>(tmp_out + row * NS * (int64_t)D);
  float4 a[MAXC];
#pragma unroll
  for (int c = 0; c < MAXC; ++c) a[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  for (int j0 = 0; j0 < NS; j0 += 32) {
    float wl = 0.f;  // weight of split j0 + lane (0 when empty or absent)
    if (j0 + lane < NS) {
      const float l = es[j0 + lane];
      if (l > 0.f) wl = l * expf(ml[j0 + lane] - M);
    }
    wsum += wl;
    const int cnt = min(32, NS - j0);
    for (int u0 = 0; u0 < cnt; u0 += 8) {
      float w[8];
      float4 v[8][MAXC];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        w[u] = __shfl_sync(0xffffffffu, wl, (u0 + u) & 31);
        const bool use = u0 + u < cnt && w[u] > 0.f;  // empty splits are never read
#pragma unroll
        for (int c = 0; c < MAXC; ++c) {
          const int d4 = lane + 32 * c;
          v[u][c] = (use && d4 < nchunk) ? base[(int64_t)(j0 + u0 + u) * nchunk + d4]
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
#pragma unroll
        for (int c = 0; c < MAXC; ++c) {
          a[c].x = fmaf(w[u], v[u][c].x, a[c].x);
          a[c].y = fmaf(w[u], v[u][c].y, a[c].y);
          a[c].z = fmaf(w[u], v[u][c].z, a[c].z);
          a[c].w = fmaf(w[u], v[u][c].w, a[c].w);
        }
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off /= 2) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
  const float inv = 1.f / wsum;
#pragma unroll
  for (int c = 0; c < MAXC; ++c) {
    const int d4 = lane + 32 * c;
    if (d4 < nchunk) {
      o[4 * d4 + 0] = Elem<OT>::from_f32(a[c].x * inv);
      o[4 * d4 + 1] = Elem<OT>::from_f32(a[c].y * inv);
      o[4 * d4 + 2] = Elem<OT>::from_f32(a[c].z * inv);
      o[4 * d4 + 3] = Elem<OT>::from_f32(a[c].w * inv);
    }
  }
}

static int grid_for(int64_t work, int threads) {
  int64_t b = (work + threads - 1) / threads;
  const int64_t cap = 152 * 16;
  return static_cast<int>(b < 1 ? 1 : (b > cap ? cap : b));
}

// ================================================================ validation
struct DecodeShape {
  int S, Hq, Hkv, D, bs, NB, MB, window;
  int q_dtype, kv_dtype;
  float k_scale, v_scale;
};

static pa_status check_decode(const DecodeShape& a, const void* out, const void* query,
                              const void* kc, const void* vc, const int32_t* bt,
                              const int32_t* cl) {
  if (a.S < 0 || a.S > 65535) return PA_ERR_SHAPE;
  if (a.S == 0) return PA_OK;
  if (!out || !query || !kc || !vc || !bt || !cl) return PA_ERR_NULL;
  if (!valid_dtype(a.q_dtype) || (a.kv_dtype != PA_KV_AUTO && a.kv_dtype != PA_KV_FP8_E4M3))
    return PA_ERR_DTYPE;
  if (a.Hq <= 0 || a.Hkv <= 0 || a.Hkv > 65535 || a.Hq % a.Hkv != 0 || a.Hq / a.Hkv > 8)
    return PA_ERR_SHAPE;
  if (a.D != 64 && a.D != 96 && a.D != 128) return PA_ERR_HEAD_DIM;
  if (a.bs != 16 && a.bs != 32 && a.bs != 64) return PA_ERR_BLOCK_SIZE;
  if (a.NB <= 0 || a.MB <= 0) return PA_ERR_SHAPE;
  if (a.window < 0 || (a.window > 0 && (a.window % a.bs != 0 || a.window / a.bs > a.MB)))
    return PA_ERR_WINDOW;
  if (a.kv_dtype == PA_KV_FP8_E4M3 &&
      !(isfinite(a.k_scale) && a.k_scale > 0.f && isfinite(a.v_scale) && a.v_scale > 0.f))
    return PA_ERR_SCALE;
  if (!aligned16(out) || !aligned16(query) || !aligned16(kc) || !aligned16(vc)) return PA_ERR_ALIGN;
  if (tma_staged(a.q_dtype, a.kv_dtype, a.D, group_bucket(a.Hq / a.Hkv), a.bs) &&
      (long long)a.NB * a.Hkv * a.bs > (1LL << 31) - 1)
    return PA_ERR_SHAPE;
  return PA_OK;
}

static int max_pages(int MB, int bs, int window) { return window > 0 ? window / bs : MB; }

static void plan(int S, int Hkv, int MB, int bs, int window, int* ns, int* pps) {
  const int64_t mp = max_pages(MB, bs, window);
  const int64_t units = (int64_t)S * Hkv;
  const int64_t target = (int64_t)kPlanSMs * kPlanCtasPerSM * kPlanWaves;
  int64_t p = (units * mp + target - 1) / target;
  if (p < kMinPagesPerSplit) p = kMinPagesPerSplit;
  if (p > kMaxPagesPerSplit) p = kMaxPagesPerSplit;
  int64_t n = (mp + p - 1) / p;
  if (n <= 1) {
    *ns = 1;
    *pps = static_cast<int>(mp);
    return;
  }
  p = (mp + n - 1) / n;  // even out the splits
  *ns = static_cast<int>(n);
  *pps = static_cast<int>(p);
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }


// ================================================================ tensor maps
// cuTensorMapEncodeTiled, reached through the runtime's driver entry point
// (nothing links against the driver library itself).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// The rows of a cache [NB * Hkv * bs][D] of 16-bit elements as a 2-D tensor
// map for the tensor-core decode: boxes of 64 elements x bs rows, 128-byte
// swizzle. Encodings are kept in a small ring keyed by (address, type, D,
// rows, bs), so steady-state calls on the same caches skip the encode.
struct TmapKey {
  const void* base;
  long long rows;
  int dtype, D, bs;
};
static std::mutex g_tmap_mu;
static constexpr int kTmapSlots = 16;
static TmapKey g_tmap_key[kTmapSlots];
static CUtensorMap g_tmap_val[kTmapSlots];
static int g_tmap_used = 0, g_tmap_next = 0;

// dtype: PA_BF16 / PA_F16 (16-bit elements, boxes of 64) or -1 (bytes, an
// FP8 or INT8 cache: boxes of 128).
static bool page_tensor_map(CUtensorMap* out, const void* base, int dtype, int D, long long rows,
                            int bs) {
  {
    std::lock_guard<std::mutex> lk(g_tmap_mu);
    for (int i = 0; i < g_tmap_used; ++i) {
      const TmapKey& k = g_tmap_key[i];
      if (k.base == base && k.rows == rows && k.dtype == dtype && k.D == D && k.bs == bs) {
        *out = g_tmap_val[i];
        return true;
      }
    }
  }
  const PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
  if (!fn) return false;
  const int eb = dtype < 0 ? 1 : 2;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * eb};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / eb), static_cast<cuuint32_t>(bs)};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType ty = dtype < 0         ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap m;
  if (fn(&m, ty, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> lk(g_tmap_mu);
  const int i = g_tmap_used < kTmapSlots ? g_tmap_used++ : g_tmap_next;
  g_tmap_next = (i + 1) % kTmapSlots;
  g_tmap_key[i] = TmapKey{base, rows, dtype, D, bs};
  g_tmap_val[i] = m;
  *out = m;
  return true;
}

// Most rows a cache read by the tensor-core decode may have: a row index is
// a 32-bit signed tensor coordinate.
constexpr long long kMaxTcRows = (1LL << 31) - 1;

static bool decode_is_tma_staged(const DecodeShape& a) {
  return tma_staged(a.q_dtype, a.kv_dtype, a.D, group_bucket(a.Hq / a.Hkv), a.bs);
}

static cudaError_t run_decode(const DecodeParams& prm_in, const DecodeShape& a, dim3 grid,
                              int mode, int* ctas, cudaStream_t st) {
  const int GT = group_bucket(a.Hq / a.Hkv);
  DecodeParams prm = prm_in;
  if (decode_is_tma_staged(a)) {
    const long long rows = (long long)a.NB * a.Hkv * a.bs;
    const int mt = a.kv_dtype == PA_KV_AUTO ? a.q_dtype : -1;
    if (rows > kMaxTcRows || !page_tensor_map(&prm.tm_k, prm.k_cache, mt, a.D, rows, a.bs) ||
        !page_tensor_map(&prm.tm_v, prm.v_cache, mt, a.D, rows, a.bs))
      return cudaErrorInvalidValue;
  }
  if (a.kv_dtype == PA_KV_AUTO) {
    switch (a.q_dtype) {
      case PA_F32: return pa_dispatch_decode_f32_f32(prm, grid, a.D, GT, a.bs, mode, ctas, st);
      case PA_BF16: return pa_dispatch_decode_bf16_bf16(prm, grid, a.D, GT, a.bs, mode, ctas, st);
      default: return pa_dispatch_decode_f16_f16(prm, grid, a.D, GT, a.bs, mode, ctas, st);
    }
  }
  if (a.kv_dtype == PA_KV_INT8) {
    return a.q_dtype == PA_BF16
               ? pa_dispatch_decode_bf16_i8(prm, grid, a.D, GT, a.bs, mode, ctas, st)
               : pa_dispatch_decode_f16_i8(prm, grid, a.D, GT, a.bs, mode, ctas, st);
  }
  switch (a.q_dtype) {
    case PA_F32: return pa_dispatch_decode_f32_e4m3(prm, grid, a.D, GT, a.bs, mode, ctas, st);
    case PA_BF16: return pa_dispatch_decode_bf16_e4m3(prm, grid, a.D, GT, a.bs, mode, ctas, st);
    default: return pa_dispatch_decode_f16_e4m3(prm, grid, a.D, GT, a.bs, mode, ctas, st);
  }
}

// Balanced-mode workspace: first the arrival counters (one int per possible
// decode CTA), then per decode CTA two partial slots of GT rows of D floats
// and their (max, sum) pairs. Only the counters need a known value (zero) at
// launch; pa_decode_workspace_clear sets them.
struct BalancedWs {
  int* arrived;
  float* piece_o;
  float* piece_ml;
};
static constexpr size_t kCounterBytes = (kMaxBalancedCtas * 4 + 255) / 256 * 256;
static_assert(kCounterBytes == 3840, "the header documents 3840 bytes of counters");
static size_t balanced_bytes(int GT, int D) {
  const size_t slots = (size_t)kMaxBalancedCtas * kPieceSlots;
  return kCounterBytes + align256(slots * GT * D * 4) + align256(slots * GT * 2 * 4);
}
static BalancedWs balanced_carve(void* ws, int GT, int D) {
  const size_t slots = (size_t)kMaxBalancedCtas * kPieceSlots;
  uint8_t* b = static_cast<uint8_t*>(ws);
  BalancedWs w;
  w.arrived = reinterpret_cast<int*>(b);
  b += kCounterBytes;
  w.piece_o = reinterpret_cast<float*>(b);
  b += align256(slots * GT * D * 4);
  w.piece_ml = reinterpret_cast<float*>(b);
  return w;
}

// Test hook of pa_test_set_unarmed_page (negative = off).
static std::atomic<int> g_unarmed_page{-1};

static DecodeParams make_params(const DecodeShape& a, const void* query, const void* kc,
                                const void* vc, const int32_t* bt, const int32_t* cl,
                                float scale, unsigned* err) {
  constexpr float kLog2e = 1.4426950408889634f;
  DecodeParams p{};
  p.unarmed_page = g_unarmed_page.load(std::memory_order_relaxed);
  p.query = query;
  p.k_cache = static_cast<const uint8_t*>(kc);
  p.v_cache = static_cast<const uint8_t*>(vc);
  p.block_tables = bt;
  p.context_lens = cl;
  p.err = err;
  p.num_seqs = a.S;
  p.num_heads = a.Hq;
  p.num_kv_heads = a.Hkv;
  p.group = a.Hq / a.Hkv;
  p.num_blocks = a.NB;
  p.max_blocks_per_seq = a.MB;
  p.window = a.window;
  const bool fp8 = a.kv_dtype == PA_KV_FP8_E4M3;
  p.q_scale = scale * kLog2e * (fp8 ? a.k_scale : 1.f);
  p.v_scale = fp8 ? a.v_scale : 1.f;
  return p;
}

static cudaError_t run_reduce(void* out, const float* tmp, const float* ml, const float* es,
                              int64_t rows, int D, int NS, int dt, cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>((rows + 3) / 4)), block(128);
  const int mc = (D + 127) / 128;  // float4 chunks per lane
#define PA_RED(OT, MC)                                                                      \
  return launch_pdl(reduce_kernel<OT, MC>, grid, block, 0, st, static_cast<OT*>(out), tmp, ml, \
                    es, rows, D, NS)
#define PA_RED_MC(OT)      \
  switch (mc) {            \
    case 1: PA_RED(OT, 1); \
    case 2: PA_RED(OT, 2); \
    case 3: PA_RED(OT, 3); \
    default: PA_RED(OT, 4); \
  }
  switch (dt) {
    case PA_F32: PA_RED_MC(float)
    case PA_BF16: PA_RED_MC(__nv_bfloat16)
    default: PA_RED_MC(__half)
  }
#undef PA_RED_MC
#undef PA_RED
}

}  // namespace pa

using namespace pa;

// ================================================================ C ABI
PA_API int pa_version(void) { return (1 << 16) | 0; }

PA_API const char* pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_NULL: return "a required pointer is NULL";
    case PA_ERR_DTYPE: return "unsupported element type or combination";
    case PA_ERR_SHAPE: return "inconsistent or unsupported sizes";
    case PA_ERR_HEAD_DIM: return "head_dim must be 64, 96 or 128";
    case PA_ERR_BLOCK_SIZE: return "block_size must be 16, 32 or 64";
    case PA_ERR_WINDOW: return "window must be >= 0, a multiple of block_size, and fit the block table";
    case PA_ERR_WORKSPACE: return "workspace too small for the split plan";
    case PA_ERR_CUDA: return "a CUDA runtime call failed";
    case PA_ERR_DEVICE: return "a kernel flagged out-of-range data (see the error bits)";
    case PA_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case PA_ERR_SCALE: return "FP8 scales must be finite and positive";
    default: return "unknown status";
  }
}

PA_API pa_status pa_slot_mapping(int64_t* slot_mapping, const int32_t* block_tables,
                                 const int32_t* seq_idx, const int32_t* positions,
                                 int num_tokens, int num_seqs, int max_blocks_per_seq,
                                 int block_size, int window, pa_stream_t stream) {
  if (num_tokens < 0 || num_seqs < 0) return PA_ERR_SHAPE;
  if (num_tokens == 0) return PA_OK;
  if (!slot_mapping || !block_tables || !positions) return PA_ERR_NULL;
  if (num_seqs <= 0 || max_blocks_per_seq <= 0) return PA_ERR_SHAPE;
  if (block_size <= 0) return PA_ERR_BLOCK_SIZE;
  if (window < 0 || (window > 0 && window % block_size != 0)) return PA_ERR_WINDOW;
  unsigned* err = error_word();
  const int threads = 256;
  const cudaError_t e = launch_pdl(
      slot_mapping_kernel, dim3((num_tokens + threads - 1) / threads), dim3(threads), 0,
      reinterpret_cast<cudaStream_t>(stream), slot_mapping, block_tables, seq_idx, positions,
      num_tokens, num_seqs, max_blocks_per_seq, block_size, window, err);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_API pa_status pa_reshape_and_cache(const void* key, const void* value, void* k_cache,
                                      void* v_cache, const int64_t* slot_mapping, int num_tokens,
                                      int num_kv_heads, int head_dim, int block_size,
                                      int num_blocks, pa_dtype in_dtype, pa_kv_dtype kv_dtype,
                                      float k_scale, float v_scale, pa_stream_t stream) {
  if (num_tokens < 0) return PA_ERR_SHAPE;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PA_ERR_NULL;
  if (!valid_dtype(in_dtype) || (kv_dtype != PA_KV_AUTO && kv_dtype != PA_KV_FP8_E4M3))
    return PA_ERR_DTYPE;
  if (num_kv_heads <= 0 || num_blocks <= 0) return PA_ERR_SHAPE;
  if (head_dim <= 0 || head_dim % 8 != 0 || head_dim > 1024) return PA_ERR_HEAD_DIM;
  if (block_size <= 0 || block_size > 1024) return PA_ERR_BLOCK_SIZE;
  if (kv_dtype == PA_KV_FP8_E4M3 &&
      !(isfinite(k_scale) && k_scale > 0.f && isfinite(v_scale) && v_scale > 0.f))
    return PA_ERR_SCALE;
  if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_ALIGN;
  unsigned* err = error_word();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int64_t capacity = (int64_t)num_blocks * block_size;
  const int threads = 256;
  cudaError_t e = cudaSuccess;
  if (kv_dtype == PA_KV_AUTO) {
    const int chunks = head_dim * dtype_bytes(in_dtype) / 16;
    const int64_t work = (int64_t)num_tokens * num_kv_heads * chunks;
    e = launch_pdl(cache_copy_kernel, dim3(grid_for(work, threads)), dim3(threads), 0, st,
                   static_cast<const uint4*>(key), static_cast<const uint4*>(value),
                   static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), slot_mapping,
                   num_tokens, num_kv_heads, chunks, block_size, capacity, err);
  } else {
    const int chunks = head_dim / 8;
    const int64_t work = (int64_t)num_tokens * num_kv_heads * chunks;
    const int grid = grid_for(work, threads);
    uint2* kc = static_cast<uint2*>(k_cache);
    uint2* vc = static_cast<uint2*>(v_cache);
    switch (in_dtype) {
      case PA_F32:
        e = launch_pdl(cache_fp8_kernel<float>, dim3(grid), dim3(threads), 0, st,
                       static_cast<const float*>(key), static_cast<const float*>(value), kc, vc,
                       slot_mapping, num_tokens, num_kv_heads, chunks, block_size, capacity,
                       k_scale, v_scale, err);
        break;
      case PA_BF16:
        e = launch_pdl(cache_fp8_kernel<__nv_bfloat16>, dim3(grid), dim3(threads), 0, st,
                       static_cast<const __nv_bfloat16*>(key),
                       static_cast<const __nv_bfloat16*>(value), kc, vc, slot_mapping, num_tokens,
                       num_kv_heads, chunks, block_size, capacity, k_scale, v_scale, err);
        break;
      default:
        e = launch_pdl(cache_fp8_kernel<__half>, dim3(grid), dim3(threads), 0, st,
                       static_cast<const __half*>(key), static_cast<const __half*>(value), kc, vc,
                       slot_mapping, num_tokens, num_kv_heads, chunks, block_size, capacity,
                       k_scale, v_scale, err);
    }
  }
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_API pa_status pa_decode_plan(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                int block_size, int max_blocks_per_seq, int window,
                                int* num_splits, int* pages_per_split) {
  (void)head_dim;
  if (!num_splits || !pages_per_split) return PA_ERR_NULL;
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || max_blocks_per_seq <= 0)
    return PA_ERR_SHAPE;
  if (block_size <= 0) return PA_ERR_BLOCK_SIZE;
  if (window < 0 || (window > 0 && window % block_size != 0)) return PA_ERR_WINDOW;
  plan(num_seqs, num_kv_heads, max_blocks_per_seq, block_size, window, num_splits,
       pages_per_split);
  return PA_OK;
}

PA_API size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads,
                                       int head_dim, int block_size, int max_blocks_per_seq,
                                       int window) {
  (void)num_seqs;
  (void)block_size;
  (void)max_blocks_per_seq;
  (void)window;
  if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || head_dim <= 0)
    return 0;
  return balanced_bytes(group_bucket(num_heads / num_kv_heads), head_dim);
}

PA_API pa_status pa_decode_partials(float* tmp_out, float* max_logits, float* exp_sums,
                                    const void* query, const void* k_cache, const void* v_cache,
                                    const int32_t* block_tables, const int32_t* context_lens,
                                    int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                    int block_size, int num_blocks, int max_blocks_per_seq,
                                    float scale, int window, pa_dtype q_dtype,
                                    pa_kv_dtype kv_dtype, float k_scale, float v_scale,
                                    int num_splits, int pages_per_split, pa_stream_t stream) {
  DecodeShape a{num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                max_blocks_per_seq, window, q_dtype, kv_dtype, k_scale, v_scale};
  pa_status rc = check_decode(a, tmp_out, query, k_cache, v_cache, block_tables, context_lens);
  if (rc != PA_OK || num_seqs == 0) return rc;
  if (!max_logits || !exp_sums) return PA_ERR_NULL;
  if (num_splits < 1 || pages_per_split < 1 || num_splits > 65535 ||
      (int64_t)num_splits * pages_per_split < max_pages(max_blocks_per_seq, block_size, window))
    return PA_ERR_SHAPE;
  DecodeParams p = make_params(a, query, k_cache, v_cache, block_tables, context_lens, scale,
                               error_word());
  p.tmp_out = tmp_out;
  p.max_logits = max_logits;
  p.exp_sums = exp_sums;
  p.partials = 1;
  p.num_splits = num_splits;
  p.pages_per_split = pages_per_split;
  const dim3 grid(num_splits, num_kv_heads, num_seqs);
  return run_decode(p, a, grid, kModeSplit, nullptr, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

PA_API pa_status pa_reduce(void* out, const float* tmp_out, const float* max_logits,
                           const float* exp_sums, int num_seqs, int num_heads, int head_dim,
                           int num_splits, pa_dtype out_dtype, pa_stream_t stream) {
  if (num_seqs < 0 || num_heads < 0) return PA_ERR_SHAPE;
  if (num_seqs == 0 || num_heads == 0) return PA_OK;
  if (!out || !tmp_out || !max_logits || !exp_sums) return PA_ERR_NULL;
  if (!valid_dtype(out_dtype)) return PA_ERR_DTYPE;
  if (head_dim <= 0 || head_dim % 4 != 0 || head_dim > 512) return PA_ERR_HEAD_DIM;
  if (num_splits < 1) return PA_ERR_SHAPE;
  if (!aligned16(tmp_out)) return PA_ERR_ALIGN;
  return run_reduce(out, tmp_out, max_logits, exp_sums, (int64_t)num_seqs * num_heads, head_dim,
                    num_splits, out_dtype, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

PA_API pa_status pa_decode_balanced(void* out, const void* query, const void* k_cache,
                                    const void* v_cache, const int32_t* block_tables,
                                    const int32_t* context_lens, int num_seqs, int num_heads,
                                    int num_kv_heads, int head_dim, int block_size,
                                    int num_blocks, int max_blocks_per_seq, float scale,
                                    int window, pa_dtype q_dtype, pa_kv_dtype kv_dtype,
                                    float k_scale, float v_scale, void* workspace,
                                    size_t workspace_bytes, int* num_ctas, pa_stream_t stream) {
  if (num_ctas) *num_ctas = 0;
  DecodeShape a{num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                max_blocks_per_seq, window, q_dtype, kv_dtype, k_scale, v_scale};
  pa_status rc = check_decode(a, out, query, k_cache, v_cache, block_tables, context_lens);
  if (rc != PA_OK || num_seqs == 0) return rc;
  if (!workspace || !num_ctas) return PA_ERR_NULL;
  const int GT = group_bucket(num_heads / num_kv_heads);
  if (workspace_bytes < balanced_bytes(GT, head_dim)) return PA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return PA_ERR_ALIGN;
  DecodeParams p = make_params(a, query, k_cache, v_cache, block_tables, context_lens, scale,
                               error_word());
  const BalancedWs w = balanced_carve(workspace, GT, head_dim);
  p.out = out;
  p.piece_o = w.piece_o;
  p.piece_ml = w.piece_ml;
  p.arrived = w.arrived;
  p.num_splits = 1;
  p.pages_per_split = 1;
  int ctas = 0;
  if (run_decode(p, a, dim3(0, 1, 1), kModeBalanced, &ctas, reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  *num_ctas = ctas;
  return PA_OK;
}

PA_API pa_status pa_decode_workspace_clear(void* workspace, size_t workspace_bytes,
                                           pa_stream_t stream) {
  if (!workspace) return PA_ERR_NULL;
  if (workspace_bytes < kCounterBytes) return PA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return PA_ERR_ALIGN;
  return launch_pdl(clear_counters_kernel, dim3(1), dim3(256), 0,
                    reinterpret_cast<cudaStream_t>(stream), static_cast<int*>(workspace),
                    static_cast<int>(kCounterBytes / 4)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

PA_API pa_status pa_decode(void* out, const void* query, const void* k_cache,
                           const void* v_cache, const int32_t* block_tables,
                           const int32_t* context_lens, int num_seqs, int num_heads,
                           int num_kv_heads, int head_dim, int block_size, int num_blocks,
                           int max_blocks_per_seq, float scale, int window, pa_dtype q_dtype,
                           pa_kv_dtype kv_dtype, float k_scale, float v_scale, void* workspace,
                           size_t workspace_bytes, pa_stream_t stream) {
  DecodeShape a{num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                max_blocks_per_seq, window, q_dtype, kv_dtype, k_scale, v_scale};
  pa_status rc = check_decode(a, out, query, k_cache, v_cache, block_tables, context_lens);
  if (rc != PA_OK || num_seqs == 0) return rc;
  const int GT = group_bucket(num_heads / num_kv_heads);
  if (workspace && workspace_bytes >= balanced_bytes(GT, head_dim) && aligned16(workspace)) {
    int ctas = 0;
    rc = pa_decode_workspace_clear(workspace, workspace_bytes, stream);
    if (rc != PA_OK) return rc;
    return pa_decode_balanced(out, query, k_cache, v_cache, block_tables, context_lens, num_seqs,
                              num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                              max_blocks_per_seq, scale, window, q_dtype, kv_dtype, k_scale,
                              v_scale, workspace, workspace_bytes, &ctas, stream);
  }
  // no usable workspace: one CTA per (sequence, kv head), straight to the output
  DecodeParams p = make_params(a, query, k_cache, v_cache, block_tables, context_lens, scale,
                               error_word());
  p.out = out;
  p.partials = 0;
  p.num_splits = 1;
  p.pages_per_split = max_pages(max_blocks_per_seq, block_size, window);
  return run_decode(p, a, dim3(1, num_kv_heads, num_seqs), kModeSplit, nullptr,
                    reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

// ================================================================ INT8 cache
PA_API pa_status pa_reshape_and_cache_int8(const void* key, const void* value, int8_t* k_cache,
                                           int8_t* v_cache, float* k_scales, float* v_scales,
                                           const int64_t* slot_mapping, int num_tokens,
                                           int num_kv_heads, int head_dim, int block_size,
                                           int num_blocks, pa_dtype in_dtype, pa_stream_t stream) {
  if (num_tokens < 0) return PA_ERR_SHAPE;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !k_cache || !v_cache || !k_scales || !v_scales || !slot_mapping)
    return PA_ERR_NULL;
  if (!valid_dtype(in_dtype)) return PA_ERR_DTYPE;
  if (num_kv_heads <= 0 || num_blocks <= 0) return PA_ERR_SHAPE;
  if (head_dim <= 0 || head_dim % 8 != 0 || head_dim > 256) return PA_ERR_HEAD_DIM;
  if (block_size <= 0 || block_size > 1024) return PA_ERR_BLOCK_SIZE;
  if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(k_scales) || !aligned16(v_scales))
    return PA_ERR_ALIGN;
  unsigned* err = error_word();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int64_t capacity = (int64_t)num_blocks * block_size;
  const int threads = 256;
  const int grid = grid_for((int64_t)num_tokens * num_kv_heads * 32, threads);
#define PA_I8W(IT, E)                                                                         \
  launch_pdl(cache_int8_kernel<IT, E>, dim3(grid), dim3(threads), 0, st,                      \
             static_cast<const IT*>(key), static_cast<const IT*>(value), k_cache, v_cache,     \
             k_scales, v_scales, slot_mapping, num_tokens, num_kv_heads, head_dim, block_size, \
             capacity, err)
#define PA_I8W_E(IT) \
  (head_dim <= 64 ? PA_I8W(IT, 2) : head_dim <= 128 ? PA_I8W(IT, 4) : PA_I8W(IT, 8))
  cudaError_t e;
  switch (in_dtype) {
    case PA_F32: e = PA_I8W_E(float); break;
    case PA_BF16: e = PA_I8W_E(__nv_bfloat16); break;
    default: e = PA_I8W_E(__half);
  }
#undef PA_I8W_E
#undef PA_I8W
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_API pa_status pa_decode_int8(void* out, const void* query, const int8_t* k_cache,
                                const int8_t* v_cache, const float* k_scales,
                                const float* v_scales, const int32_t* block_tables,
                                const int32_t* context_lens, int num_seqs, int num_heads,
                                int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                int max_blocks_per_seq, float scale, int window,
                                pa_dtype q_dtype, void* workspace, size_t workspace_bytes,
                                pa_stream_t stream) {
  // the shared checks, on the shape with a native cache
  DecodeShape a{num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                max_blocks_per_seq, window, q_dtype, PA_KV_AUTO, 1.f, 1.f};
  pa_status rc = check_decode(a, out, query, k_cache, v_cache, block_tables, context_lens);
  if (rc != PA_OK || num_seqs == 0) return rc;
  if (q_dtype != PA_BF16 && q_dtype != PA_F16) return PA_ERR_DTYPE;
  if (!k_scales || !v_scales) return PA_ERR_NULL;
  if (!aligned16(k_scales) || !aligned16(v_scales)) return PA_ERR_ALIGN;
  a.kv_dtype = PA_KV_INT8;
  DecodeParams p = make_params(a, query, k_cache, v_cache, block_tables, context_lens, scale,
                               error_word());
  p.k_scales = k_scales;
  p.v_scales = v_scales;
  p.out = out;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int GT = group_bucket(num_heads / num_kv_heads);
  if (workspace && workspace_bytes >= balanced_bytes(GT, head_dim) && aligned16(workspace)) {
    rc = pa_decode_workspace_clear(workspace, workspace_bytes, stream);
    if (rc != PA_OK) return rc;
    const BalancedWs w = balanced_carve(workspace, GT, head_dim);
    p.piece_o = w.piece_o;
    p.piece_ml = w.piece_ml;
    p.arrived = w.arrived;
    p.num_splits = 1;
    p.pages_per_split = 1;
    int ctas = 0;
    return run_decode(p, a, dim3(0, 1, 1), kModeBalanced, &ctas, st) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
  }
  // no usable workspace: one CTA per (sequence, kv head), straight to the output
  p.partials = 0;
  p.num_splits = 1;
  p.pages_per_split = max_pages(max_blocks_per_seq, block_size, window);
  return run_decode(p, a, dim3(1, num_kv_heads, num_seqs), kModeSplit, nullptr, st) ==
                 cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

// ================================================================ prefill
PA_API pa_status pa_prefill(void* out, const void* query, const void* k_cache,
                            const void* v_cache, const int32_t* block_tables,
                            const int32_t* cu_q, const int32_t* context_lens, int num_tokens,
                            int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                            int block_size, int num_blocks, int max_blocks_per_seq,
                            int max_q_len, float scale, pa_dtype q_dtype, pa_stream_t stream) {
  if (num_tokens < 0 || num_seqs < 0 || num_seqs > 65535) return PA_ERR_SHAPE;
  if (num_tokens == 0 || num_seqs == 0) return PA_OK;
  if (!out || !query || !k_cache || !v_cache || !block_tables || !cu_q || !context_lens)
    return PA_ERR_NULL;
  if (q_dtype != PA_BF16 && q_dtype != PA_F16) return PA_ERR_DTYPE;
  if (num_heads <= 0 || num_kv_heads <= 0 || num_kv_heads > 65535 ||
      num_heads % num_kv_heads != 0 || num_heads / num_kv_heads > 8)
    return PA_ERR_SHAPE;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_HEAD_DIM;
  if (block_size != 16 && block_size != 32 && block_size != 64) return PA_ERR_BLOCK_SIZE;
  if (num_blocks <= 0 || max_blocks_per_seq <= 0 || max_q_len < 1 || max_q_len > num_tokens)
    return PA_ERR_SHAPE;
  if ((int64_t)max_blocks_per_seq * block_size > INT32_MAX) return PA_ERR_SHAPE;
  // pages are staged by tensor copies: 32-bit row coordinates
  const long long cache_rows = (long long)num_blocks * num_kv_heads * block_size;
  if (cache_rows > kMaxTcRows) return PA_ERR_SHAPE;
  if (!aligned16(out) || !aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_ALIGN;
  constexpr float kLog2e = 1.4426950408889634f;
  PrefillParams p{};
  if (!page_tensor_map(&p.tm_k, k_cache, q_dtype, head_dim, cache_rows, block_size) ||
      !page_tensor_map(&p.tm_v, v_cache, q_dtype, head_dim, cache_rows, block_size))
    return PA_ERR_CUDA;
  p.out = out;
  p.query = query;
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.block_tables = block_tables;
  p.cu_q = cu_q;
  p.context_lens = context_lens;
  p.err = error_word();
  p.num_seqs = num_seqs;
  p.num_heads = num_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_heads / num_kv_heads;
  p.head_dim = head_dim;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.num_tokens = num_tokens;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.max_q_len = max_q_len;
  p.scale_log2 = scale * kLog2e;
  return launch_prefill_attention(p, q_dtype, 0, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

// Prefill over an 8-bit cache: kind 1 = INT8 codes with row scales
// (k_scales, v_scales), kind 2 = FP8 E4M3 codes (k_scale, v_scale).
static pa_status prefill_8bit(int kind, void* out, const void* query, const void* k_cache,
                              const void* v_cache, const float* k_scales, const float* v_scales,
                              float k_scale, float v_scale, const int32_t* block_tables,
                              const int32_t* cu_q, const int32_t* context_lens, int num_tokens,
                              int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                              int block_size, int num_blocks, int max_blocks_per_seq,
                              int max_q_len, float scale, pa_dtype q_dtype, pa_stream_t stream) {
  if (num_tokens < 0 || num_seqs < 0 || num_seqs > 65535) return PA_ERR_SHAPE;
  if (num_tokens == 0 || num_seqs == 0) return PA_OK;
  if (!out || !query || !k_cache || !v_cache || !block_tables || !cu_q || !context_lens ||
      (kind == 1 && (!k_scales || !v_scales)))
    return PA_ERR_NULL;
  if (q_dtype != PA_BF16 && q_dtype != PA_F16) return PA_ERR_DTYPE;
  if (num_heads <= 0 || num_kv_heads <= 0 || num_kv_heads > 65535 ||
      num_heads % num_kv_heads != 0 || num_heads / num_kv_heads > 8)
    return PA_ERR_SHAPE;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_HEAD_DIM;
  if (block_size != 16 && block_size != 32 && block_size != 64) return PA_ERR_BLOCK_SIZE;
  if (num_blocks <= 0 || max_blocks_per_seq <= 0 || max_q_len < 1 || max_q_len > num_tokens)
    return PA_ERR_SHAPE;
  if ((int64_t)max_blocks_per_seq * block_size > INT32_MAX) return PA_ERR_SHAPE;
  if (kind == 2 && !(isfinite(k_scale) && k_scale > 0.f && isfinite(v_scale) && v_scale > 0.f))
    return PA_ERR_SCALE;
  if (!aligned16(out) || !aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (kind == 1 && (!aligned16(k_scales) || !aligned16(v_scales))))
    return PA_ERR_ALIGN;
  constexpr float kLog2e = 1.4426950408889634f;
  PrefillParams p{};
  p.out = out;
  p.query = query;
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.k_scales = k_scales;
  p.v_scales = v_scales;
  p.block_tables = block_tables;
  p.cu_q = cu_q;
  p.context_lens = context_lens;
  p.err = error_word();
  p.num_seqs = num_seqs;
  p.num_heads = num_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_heads / num_kv_heads;
  p.head_dim = head_dim;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.num_tokens = num_tokens;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.max_q_len = max_q_len;
  p.scale_log2 = scale * kLog2e * (kind == 2 ? k_scale : 1.f);
  p.v_scale = kind == 2 ? v_scale : 1.f;
  return launch_prefill_attention(p, q_dtype, kind, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

PA_API pa_status pa_prefill_int8(void* out, const void* query, const int8_t* k_cache,
                                 const int8_t* v_cache, const float* k_scales,
                                 const float* v_scales, const int32_t* block_tables,
                                 const int32_t* cu_q, const int32_t* context_lens,
                                 int num_tokens, int num_seqs, int num_heads, int num_kv_heads,
                                 int head_dim, int block_size, int num_blocks,
                                 int max_blocks_per_seq, int max_q_len, float scale,
                                 pa_dtype q_dtype, pa_stream_t stream) {
  return prefill_8bit(1, out, query, k_cache, v_cache, k_scales, v_scales, 1.f, 1.f,
                      block_tables, cu_q, context_lens, num_tokens, num_seqs, num_heads,
                      num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq,
                      max_q_len, scale, q_dtype, stream);
}

PA_API pa_status pa_prefill_fp8(void* out, const void* query, const uint8_t* k_cache,
                                const uint8_t* v_cache, const int32_t* block_tables,
                                const int32_t* cu_q, const int32_t* context_lens, int num_tokens,
                                int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                int block_size, int num_blocks, int max_blocks_per_seq,
                                int max_q_len, float scale, float k_scale, float v_scale,
                                pa_dtype q_dtype, pa_stream_t stream) {
  return prefill_8bit(2, out, query, k_cache, v_cache, nullptr, nullptr, k_scale, v_scale,
                      block_tables, cu_q, context_lens, num_tokens, num_seqs, num_heads,
                      num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq,
                      max_q_len, scale, q_dtype, stream);
}

// ================================================================ cascade
// Split of the shared prefix into ranges of whole 64-token tiles: as many as
// keep (128-row query tiles x kv heads x splits) within one wave of one CTA
// per SM (a second, partial wave would double the time), at least one. The
// number of splits never decreases as sms grows, so a workspace sized for
// kPlanSMs holds the plan of any device with at most that many SMs.
static void cascade_plan(int S, int G, int Hkv, int prefix_tokens, int sms, int* nsp, int* tps) {
  const int qtiles = (S * G + kPrefixCtaRows - 1) / kPrefixCtaRows;
  const int tiles = (prefix_tokens + kPrefixTile - 1) / kPrefixTile;
  const int64_t want = (int64_t)sms / ((int64_t)qtiles * Hkv);
  int n = static_cast<int>(want < 1 ? 1 : (want > tiles ? tiles : want));
  const int tiles_per = (tiles + n - 1) / n;
  *tps = tiles_per * kPrefixTile;
  *nsp = (tiles + tiles_per - 1) / tiles_per;
}

// The current device's SM count for a launch-time plan, capped at kPlanSMs
// (the count the workspace queries assume), read once per device.
static int launch_plan_sms() {
  static std::atomic<int> known[32];
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return kPlanSMs;
  if (dev < 32 && (sms = known[dev].load(std::memory_order_relaxed)) > 0) return sms;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms <= 0)
    return kPlanSMs;
  sms = sms < kPlanSMs ? sms : kPlanSMs;
  if (dev < 32) known[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

static pa_status check_cascade(const DecodeShape& a, int prefix_pages) {
  if (a.q_dtype != PA_BF16 && a.q_dtype != PA_F16) return PA_ERR_DTYPE;
  if (a.D != 64 && a.D != 128) return PA_ERR_HEAD_DIM;
  if (prefix_pages < 1 || prefix_pages > a.MB) return PA_ERR_SHAPE;
  // the prefix kernel stages 16-bit pages by tensor copies: 32-bit row coordinates
  if (a.kv_dtype == PA_KV_AUTO && (long long)a.NB * a.Hkv * a.bs > kMaxTcRows)
    return PA_ERR_SHAPE;
  return PA_OK;
}

PA_API size_t pa_decode_cascade_workspace_size(int num_seqs, int num_heads, int num_kv_heads,
                                               int head_dim, int block_size, int prefix_pages) {
  if (num_seqs <= 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 ||
      head_dim <= 0 || block_size <= 0 || prefix_pages <= 0)
    return 0;
  int nsp = 0, tps = 0;
  cascade_plan(num_seqs, num_heads / num_kv_heads, num_kv_heads, prefix_pages * block_size,
               kPlanSMs, &nsp, &tps);
  const size_t rows = (size_t)num_seqs * num_heads * (nsp + 1);
  return align256(rows * head_dim * 4) + 2 * align256(rows * 4);
}

// The cascade for every cache kind: a.kv_dtype AUTO (16-bit, the query's
// type), FP8_E4M3 (a.k_scale, a.v_scale) or INT8 (row scales k_scales,
// v_scales).
static pa_status cascade_impl(void* out, const void* query, const void* k_cache,
                              const void* v_cache, const float* k_scales, const float* v_scales,
                              const int32_t* block_tables, const int32_t* context_lens,
                              DecodeShape a, float scale, int prefix_pages, void* workspace,
                              size_t workspace_bytes, pa_stream_t stream) {
  const int num_seqs = a.S, num_heads = a.Hq, num_kv_heads = a.Hkv, head_dim = a.D;
  const int block_size = a.bs, num_blocks = a.NB, max_blocks_per_seq = a.MB;
  const int q_dtype = a.q_dtype;
  const bool int8 = a.kv_dtype == PA_KV_INT8;
  // the shared checks (an INT8 cache on the shape with a native cache)
  DecodeShape chk = a;
  if (int8) chk.kv_dtype = PA_KV_AUTO;
  pa_status rc = check_decode(chk, out, query, k_cache, v_cache, block_tables, context_lens);
  if (rc != PA_OK || num_seqs == 0) return rc;
  if (int8 && (!k_scales || !v_scales)) return PA_ERR_NULL;
  if (int8 && (!aligned16(k_scales) || !aligned16(v_scales))) return PA_ERR_ALIGN;
  rc = check_cascade(a, prefix_pages);
  if (rc != PA_OK) return rc;
  if (!workspace) return PA_ERR_NULL;
  const size_t need = pa_decode_cascade_workspace_size(num_seqs, num_heads, num_kv_heads,
                                                       head_dim, block_size, prefix_pages);
  if (workspace_bytes < need) return PA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return PA_ERR_ALIGN;
  const int G = num_heads / num_kv_heads;
  int nsp = 0, tps = 0;
  cascade_plan(num_seqs, G, num_kv_heads, prefix_pages * block_size, launch_plan_sms(), &nsp,
               &tps);
  const int ns = nsp + 1;
  const size_t rows = (size_t)num_seqs * num_heads * ns;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  float* tmp = reinterpret_cast<float*>(w);
  float* ml = reinterpret_cast<float*>(w + align256(rows * head_dim * 4));
  float* es = reinterpret_cast<float*>(w + align256(rows * head_dim * 4) + align256(rows * 4));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  unsigned* err = error_word();

  // The prefix launch goes first and waits for the launches before it; the
  // suffix launch then starts at once and runs beside it (they share only
  // inputs), and waits for it at its end, so the combine sees both.
  // slots 1 .. nsp: the shared prefix, all sequences' query heads at once
  PrefixParams q{};
  q.tmp_out = tmp;
  q.max_logits = ml;
  q.exp_sums = es;
  q.query = query;
  q.k_cache = static_cast<const uint8_t*>(k_cache);
  q.v_cache = static_cast<const uint8_t*>(v_cache);
  q.block_tables = block_tables;
  q.context_lens = context_lens;
  q.err = err;
  q.num_seqs = num_seqs;
  q.num_heads = num_heads;
  q.num_kv_heads = num_kv_heads;
  q.group = G;
  q.head_dim = head_dim;
  q.block_size = block_size;
  q.num_blocks = num_blocks;
  q.max_blocks_per_seq = max_blocks_per_seq;
  q.prefix_pages = prefix_pages;
  q.prefix_tokens = prefix_pages * block_size;
  q.num_slots = ns;
  q.slot0 = 1;
  q.num_prefix_splits = nsp;
  q.tokens_per_split = tps;
  const bool fp8 = a.kv_dtype == PA_KV_FP8_E4M3;
  q.scale_log2 = scale * 1.4426950408889634f * (fp8 ? a.k_scale : 1.f);
  q.v_scale = fp8 ? a.v_scale : 1.f;
  q.k_scales = k_scales;
  q.v_scales = v_scales;
  if (a.kv_dtype == PA_KV_AUTO) {
    const long long rows = (long long)num_blocks * num_kv_heads * block_size;
    if (!page_tensor_map(&q.tm_k, k_cache, q_dtype, head_dim, rows, block_size) ||
        !page_tensor_map(&q.tm_v, v_cache, q_dtype, head_dim, rows, block_size))
      return PA_ERR_CUDA;
  }
  const int kind = int8 ? 1 : fp8 ? 2 : 0;
  if (launch_prefix_attention(q, q_dtype, kind, st) != cudaSuccess) return PA_ERR_CUDA;
  // slot 0: each sequence's own pages after the prefix, one CTA per (sequence, kv head)
  DecodeParams p = make_params(a, query, k_cache, v_cache, block_tables, context_lens, scale, err);
  p.k_scales = k_scales;
  p.v_scales = v_scales;
  p.tmp_out = tmp;
  p.max_logits = ml;
  p.exp_sums = es;
  p.partials = 1;
  p.num_splits = ns;
  p.first_page = prefix_pages;
  p.pages_per_split = max_blocks_per_seq - prefix_pages > 0 ? max_blocks_per_seq - prefix_pages : 1;
  p.join_at_end = 1;  // runs beside the prefix launch, which it waits for at its end
  if (run_decode(p, a, dim3(1, num_kv_heads, num_seqs), kModeSplit, nullptr, st) != cudaSuccess)
    return PA_ERR_CUDA;
  // the log-sum-exp combination of the ns slots
  return run_reduce(out, tmp, ml, es, (int64_t)num_seqs * num_heads, head_dim, ns, q_dtype, st) ==
                 cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

PA_API pa_status pa_decode_cascade(void* out, const void* query, const void* k_cache,
                                   const void* v_cache, const int32_t* block_tables,
                                   const int32_t* context_lens, int num_seqs, int num_heads,
                                   int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                   int max_blocks_per_seq, float scale, pa_dtype q_dtype,
                                   int prefix_pages, void* workspace, size_t workspace_bytes,
                                   pa_stream_t stream) {
  const DecodeShape a{num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                      max_blocks_per_seq, 0, q_dtype, PA_KV_AUTO, 1.f, 1.f};
  return cascade_impl(out, query, k_cache, v_cache, nullptr, nullptr, block_tables, context_lens,
                      a, scale, prefix_pages, workspace, workspace_bytes, stream);
}

PA_API pa_status pa_decode_cascade_fp8(void* out, const void* query, const uint8_t* k_cache,
                                       const uint8_t* v_cache, const int32_t* block_tables,
                                       const int32_t* context_lens, int num_seqs, int num_heads,
                                       int num_kv_heads, int head_dim, int block_size,
                                       int num_blocks, int max_blocks_per_seq, float scale,
                                       float k_scale, float v_scale, pa_dtype q_dtype,
                                       int prefix_pages, void* workspace, size_t workspace_bytes,
                                       pa_stream_t stream) {
  const DecodeShape a{num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                      max_blocks_per_seq, 0, q_dtype, PA_KV_FP8_E4M3, k_scale, v_scale};
  return cascade_impl(out, query, k_cache, v_cache, nullptr, nullptr, block_tables, context_lens,
                      a, scale, prefix_pages, workspace, workspace_bytes, stream);
}

PA_API pa_status pa_decode_cascade_int8(void* out, const void* query, const int8_t* k_cache,
                                        const int8_t* v_cache, const float* k_scales,
                                        const float* v_scales, const int32_t* block_tables,
                                        const int32_t* context_lens, int num_seqs, int num_heads,
                                        int num_kv_heads, int head_dim, int block_size,
                                        int num_blocks, int max_blocks_per_seq, float scale,
                                        pa_dtype q_dtype, int prefix_pages, void* workspace,
                                        size_t workspace_bytes, pa_stream_t stream) {
  const DecodeShape a{num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                      max_blocks_per_seq, 0, q_dtype, PA_KV_INT8, 1.f, 1.f};
  return cascade_impl(out, query, k_cache, v_cache, k_scales, v_scales, block_tables,
                      context_lens, a, scale, prefix_pages, workspace, workspace_bytes, stream);
}

PA_API pa_status pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* block_pairs,
                                int num_pairs, int num_kv_heads, int head_dim, int block_size,
                                int num_blocks, int elem_bytes, pa_stream_t stream) {
  if (num_pairs < 0) return PA_ERR_SHAPE;
  if (num_pairs == 0) return PA_OK;
  if (!k_cache || !v_cache || !block_pairs) return PA_ERR_NULL;
  if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4) return PA_ERR_DTYPE;
  if (num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0) return PA_ERR_SHAPE;
  const size_t block_bytes = (size_t)num_kv_heads * block_size * head_dim * elem_bytes;
  if (block_bytes % 16 != 0) return PA_ERR_HEAD_DIM;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_ALIGN;
  return launch_copy_blocks(static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache),
                            block_pairs, num_pairs, num_blocks, block_bytes, error_word(),
                            reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

// ================================================================ pool sizing
PA_API int64_t pa_block_budget(pa_budget_kind kind, double amount, size_t available_bytes,
                               int num_layers, int num_kv_heads, int head_dim, int block_size,
                               pa_dtype dtype, pa_kv_dtype kv_dtype) {
  if (num_layers <= 0 || num_kv_heads <= 0 || block_size <= 0) return PA_ERR_SHAPE;
  if (head_dim <= 0) return PA_ERR_HEAD_DIM;
  if (!valid_dtype(dtype) ||
      (kv_dtype != PA_KV_AUTO && kv_dtype != PA_KV_FP8_E4M3 && kv_dtype != PA_KV_INT8))
    return PA_ERR_DTYPE;
  if (!(amount >= 0.0) || !isfinite(amount)) return PA_ERR_SHAPE;
  const int64_t elem = kv_dtype != PA_KV_AUTO ? 1 : (dtype == PA_F32 ? 4 : 2);
  // bytes of one cached row: its elements, plus its fp32 scale for INT8
  const double row_bytes = (double)head_dim * elem + (kv_dtype == PA_KV_INT8 ? 4.0 : 0.0);
  const double block_bytes = (double)num_layers * 2.0 * num_kv_heads * block_size * row_bytes;
  double blocks = 0.0;
  switch (kind) {
    case PA_BUDGET_MB:
      blocks = std::floor(amount * 1048576.0 / block_bytes);
      break;
    case PA_BUDGET_FRACTION:
      if (amount > 1.0) return PA_ERR_SHAPE;
      blocks = std::floor(amount * (double)available_bytes / block_bytes);
      break;
    case PA_BUDGET_CONTEXT:
      blocks = std::ceil(amount / block_size);
      break;
    default:
      return PA_ERR_SHAPE;
  }
  if (blocks > 9.0e18) return PA_ERR_SHAPE;
  return static_cast<int64_t>(blocks);
}

PA_API void pa_test_set_unarmed_page(int page) { g_unarmed_page.store(page < 0 ? -1 : page); }

PA_API pa_status pa_get_device_error(pa_stream_t stream, uint32_t* error_bits) {
  if (error_bits) *error_bits = 0;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PA_ERR_CUDA;
  unsigned* dev = error_word();
  if (!dev) return PA_ERR_CUDA;
  unsigned bits = 0;
  if (cudaMemcpy(&bits, dev, sizeof(bits), cudaMemcpyDeviceToHost) != cudaSuccess)
    return PA_ERR_CUDA;
  if (bits) {
    const unsigned zero = 0;
    if (cudaMemcpy(dev, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return PA_ERR_CUDA;
  }
  if (error_bits) *error_bits = bits;
  return bits ? PA_ERR_DEVICE : PA_OK;
}
