// pa_cascade.cu -- shared-prefix attention on the tensor cores, and block
// copies for copy-on-write.
//
// The prefix part of a cascade decode is a real dense contraction (every
// K/V row of the shared prefix is used by all S * G query rows of its kv
// head), so it runs on warp-level MMAs (m16n8k16, bf16/f16 in, fp32
// accumulate), flash-attention style: a CTA holds 64 query rows (16 per
// warp) in registers, streams the prefix in tiles of 64 tokens through
// double-buffered shared memory (16-byte async copies into an XOR-swizzled
// layout, so that the 8 rows an ldmatrix reads fall in 8 different bank
// groups), computes S = Q K^T, keeps a running maximum and sum per row, and
// accumulates O = P V with P rounded to the input type. The decode kernel
// proper stays on CUDA cores: there each K/V row has one query row per head.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_cascade.cuh"
#include "pa_device.cuh"

namespace pa {
namespace {

constexpr int kThreads = 128;  // 4 warps x 16 query rows

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  // 16 bytes global -> shared, zero-filled when !valid (src is not read then)
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Byte offset of 16-byte chunk c of row r in a tile of rows of CPR chunks:
// the chunk index is XORed with r mod 8, so the same chunk of 8 consecutive
// rows lands in 8 different 16-byte bank groups.
template <int CPR>
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>(r * CPR * 16 + ((c ^ (r & 7)) << 4));
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefix_attention_kernel(const __grid_constant__ PrefixParams p) {
  constexpr int CPR = D / 8;                // 16-byte chunks per row
  constexpr int TILE = kPrefixTile;         // tokens per K/V tile
  constexpr int TBYTES = TILE * D * 2;      // bytes of one K or V tile
  constexpr int KS = D / 16;                // k-steps of Q K^T
  constexpr int NT = TILE / 8;              // 8-token n-tiles of S
  constexpr int NO = D / 8;                 // 8-column n-tiles of O
  static_assert(CPR >= 8, "the swizzle needs 8 chunks per row");
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sq = smem;                       // [64][D]
  uint8_t* sk = smem + kPrefixRows * D * 2; // [2][TILE][D]
  uint8_t* sv = sk + 2 * TBYTES;            // [2][TILE][D]
  int* sblk = reinterpret_cast<int*>(sv + 2 * TBYTES);  // the split's block ids

  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qt = blockIdx.x, split = blockIdx.y, g = blockIdx.z;
  const int S = p.num_seqs, Hq = p.num_heads, Hkv = p.num_kv_heads, G = p.group;
  const int bs = p.block_size, rows_total = S * G;
  const int t_begin = split * p.tokens_per_split;
  const int t_end = min(p.prefix_tokens, t_begin + p.tokens_per_split);
  const int slot = p.slot0 + split;

  // the precondition, checked on a slice per CTA: every row's first
  // prefix_pages entries equal row 0's, and every context covers the prefix
  {
    const int cta = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
    const int nctas = gridDim.x * gridDim.y * gridDim.z;
    for (int s = 1 + cta; s < S; s += nctas)
      for (int i = tid; i < p.prefix_pages; i += kThreads)
        if (p.block_tables[(size_t)s * p.max_blocks_per_seq + i] != p.block_tables[i])
          raise_error(p.err, PA_DEVERR_BLOCK_ID);
    for (int s = cta * kThreads + tid; s < S; s += nctas * kThreads)
      if (p.context_lens[s] < p.prefix_tokens) raise_error(p.err, PA_DEVERR_CONTEXT_LEN);
  }

  if (t_begin >= t_end) {  // a split with no prefix token: empty partials
    for (int i = tid; i < kPrefixRows; i += kThreads) {
      const int r = qt * kPrefixRows + i;
      if (r < rows_total) {
        const size_t row = (size_t)(r / G) * Hq + g * G + r % G;
        p.max_logits[row * p.num_slots + slot] = -INFINITY;
        p.exp_sums[row * p.num_slots + slot] = 0.f;
      }
    }
    return;
  }
  // block ids of the split's pages
  const int pg_begin = t_begin / bs, pg_end = (t_end + bs - 1) / bs;
  for (int i = pg_begin + tid; i < pg_end; i += kThreads) {
    int b = p.block_tables[i];
    if (b < 0 || b >= p.num_blocks) {
      raise_error(p.err, PA_DEVERR_BLOCK_ID);
      b = -1;
    }
    sblk[i - pg_begin] = b;
  }

  // Q rows of this CTA -> shared memory (rows past S * G are zero)
  const uint32_t sq_u = smem_u32(sq), sk_u = smem_u32(sk), sv_u = smem_u32(sv);
  for (int i = tid; i < kPrefixRows * CPR; i += kThreads) {
    const int rr = i / CPR, c = i % CPR, r = qt * kPrefixRows + rr;
    const bool ok = r < rows_total;
    const size_t row = ok ? (size_t)(r / G) * Hq + g * G + r % G : 0;
    cp_async16(sq_u + swz<CPR>(rr, c),
               static_cast<const uint8_t*>(p.query) + (row * D + c * 8) * 2, ok);
  }
  __syncthreads();  // sblk
  const size_t head_stride = (size_t)bs * D * 2;  // bytes of one (block, kv head) page
  auto load_tile = [&](int tile, int buf) {
    const int t0 = t_begin + tile * TILE;
    for (int i = tid; i < TILE * CPR; i += kThreads) {
      const int rr = i / CPR, c = i % CPR, t = t0 + rr;
      int b = -1;
      if (t < t_end) b = sblk[t / bs - pg_begin];
      const bool ok = b >= 0;
      const size_t off = ok ? ((size_t)b * Hkv + g) * head_stride + (size_t)(t % bs) * D * 2 + c * 16
                            : 0;
      cp_async16(sk_u + buf * TBYTES + swz<CPR>(rr, c), p.k_cache + off, ok);
      cp_async16(sv_u + buf * TBYTES + swz<CPR>(rr, c), p.v_cache + off, ok);
    }
  };
  const int ntiles = (t_end - t_begin + TILE - 1) / TILE;
  load_tile(0, 0);
  cp_async_commit();  // group: Q + tile 0

  // Q fragments of this warp's 16 rows
  cp_async_wait<0>();
  __syncthreads();
  uint32_t qa[KS][4];
#pragma unroll
  for (int kk = 0; kk < KS; ++kk)
    ldsm_x4(sq_u + swz<CPR>(warp * 16 + (lane & 15), 2 * kk + (lane >> 4)), qa[kk][0], qa[kk][1],
            qa[kk][2], qa[kk][3]);

  float o[NO][4];
#pragma unroll
  for (int n = 0; n < NO; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // rows lane/4 and lane/4 + 8
  const int tq = lane & 3;

  for (int tile = 0; tile < ntiles; ++tile) {
    const int buf = tile & 1;
    if (tile + 1 < ntiles) load_tile(tile + 1, buf ^ 1);
    cp_async_commit();
    cp_async_wait<1>();  // this tile's copies are done
    __syncthreads();
    const uint32_t kb = sk_u + buf * TBYTES, vb = sv_u + buf * TBYTES;

    // S = Q K^T for 16 rows x 64 tokens; the 8 token tiles are independent
    // accumulators, so each k-step issues 8 MMAs that do not wait on each
    // other
    float s[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KS; kk += 2) {
      uint32_t b2[NT], b3[NT];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        uint32_t b0, b1;
        ldsm_x4(kb + swz<CPR>(8 * j + (lane & 7), 2 * kk + (lane >> 3)), b0, b1, b2[j], b3[j]);
        Mma<T>::run(s[j], qa[kk], b0, b1);
      }
#pragma unroll
      for (int j = 0; j < NT; ++j) Mma<T>::run(s[j], qa[kk + 1], b2[j], b3[j]);
    }
    // scale to log2 units, mask tokens past the range, running maximum
    const int t0 = t_begin + tile * TILE;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool ok = t0 + 8 * j + 2 * tq + (e & 1) < t_end;
        s[j][e] = ok ? s[j][e] * p.scale_log2 : -INFINITY;
        if (e < 2) mx0 = fmaxf(mx0, s[j][e]);
        else mx1 = fmaxf(mx1, s[j][e]);
      }
#pragma unroll
    for (int off = 1; off <= 2; off *= 2) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
    // every tile holds at least one valid token, so n0, n1 are finite
    const float a0 = exp2f(m0 - n0), a1 = exp2f(m1 - n1);
    m0 = n0;
    m1 = n1;
    l0 *= a0;
    l1 *= a1;
#pragma unroll
    for (int n = 0; n < NO; ++n) {
      o[n][0] *= a0;
      o[n][1] *= a0;
      o[n][2] *= a1;
      o[n][3] *= a1;
    }
    // P as A fragments (16 tokens per k-step), row sums from the fp32 values
    uint32_t pa[NT / 2][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const float p0 = exp2f(s[j][0] - n0), p1 = exp2f(s[j][1] - n0);
      const float p2 = exp2f(s[j][2] - n1), p3 = exp2f(s[j][3] - n1);
      l0 += p0 + p1;
      l1 += p2 + p3;
      pa[j / 2][(j & 1) * 2 + 0] = Mma<T>::pack(p0, p1);
      pa[j / 2][(j & 1) * 2 + 1] = Mma<T>::pack(p2, p3);
    }
    // O += P V
#pragma unroll
    for (int kk = 0; kk < NT / 2; ++kk)
#pragma unroll
      for (int n = 0; n < NO; n += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + swz<CPR>(16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1), n + (lane >> 4)), b0,
                  b1, b2, b3);
        Mma<T>::run(o[n], pa[kk], b0, b1);
        Mma<T>::run(o[n + 1], pa[kk], b2, b3);
      }
    __syncthreads();  // the buffer is refilled two tiles on
  }

  // row sums over the quad, then the partials of this warp's rows
#pragma unroll
  for (int off = 1; off <= 2; off *= 2) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  constexpr float kLn2 = 0.69314718055994530942f;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = qt * kPrefixRows + warp * 16 + (lane >> 2) + 8 * half;
    if (r >= rows_total) continue;
    const size_t row = (size_t)(r / G) * Hq + g * G + r % G;
    const float l = half ? l1 : l0, m = half ? m1 : m0;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    float* dst = p.tmp_out + (row * p.num_slots + slot) * D;
#pragma unroll
    for (int n = 0; n < NO; ++n)
      *reinterpret_cast<float2*>(dst + 8 * n + 2 * tq) =
          make_float2(o[n][2 * half] * inv, o[n][2 * half + 1] * inv);
    if (tq == 0) {
      p.max_logits[row * p.num_slots + slot] = l > 0.f ? m * kLn2 : -INFINITY;
      p.exp_sums[row * p.num_slots + slot] = l;
    }
  }
}

// Causal prefill over the paged cache: one CTA per (64-row query tile, kv
// head, sequence), with the tiles, fragments and online softmax of the prefix
// kernel above. The CTA's rows are (token, head-in-group) pairs of one
// sequence; it streams that sequence's pages from position 0 up to the
// position of its last row, and masks key t for a row at position pos when
// t > pos. Every row sees position 0, so its running maximum is finite from
// the first tile on.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_attention_kernel(const __grid_constant__ PrefillParams p) {
  constexpr int CPR = D / 8;
  constexpr int TILE = kPrefixTile;
  constexpr int TBYTES = TILE * D * 2;
  constexpr int KS = D / 16;
  constexpr int NT = TILE / 8;
  constexpr int NO = D / 8;
  static_assert(CPR >= 8, "the swizzle needs 8 chunks per row");
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sq = smem;                        // [64][D]
  uint8_t* sk = smem + kPrefixRows * D * 2;  // [2][TILE][D]
  uint8_t* sv = sk + 2 * TBYTES;             // [2][TILE][D]

  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qt = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int Hq = p.num_heads, Hkv = p.num_kv_heads, G = p.group, bs = p.block_size;
  const int MB = p.max_blocks_per_seq;
  const bool reporter = qt == 0 && g == 0 && tid == 0;  // flags a sequence's errors once

  // this sequence's query tokens [q0, q0 + q_len) and context of n tokens
  const int q0 = p.cu_q[s];
  int q_len = p.cu_q[s + 1] - q0;
  const int n = p.context_lens[s];
  if (q_len < 0 || q0 < 0 || q0 > p.num_tokens - max(q_len, 0) || q_len > p.max_q_len) {
    if (reporter) raise_error(p.err, PA_DEVERR_SEQ);
    return;  // offsets that do not fit the batch: nothing of this sequence is written
  }
  const int rows_total = q_len * G;
  if (qt * kPrefixRows >= rows_total) return;
  T* out = static_cast<T*>(p.out);
  if (n < q_len || n > MB * bs) {  // the chunk does not fit its context: zero rows
    if (reporter) raise_error(p.err, PA_DEVERR_CONTEXT_LEN);
    for (int i = tid; i < kPrefixRows * D; i += kThreads) {
      const int r = qt * kPrefixRows + i / D;
      if (r < rows_total)
        out[((size_t)(q0 + r / G) * Hq + g * G + r % G) * D + i % D] = Elem<T>::from_f32(0.f);
    }
    return;
  }
  const int pos0 = n - q_len;  // position of the chunk's first token
  const int r_last = min(qt * kPrefixRows + kPrefixRows, rows_total) - 1;
  const int kv_end = pos0 + r_last / G + 1;  // keys this CTA needs: positions [0, kv_end)

  // Q rows of this CTA -> shared memory (rows past the sequence's are zero)
  const uint32_t sq_u = smem_u32(sq), sk_u = smem_u32(sk), sv_u = smem_u32(sv);
  for (int i = tid; i < kPrefixRows * CPR; i += kThreads) {
    const int rr = i / CPR, c = i % CPR, r = qt * kPrefixRows + rr;
    const bool ok = r < rows_total;
    const size_t row = ok ? (size_t)(q0 + r / G) * Hq + g * G + r % G : 0;
    cp_async16(sq_u + swz<CPR>(rr, c),
               static_cast<const uint8_t*>(p.query) + (row * D + c * 8) * 2, ok);
  }
  const size_t head_stride = (size_t)bs * D * 2;  // bytes of one (block, kv head) page
  const int32_t* table = p.block_tables + (size_t)s * MB;
  auto load_tile = [&](int tile, int buf) {
    const int t0 = tile * TILE;
    for (int i = tid; i < TILE * CPR; i += kThreads) {
      const int rr = i / CPR, c = i % CPR, t = t0 + rr;
      int b = -1;
      if (t < kv_end) {
        b = __ldg(table + t / bs);
        if (b < 0 || b >= p.num_blocks) {
          if (c == 0) raise_error(p.err, PA_DEVERR_BLOCK_ID);
          b = -1;
        }
      }
      const bool ok = b >= 0;
      const size_t off = ok ? ((size_t)b * Hkv + g) * head_stride + (size_t)(t % bs) * D * 2 + c * 16
                            : 0;
      cp_async16(sk_u + buf * TBYTES + swz<CPR>(rr, c), p.k_cache + off, ok);
      cp_async16(sv_u + buf * TBYTES + swz<CPR>(rr, c), p.v_cache + off, ok);
    }
  };
  const int ntiles = (kv_end + TILE - 1) / TILE;
  load_tile(0, 0);
  cp_async_commit();  // group: Q + tile 0

  cp_async_wait<0>();
  __syncthreads();
  uint32_t qa[KS][4];
#pragma unroll
  for (int kk = 0; kk < KS; ++kk)
    ldsm_x4(sq_u + swz<CPR>(warp * 16 + (lane & 15), 2 * kk + (lane >> 4)), qa[kk][0], qa[kk][1],
            qa[kk][2], qa[kk][3]);

  // positions of this lane's two rows (a row past the sequence's takes the
  // CTA's last position: finite values that are never stored)
  const int rA = qt * kPrefixRows + warp * 16 + (lane >> 2), rB = rA + 8;
  const int posA = rA < rows_total ? pos0 + rA / G : kv_end - 1;
  const int posB = rB < rows_total ? pos0 + rB / G : kv_end - 1;

  float o[NO][4];
#pragma unroll
  for (int nn = 0; nn < NO; ++nn) o[nn][0] = o[nn][1] = o[nn][2] = o[nn][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // rows rA and rB
  const int tq = lane & 3;

  for (int tile = 0; tile < ntiles; ++tile) {
    const int buf = tile & 1;
    if (tile + 1 < ntiles) load_tile(tile + 1, buf ^ 1);
    cp_async_commit();
    cp_async_wait<1>();  // this tile's copies are done
    __syncthreads();
    const uint32_t kb = sk_u + buf * TBYTES, vb = sv_u + buf * TBYTES;

    float sc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KS; kk += 2) {
      uint32_t b2[NT], b3[NT];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        uint32_t b0, b1;
        ldsm_x4(kb + swz<CPR>(8 * j + (lane & 7), 2 * kk + (lane >> 3)), b0, b1, b2[j], b3[j]);
        Mma<T>::run(sc[j], qa[kk], b0, b1);
      }
#pragma unroll
      for (int j = 0; j < NT; ++j) Mma<T>::run(sc[j], qa[kk + 1], b2[j], b3[j]);
    }
    // scale to log2 units, causal mask, running maximum
    const int t0 = tile * TILE;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int t = t0 + 8 * j + 2 * tq + (e & 1);
        const bool ok = t <= (e < 2 ? posA : posB);
        sc[j][e] = ok ? sc[j][e] * p.scale_log2 : -INFINITY;
        if (e < 2) mx0 = fmaxf(mx0, sc[j][e]);
        else mx1 = fmaxf(mx1, sc[j][e]);
      }
#pragma unroll
    for (int off = 1; off <= 2; off *= 2) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    // m0, m1 are finite after the first tile (position 0 is always seen), so
    // a tile wholly past a row's position leaves it unchanged (factor 1, p 0)
    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
    const float a0 = exp2f(m0 - n0), a1 = exp2f(m1 - n1);
    m0 = n0;
    m1 = n1;
    l0 *= a0;
    l1 *= a1;
#pragma unroll
    for (int nn = 0; nn < NO; ++nn) {
      o[nn][0] *= a0;
      o[nn][1] *= a0;
      o[nn][2] *= a1;
      o[nn][3] *= a1;
    }
    uint32_t pa[NT / 2][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const float p0 = exp2f(sc[j][0] - n0), p1 = exp2f(sc[j][1] - n0);
      const float p2 = exp2f(sc[j][2] - n1), p3 = exp2f(sc[j][3] - n1);
      l0 += p0 + p1;
      l1 += p2 + p3;
      pa[j / 2][(j & 1) * 2 + 0] = Mma<T>::pack(p0, p1);
      pa[j / 2][(j & 1) * 2 + 1] = Mma<T>::pack(p2, p3);
    }
#pragma unroll
    for (int kk = 0; kk < NT / 2; ++kk)
#pragma unroll
      for (int nn = 0; nn < NO; nn += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + swz<CPR>(16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1), nn + (lane >> 4)),
                  b0, b1, b2, b3);
        Mma<T>::run(o[nn], pa[kk], b0, b1);
        Mma<T>::run(o[nn + 1], pa[kk], b2, b3);
      }
    __syncthreads();  // the buffer is refilled two tiles on
  }

#pragma unroll
  for (int off = 1; off <= 2; off *= 2) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = half ? rB : rA;
    if (r >= rows_total) continue;
    const size_t row = (size_t)(q0 + r / G) * Hq + g * G + r % G;
    const float inv = 1.f / (half ? l1 : l0);
    uint32_t* dst = reinterpret_cast<uint32_t*>(out + row * D);
#pragma unroll
    for (int nn = 0; nn < NO; ++nn)
      dst[4 * nn + tq] = Mma<T>::pack(o[nn][2 * half] * inv, o[nn][2 * half + 1] * inv);
  }
}

__global__ void copy_blocks_kernel(uint8_t* k_cache, uint8_t* v_cache, const int32_t* pairs,
                                   int num_blocks, size_t block_bytes, unsigned* err) {
  pdl_wait();
  pdl_trigger();
  const int src = pairs[2 * blockIdx.x], dst = pairs[2 * blockIdx.x + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0) raise_error(err, PA_DEVERR_BLOCK_ID);
    return;
  }
  uint8_t* base = blockIdx.y ? v_cache : k_cache;
  const uint4* s = reinterpret_cast<const uint4*>(base + (size_t)src * block_bytes);
  uint4* d = reinterpret_cast<uint4*>(base + (size_t)dst * block_bytes);
  for (size_t i = threadIdx.x; i < block_bytes / 16; i += blockDim.x) d[i] = s[i];
}

template <typename T, int D>
cudaError_t launch_prefix(const PrefixParams& p, cudaStream_t st) {
  const int smem = kPrefixRows * D * 2 + 4 * kPrefixTile * D * 2 +
                   4 * ((p.tokens_per_split + p.block_size - 1) / p.block_size + 1);
  auto kern = prefix_attention_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((p.num_seqs * p.group + kPrefixRows - 1) / kPrefixRows, p.num_prefix_splits,
                  p.num_kv_heads);
  return launch_pdl(kern, grid, dim3(kThreads), smem, st, p);
}

template <typename T, int D>
cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t st) {
  const int smem = kPrefixRows * D * 2 + 4 * kPrefixTile * D * 2;
  auto kern = prefill_attention_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long tiles = ((long long)p.max_q_len * p.group + kPrefixRows - 1) / kPrefixRows;
  const dim3 grid(static_cast<unsigned>(tiles), p.num_kv_heads, p.num_seqs);
  return launch_pdl(kern, grid, dim3(kThreads), smem, st, p);
}

}  // namespace

cudaError_t launch_prefix_attention(const PrefixParams& p, int dtype, cudaStream_t st) {
  if (dtype == PA_BF16) {
    if (p.head_dim == 64) return launch_prefix<__nv_bfloat16, 64>(p, st);
    if (p.head_dim == 128) return launch_prefix<__nv_bfloat16, 128>(p, st);
  } else if (dtype == PA_F16) {
    if (p.head_dim == 64) return launch_prefix<__half, 64>(p, st);
    if (p.head_dim == 128) return launch_prefix<__half, 128>(p, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_prefill_attention(const PrefillParams& p, int dtype, cudaStream_t st) {
  if (dtype == PA_BF16) {
    if (p.head_dim == 64) return launch_prefill<__nv_bfloat16, 64>(p, st);
    if (p.head_dim == 128) return launch_prefill<__nv_bfloat16, 128>(p, st);
  } else if (dtype == PA_F16) {
    if (p.head_dim == 64) return launch_prefill<__half, 64>(p, st);
    if (p.head_dim == 128) return launch_prefill<__half, 128>(p, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_copy_blocks(uint8_t* k_cache, uint8_t* v_cache, const int32_t* block_pairs,
                               int num_pairs, int num_blocks, size_t block_bytes, unsigned* err,
                               cudaStream_t st) {
  if (num_pairs <= 0) return cudaSuccess;
  return launch_pdl(copy_blocks_kernel, dim3(num_pairs, 2), dim3(256), 0, st, k_cache, v_cache,
                    block_pairs, num_blocks, block_bytes, err);
}

}  // namespace pa
