// pa_cascade.cu -- shared-prefix attention on the tensor cores, paged
// prefill attention, and block copies for copy-on-write.
//
// The prefix part of a cascade decode is a real dense contraction (every
// K/V row of the shared prefix is used by all S * G query rows of its kv
// head), so it runs on the fifth-generation tensor cores (tcgen05 MMAs with
// TMEM accumulators, operands staged by tensor copies), flash-attention
// style; see prefix_attention_kernel. The prefill kernel runs warp-level MMAs
// (m16n8k16, bf16/f16 in, fp32 accumulate) over 64-row query tiles with K/V
// tiles in double-buffered, XOR-swizzled shared memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "pa_cascade.cuh"
#include "pa_device.cuh"

namespace pa {
namespace {

constexpr int kPrefillThreads = 256;  // 8 warps x 16 query rows

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

// Shared-prefix attention on the fifth-generation tensor cores. A CTA takes
// 128 query rows (all sequences' query heads of one kv head, row r = s G + h)
// and one range of the prefix, in tiles of 64 tokens:
//   S = Q K^T   (M 128 x N 64, K = D)        -> TMEM, two buffers
//   softmax     (one thread per row, lazy running maximum in log2 units)
//   O += P V    (M 128 x N D, K = 64 tokens) -> TMEM
// Q is staged once, K/V tiles come by 2-D tensor copies of whole pages (the
// prefix's block ids from row 0 of the block tables), P is written to shared
// memory by the softmax threads; all three operands use the 128-byte swizzle.
// Warps 0-3: softmax (thread t owns row t, TMEM lane t); warp 4: MMA issue
// and TMEM allocation; warp 5: tensor copies. Every wait is bounded.
constexpr int kTcRows = kPrefixTcRows;
constexpr int kTcTile = kPrefixTile;
#ifndef PA_PREFIX_STAGES
#define PA_PREFIX_STAGES 4
#endif
constexpr int kTcStages = PA_PREFIX_STAGES;
constexpr int kTcThreads = 192;

template <int D>
struct PrefixTcLayout {
  static constexpr int KB = D / 64;                  // 128-byte column blocks of a row
  static constexpr int QBYTES = KB * kTcRows * 128;  // Q: [KB][128 rows][128 B]
  static constexpr int TBYTES = KB * kTcTile * 128;  // one K or V tile: [KB][64 tokens][128 B]
  static constexpr int PBYTES = kTcRows * 128;       // P: [128 rows][64 tokens = 128 B]
  static constexpr int OFF_KV = QBYTES;
  static constexpr int OFF_P = OFF_KV + kTcStages * 2 * TBYTES;
  static constexpr int OFF_BAR = OFF_P + 2 * PBYTES;
  static constexpr int NBAR = 2 * kTcStages + 8;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;  // + alignment of the base to 1024
  static constexpr uint32_t TMEM_COLS = 256;         // S: 2 x 64, O: D
  static_assert(2 * kTcTile + D <= 256, "TMEM columns");
};

template <typename T, int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefix_attention_kernel(const __grid_constant__ PrefixParams p) {
  using Ly = PrefixTcLayout<D>;
  constexpr int KB = Ly::KB;
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* kv_full = reinterpret_cast<uint64_t*>(smem + Ly::OFF_BAR);
  uint64_t* kv_empty = kv_full + kTcStages;
  uint64_t* s_full = kv_empty + kTcStages;  // [2]
  uint64_t* s_free = s_full + 2;            // [2]
  uint64_t* p_full = s_free + 2;            // [2]
  uint64_t* pv_done = p_full + 2;           // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Ly::OFF_MISC);

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
      for (int i = tid; i < p.prefix_pages; i += kTcThreads)
        if (p.block_tables[(size_t)s * p.max_blocks_per_seq + i] != p.block_tables[i])
          raise_error(p.err, PA_DEVERR_BLOCK_ID);
    for (int s = cta * kTcThreads + tid; s < S; s += nctas * kTcThreads)
      if (p.context_lens[s] < p.prefix_tokens) raise_error(p.err, PA_DEVERR_CONTEXT_LEN);
  }
  if (t_begin >= t_end) {  // a split with no prefix token: empty partials
    for (int i = tid; i < kTcRows; i += kTcThreads) {
      const int r = qt * kTcRows + i;
      if (r < rows_total) {
        const size_t row = (size_t)(r / G) * Hq + g * G + r % G;
        p.max_logits[row * p.num_slots + slot] = -INFINITY;
        p.exp_sums[row * p.num_slots + slot] = 0.f;
      }
    }
    return;
  }
  const int ntiles = (t_end - t_begin + kTcTile - 1) / kTcTile;

  // ---- set-up: barriers, TMEM, Q rows (rows past S * G are zero)
  if (tid == 0) {
    for (int i = 0; i < kTcStages; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], kTcRows);
      mbar_init(&p_full[i], kTcRows);
      mbar_init(&pv_done[i], 1);
    }
    fence_mbar_init();
  }
  if (warp == 4) {
    __syncwarp();
    tmem_alloc(tmem_slot, Ly::TMEM_COLS);
  }
  const uint32_t sq = smem_u32(smem);
  // asynchronous 16-byte copies, all in flight at once (zero-filled rows
  // past S * G)
  for (int i = tid; i < kTcRows * KB * 8; i += kTcThreads) {
    const int rr = i / (KB * 8), c = i % (KB * 8), r = qt * kTcRows + rr;
    const bool ok = r < rows_total;
    const size_t row = ok ? (size_t)(r / G) * Hq + g * G + r % G : 0;
    const int kb = c >> 3, ch = c & 7;
    cp_async16(sq + kb * (kTcRows * 128) + rr * 128 + ((ch ^ (rr & 7)) << 4),
               static_cast<const uint8_t*>(p.query) + (row * D + c * 8) * 2, ok);
  }
  cp_async_commit();
  cp_async_wait<0>();
  fence_proxy_async_smem();
  tc05_fence_before();
  __syncthreads();
  tc05_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_s = tmem, t_o = tmem + 2 * kTcTile;  // S buffers at columns 0 / 64, O at 128
  bool failed = false;

  if (warp == 5) {
    // ================================================ tensor copies of K/V tiles
    if (lane == 0) {
      const long long rows = (long long)p.num_blocks * Hkv * bs;
      int issued = 0;
      for (int i = 0; i < ntiles && !failed; ++i) {
        const int st = i % kTcStages;
        if (i >= kTcStages && !mbar_wait_bounded(&kv_empty[st], ((i / kTcStages) - 1) & 1)) {
          raise_error(p.err, PA_DEVERR_TIMEOUT);
          failed = true;
          break;
        }
        mbar_arrive_expect_tx(&kv_full[st], 2 * Ly::TBYTES);
        uint8_t* kdst = smem + Ly::OFF_KV + st * 2 * Ly::TBYTES;
        uint8_t* vdst = kdst + Ly::TBYTES;
        const int t0 = t_begin + i * kTcTile;
        for (int pp = 0; pp < kTcTile / bs; ++pp) {
          const int t = t0 + pp * bs;
          // pages past the range and bad block ids read as zeros (a box
          // wholly past the tensor is filled with zeros)
          int y = static_cast<int>(rows);
          if (t < t_end) {
            const int b = __ldg(p.block_tables + t / bs);
            if (b >= 0 && b < p.num_blocks)
              y = (b * Hkv + g) * bs;
            else
              raise_error(p.err, PA_DEVERR_BLOCK_ID);
          }
#pragma unroll
          for (int j = 0; j < KB; ++j) {
            tma_load_2d(kdst + j * (kTcTile * 128) + pp * bs * 128, &p.tm_k, 64 * j, y, &kv_full[st]);
            tma_load_2d(vdst + j * (kTcTile * 128) + pp * bs * 128, &p.tm_v, 64 * j, y, &kv_full[st]);
          }
        }
        ++issued;
      }
      // never leave with copies in flight
      for (int k = issued > kTcStages ? issued - kTcStages : 0; k < issued; ++k)
        if (!mbar_wait_bounded(&kv_full[k % kTcStages], (k / kTcStages) & 1))
          raise_error(p.err, PA_DEVERR_TIMEOUT);
    }
  } else if (warp == 4) {
    // ================================================ MMA issue (one thread)
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc_f16(kBf16, kTcRows, kTcTile, false);
      constexpr uint32_t idesc_o = umma_idesc_f16(kBf16, kTcRows, D, true);
      const uint32_t skv = smem_u32(smem + Ly::OFF_KV), sp = smem_u32(smem + Ly::OFF_P);
      auto issue_s = [&](int i) -> bool {
        const int st = i % kTcStages;
        if (!mbar_wait_bounded(&kv_full[st], (i / kTcStages) & 1)) return false;
        if (i >= 2 && !mbar_wait_bounded(&s_free[i & 1], ((i >> 1) - 1) & 1)) return false;
        tc05_fence_after();
        const uint32_t kt = skv + st * 2 * Ly::TBYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t qa = sq + (kk >> 2) * (kTcRows * 128) + (kk & 3) * 32;
          const uint32_t kbd = kt + (kk >> 2) * (kTcTile * 128) + (kk & 3) * 32;
          umma_f16(t_s + (i & 1) * kTcTile, umma_sdesc_sw128(qa, 16, 1024),
                   umma_sdesc_sw128(kbd, 16, 1024), idesc_s, kk > 0);
        }
        umma_commit(&s_full[i & 1]);
        return true;
      };
      bool ok = issue_s(0);
      for (int i = 0; i < ntiles && ok; ++i) {
        if (i + 1 < ntiles) ok = issue_s(i + 1);
        if (!ok) break;
        if (!mbar_wait_bounded(&p_full[i & 1], (i >> 1) & 1)) {
          ok = false;
          break;
        }
        tc05_fence_after();
        const uint32_t vt = skv + (i % kTcStages) * 2 * Ly::TBYTES + Ly::TBYTES;
        const uint32_t pa = sp + (i & 1) * Ly::PBYTES;
#pragma unroll
        for (int kk = 0; kk < kTcTile / 16; ++kk)
          umma_f16(t_o, umma_sdesc_sw128(pa + kk * 32, 16, 1024),
                   umma_sdesc_sw128(vt + kk * 2048, kTcTile * 128, 1024), idesc_o,
                   i > 0 || kk > 0);
        umma_commit(&pv_done[i & 1]);
        if (i + kTcStages < ntiles) umma_commit(&kv_empty[i % kTcStages]);  // a later tile refills it
      }
      if (!ok) raise_error(p.err, PA_DEVERR_TIMEOUT);
    }
  } else {
    // ================================================ softmax, one row per thread
    // (tcgen05.ld / st are warp-wide: every decision that leads to one is
    // taken by the whole warp)
    const int row_in = tid;  // 0 .. 127 = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    constexpr float kLazy = 8.f;
    float m = -INFINITY, l = 0.f;
    uint8_t* prow = smem + Ly::OFF_P + row_in * 128;
    for (int i = 0; i < ntiles; ++i) {
      if (__any_sync(0xffffffffu, !mbar_wait_bounded(&s_full[i & 1], (i >> 1) & 1))) {
        raise_error(p.err, PA_DEVERR_TIMEOUT);
        failed = true;
        break;
      }
      tc05_fence_after();
      __syncwarp();
      uint32_t sr[2][32];
      tmem_ld32(t_s + (i & 1) * kTcTile + lane_off, sr[0]);
      tmem_ld32(t_s + (i & 1) * kTcTile + 32 + lane_off, sr[1]);
      tmem_wait_ld();
      tc05_fence_before();
      mbar_arrive(&s_free[i & 1]);
      // logits in log2 units; columns past the range (only in a partial
      // last tile) are -inf
      const int valid = t_end - (t_begin + i * kTcTile);  // >= 1
      const float sl = p.scale_log2;
      float x[kTcTile];
#pragma unroll
      for (int c = 0; c < kTcTile; ++c) x[c] = __uint_as_float(sr[c >> 5][c & 31]) * sl;
      if (valid < kTcTile) {  // CTA-uniform
#pragma unroll
        for (int c = 0; c < kTcTile; ++c) x[c] = c < valid ? x[c] : -INFINITY;
      }
      float mx = x[0];
#pragma unroll
      for (int c = 1; c < kTcTile; ++c) mx = fmaxf(mx, x[c]);
      if (__any_sync(0xffffffffu, mx > m + kLazy)) {
        const float mn = fmaxf(m, mx);
        if (i > 0) {
          // O holds the tiles so far: scale it by 2^(m - mn) once the last
          // P V has landed
          if (__any_sync(0xffffffffu,
                         !mbar_wait_bounded(&pv_done[(i - 1) & 1], ((i - 1) >> 1) & 1))) {
            raise_error(p.err, PA_DEVERR_TIMEOUT);
            failed = true;
            break;
          }
          tc05_fence_after();
          __syncwarp();
          const float al = exp2f(m - mn);
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tmem_ld32(t_o + c0 + lane_off, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * al);
            tmem_st32(t_o + c0 + lane_off, o);
          }
          tmem_wait_st();
          l *= al;
        }
        m = mn;
      }
      // weights rounded to the input type for the MMA; the running sum takes
      // the fp32 values
      uint32_t pk[kTcTile / 2];
      float l0 = 0.f, l1 = 0.f;
#pragma unroll
      for (int c = 0; c < kTcTile; c += 2) {
        const float p0 = ex2_approx(x[c] - m), p1 = ex2_approx(x[c + 1] - m);
        l0 += p0;
        l1 += p1;
        pk[c / 2] = Mma<T>::pack(p0, p1);
      }
      l += l0 + l1;
      if (i >= 2 &&
          __any_sync(0xffffffffu, !mbar_wait_bounded(&pv_done[i & 1], ((i >> 1) - 1) & 1))) {
        raise_error(p.err, PA_DEVERR_TIMEOUT);
        failed = true;
        break;
      }
      uint8_t* pb = prow + (i & 1) * Ly::PBYTES;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch)
        *reinterpret_cast<uint4*>(pb + ((ch ^ (row_in & 7)) << 4)) =
            make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
      fence_proxy_async_smem();
      tc05_fence_before();
      mbar_arrive(&p_full[i & 1]);
    }
    // ---- the row's partial: O / l, the maximum in natural-log units, l
    if (!failed && __any_sync(0xffffffffu, !mbar_wait_bounded(&pv_done[(ntiles - 1) & 1],
                                                             ((ntiles - 1) >> 1) & 1))) {
      raise_error(p.err, PA_DEVERR_TIMEOUT);
      failed = true;
    }
    tc05_fence_after();
    __syncwarp();
    const int r = qt * kTcRows + row_in;
    if (!failed) {  // warp-uniform
      constexpr float kLn2 = 0.69314718055994530942f;
      const bool mine = r < rows_total;
      const size_t row = mine ? (size_t)(r / G) * Hq + g * G + r % G : 0;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      float* dst = p.tmp_out + (row * p.num_slots + slot) * D;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(t_o + c0 + lane_off, o);
        tmem_wait_ld();
        if (mine) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(dst + c0 + e) =
                make_float4(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv,
                            __uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
        }
      }
      if (mine) {
        p.max_logits[row * p.num_slots + slot] = l > 0.f ? m * kLn2 : -INFINITY;
        p.exp_sums[row * p.num_slots + slot] = l;
      }
    }
  }
  // every TMEM access is done before the columns are released
  tc05_fence_before();
  __syncthreads();
  tc05_fence_after();
  if (warp == 4) {
    __syncwarp();
    tmem_dealloc(tmem, Ly::TMEM_COLS);
  }
}

// Causal prefill over the paged cache: one CTA per (128-row query tile, kv
// head, sequence), eight warps of 16 rows each, every K/V tile staged once
// for all 128 rows. The CTA's rows are (token, head-in-group) pairs of one
// sequence; it streams that sequence's pages from position 0 up to the
// position of its last row, and masks key t for a row at position pos when
// t > pos. Every row sees position 0, so its running maximum is finite from
// the first tile on.
template <typename T, int D>
__global__ void __launch_bounds__(kPrefillThreads, 1)
    prefill_attention_kernel(const __grid_constant__ PrefillParams p) {
  constexpr int CPR = D / 8;
  constexpr int TILE = kPrefixTile;
  constexpr int TBYTES = TILE * D * 2;
  constexpr int KS = D / 16;
  constexpr int NT = TILE / 8;
  constexpr int NO = D / 8;
  static_assert(CPR >= 8, "the swizzle needs 8 chunks per row");
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sq = smem;                         // [128][D]
  uint8_t* sk = smem + kPrefillRows * D * 2;  // [2][TILE][D]
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
  if (qt * kPrefillRows >= rows_total) return;
  T* out = static_cast<T*>(p.out);
  if (n < q_len || n > MB * bs) {  // the chunk does not fit its context: zero rows
    if (reporter) raise_error(p.err, PA_DEVERR_CONTEXT_LEN);
    for (int i = tid; i < kPrefillRows * D; i += kPrefillThreads) {
      const int r = qt * kPrefillRows + i / D;
      if (r < rows_total)
        out[((size_t)(q0 + r / G) * Hq + g * G + r % G) * D + i % D] = Elem<T>::from_f32(0.f);
    }
    return;
  }
  const int pos0 = n - q_len;  // position of the chunk's first token
  const int r_last = min(qt * kPrefillRows + kPrefillRows, rows_total) - 1;
  const int kv_end = pos0 + r_last / G + 1;  // keys this CTA needs: positions [0, kv_end)

  // Q rows of this CTA -> shared memory (rows past the sequence's are zero)
  const uint32_t sq_u = smem_u32(sq), sk_u = smem_u32(sk), sv_u = smem_u32(sv);
  for (int i = tid; i < kPrefillRows * CPR; i += kPrefillThreads) {
    const int rr = i / CPR, c = i % CPR, r = qt * kPrefillRows + rr;
    const bool ok = r < rows_total;
    const size_t row = ok ? (size_t)(q0 + r / G) * Hq + g * G + r % G : 0;
    cp_async16(sq_u + swz<CPR>(rr, c),
               static_cast<const uint8_t*>(p.query) + (row * D + c * 8) * 2, ok);
  }
  const size_t head_stride = (size_t)bs * D * 2;  // bytes of one (block, kv head) page
  const int32_t* table = p.block_tables + (size_t)s * MB;
  auto load_tile = [&](int tile, int buf) {
    const int t0 = tile * TILE;
    for (int i = tid; i < TILE * CPR; i += kPrefillThreads) {
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
  const int rA = qt * kPrefillRows + warp * 16 + (lane >> 2), rB = rA + 8;
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
  const int smem = PrefixTcLayout<D>::SMEM;
  auto kern = prefix_attention_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((p.num_seqs * p.group + kPrefixTcRows - 1) / kPrefixTcRows, p.num_prefix_splits,
                  p.num_kv_heads);
  return launch_pdl(kern, grid, dim3(kTcThreads), smem, st, p);
}

template <typename T, int D>
cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t st) {
  const int smem = kPrefillRows * D * 2 + 4 * kPrefixTile * D * 2;
  auto kern = prefill_attention_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long tiles = ((long long)p.max_q_len * p.group + kPrefillRows - 1) / kPrefillRows;
  const dim3 grid(static_cast<unsigned>(tiles), p.num_kv_heads, p.num_seqs);
  return launch_pdl(kern, grid, dim3(kPrefillThreads), smem, st, p);
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
