// pa_cascade.cu -- attention with many query rows per K/V row on the
// fifth-generation tensor cores (the shared prefix of a cascade decode and
// the paged prefill), and block copies for copy-on-write.
//
// The prefix part of a cascade decode (every K/V row of the shared prefix is
// used by all S * G query rows of its kv head) and a prefill chunk (every K/V
// row of a sequence is used by all of the chunk's rows at or after its
// position) are real dense contractions, so both run tcgen05 MMAs with TMEM
// accumulators on operands staged by tensor copies, flash-attention style;
// see tc05_attention_cta.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "pa_cascade.cuh"
#include "pa_device.cuh"

namespace pa {
namespace {

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

// ---------------------------------------------------------------------------
// Attention of 128 query rows against a run of paged keys on the
// fifth-generation tensor cores (shared by the prefix and prefill kernels).
// Keys [k_begin, k_end) are taken in tiles of 64:
//   S = Q K^T   (M 128 x N 64, K = D)        -> TMEM, two buffers
//   softmax     (one thread per row, lazy running maximum in log2 units)
//   O += P V    (M 128 x N D, K = 64 tokens) -> TMEM
// Q is staged once, K/V tiles of 16-bit caches come by 2-D tensor copies of
// whole pages, P is written to shared memory by the softmax threads; all
// three operands use the 128-byte swizzle. Warps 0-3: softmax (thread t owns
// row t, TMEM lane t); warp 4: MMA issue and TMEM allocation; warp 5: copies.
// An 8-bit cache (INT8 with row scales, or FP8 E4M3) comes by 1-D bulk
// copies of its pages (and INT8 row scales) into a raw ring, and warps 6-9
// widen the codes exactly to f16 into the swizzled K/V tiles (one row per
// thread); q is carried in f16 (exact inside f16's range). INT8: the K row
// scales multiply the logits, the V row scales the weights before they are
// rounded, and the running sum takes the bare weights. E4M3: the callers
// fold k_scale into the logit scale and v_scale into the output. Every wait
// is bounded, and every warp-wide TMEM access is taken by the whole warp.
constexpr int kTcRows = kPrefixTcRows;
constexpr int kTcTile = kPrefixTile;
// Cache kinds of the routine: 16-bit elements (the MMA type), or 8-bit codes
// widened to f16 in shared memory: INT8 with a scale per cached row, or FP8
// E4M3 whose per-tensor scales the callers fold into the logit scale and the
// output.
enum : int { kKc16 = 0, kKcI8 = 1, kKcE4 = 2 };
#ifndef PA_PREFIX_STAGES
#define PA_PREFIX_STAGES 4
#endif

template <int D, bool I8, int QTILES>
struct PrefixTcLayout {
  static constexpr int KB = D / 64;                  // 128-byte column blocks of a row
  // 128-row query tiles per CTA (two share every K/V tile; an INT8 cache's
  // raw ring leaves room for one)
  static constexpr int QTL = QTILES;
  static_assert(QTL == 1 || (QTL == 2 && !I8), "query tiles per CTA");
  static constexpr int ROWS = QTL * kTcRows;          // query rows per CTA
  static constexpr int SMX = 4 * QTL;                 // softmax warps (one thread per row)
  static constexpr int MMA_WARP = SMX, COPY_WARP = SMX + 1, CONV_WARP = SMX + 2;
  static constexpr int THREADS = (SMX + 2 + (I8 ? 4 : 0)) * 32;
  static constexpr int STAGES = I8 ? 3 : (QTL == 2 && D == 128 ? 3 : PA_PREFIX_STAGES);
#ifndef PA_PREFILL_RAW_STAGES
#define PA_PREFILL_RAW_STAGES 3
#endif
  static constexpr int RSTAGES = I8 ? PA_PREFILL_RAW_STAGES : 0;  // raw INT8 tiles
  static constexpr int QBYTES1 = KB * kTcRows * 128;  // one Q tile: [KB][128 rows][128 B]
  static constexpr int QBYTES = QTL * QBYTES1;
  static constexpr int TBYTES = KB * kTcTile * 128;  // one K or V tile: [KB][64 tokens][128 B]
  static constexpr int PBYTES = kTcRows * 128;       // P of one Q tile: [128 rows][64 tokens]
  static constexpr int RAWT = kTcTile * D;           // INT8 codes of one K or V tile
  static constexpr int RAWB = 2 * RAWT + 2 * kTcTile * 4;  // codes + row scales
  static constexpr int OFF_KV = QBYTES;
  static constexpr int OFF_P = OFF_KV + STAGES * 2 * TBYTES;  // [2 buffers][QTL][PBYTES]
  static constexpr int OFF_SC = OFF_P + 2 * QTL * PBYTES;  // INT8: [STAGES][K, V][64] row scales
  static constexpr int OFF_RAW = OFF_SC + (I8 ? STAGES * 2 * kTcTile * 4 : 0);
  static constexpr int OFF_BAR = OFF_RAW + RSTAGES * RAWB;
  static constexpr int NBAR = 2 * STAGES + 8 + (I8 ? 2 * RSTAGES + STAGES : 0);
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;  // + alignment of the base to 1024
  // TMEM columns: S of tile q, buffer b at q 128 + b 64; O of tile q at
  // QTL 128 + q D
  static constexpr uint32_t TMEM_COLS = QTL * (2 * kTcTile + D) <= 256 ? 256 : 512;
  static_assert(QTL * (2 * kTcTile + D) <= 512, "TMEM columns");
  static_assert(OFF_RAW % 16 == 0 && RAWB % 16 == 0 && OFF_BAR % 8 == 0, "alignment");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

// Where the CTA's keys and queries are.
struct Tc05Args {
  const CUtensorMap* tm_k;  // 16-bit caches as [NB Hkv bs rows][D]: boxes of 64 x bs, 128-B swizzle
  const CUtensorMap* tm_v;
  const uint8_t* k_codes;   // INT8 caches [NB][Hkv][bs][D] and row scales [NB][Hkv][bs]
  const uint8_t* v_codes;
  const float* k_scales;
  const float* v_scales;
  const void* q_base;       // any valid query address (source of zero-filling copies)
  int g, Hkv, bs, num_blocks;
  int k_begin, k_end;       // key positions attended (k_begin a multiple of bs)
  int min_pos;              // CAUSAL: the smallest row position of the tile
  float scale_log2;
  unsigned* err;
};

// One CTA's attention. QT is the query type; the MMAs take T = QT (16-bit
// caches) or f16 (INT8). Callbacks:
//   q_row(rr)      the global address of tile row rr's D query elements, or
//                  nullptr (a padding row: zeros)
//   page_block(t)  block id of the page holding key position t (its range is
//                  checked here: a bad id is flagged and reads as zeros)
//   row_pos(rr)    CAUSAL: row rr attends keys <= row_pos(rr)
//   sink(rr, c0, o, inv_l, m_log2, l)   row rr's output columns [c0, c0 + 32)
//                  (un-normalised; times inv_l = 1 / l), called for every
//                  chunk by every softmax thread
//   copy_idle(lane)  side work for the copy warp once its copies are issued
//                  (lanes 1-31 start it while lane 0 is still issuing)
template <typename QT, int D, bool CAUSAL, int KC, int QTILES, typename QRow,
          typename PageBlock, typename RowPos, typename Sink, typename Idle>
__device__ __forceinline__ void tc05_attention_cta(uint8_t* smem, const Tc05Args& a, QRow q_row,
                                                   PageBlock page_block, RowPos row_pos,
                                                   Sink sink, Idle copy_idle) {
  constexpr bool I8 = KC != kKc16;   // 8-bit codes, widened by the converter warps
  constexpr bool ROW_SC = KC == kKcI8;   // with a scale per cached row
  using Ly = PrefixTcLayout<D, I8, QTILES>;
  using T = typename std::conditional<I8, __half, QT>::type;  // MMA operand type
  constexpr int KB = Ly::KB, ST = Ly::STAGES, RS = Ly::RSTAGES, QTL = Ly::QTL, ROWS = Ly::ROWS;
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  uint64_t* kv_full = reinterpret_cast<uint64_t*>(smem + Ly::OFF_BAR);  // [ST] 16-bit: copies done
  uint64_t* kv_empty = kv_full + ST;        // [ST] P V of the tile done
  uint64_t* s_full = kv_empty + ST;         // [2]
  uint64_t* s_free = s_full + 2;            // [2]
  uint64_t* p_full = s_free + 2;            // [2]
  uint64_t* pv_done = p_full + 2;           // [2]
  uint64_t* raw_full = pv_done + 2;         // [RS] INT8: codes and scales landed
  uint64_t* raw_empty = raw_full + RS;      // [RS] INT8: widened
  uint64_t* conv_full = raw_empty + RS;     // [ST] INT8: tile widened into slot
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Ly::OFF_MISC);
  float* sc = reinterpret_cast<float*>(smem + Ly::OFF_SC);  // INT8 row scales of the slots
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ntiles = (a.k_end - a.k_begin + kTcTile - 1) / kTcTile;
  unsigned* err = a.err;

  // ---- set-up: barriers, TMEM, Q rows (asynchronous 16-byte copies, all in
  // flight at once; padding rows zero-filled)
  if (tid == 0) {
    for (int i = 0; i < ST; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
      if (I8) mbar_init(&conv_full[i], kTcRows);
    }
    for (int i = 0; i < RS; ++i) {
      mbar_init(&raw_full[i], 1);
      mbar_init(&raw_empty[i], kTcRows);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], ROWS);
      mbar_init(&p_full[i], ROWS);
      mbar_init(&pv_done[i], 1);
    }
    fence_mbar_init();
  }
  if (warp == Ly::MMA_WARP) {
    __syncwarp();
    tmem_alloc(tmem_slot, Ly::TMEM_COLS);
  }
  const uint32_t sq = smem_u32(smem);
  for (int i = tid; i < ROWS * KB * 8; i += Ly::THREADS) {
    const int rr = i / (KB * 8), c = i % (KB * 8);
    const uint8_t* src = q_row(rr);
    const int q = rr / kTcRows, r1 = rr % kTcRows, kb = c >> 3, ch = c & 7;
    cp_async16(sq + q * Ly::QBYTES1 + kb * (kTcRows * 128) + r1 * 128 + ((ch ^ (r1 & 7)) << 4),
               src ? src + c * 16 : a.q_base, src != nullptr);
  }
  cp_async_commit();
  cp_async_wait<0>();
  if constexpr (I8 && std::is_same<QT, __nv_bfloat16>::value) {
    // q to f16 in place, 16-byte chunk by chunk
    __syncthreads();
    for (int i = tid; i < ROWS * KB * 8; i += Ly::THREADS) {
      uint4* c = reinterpret_cast<uint4*>(smem + 16 * i);
      uint4 v = *c;
      uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w[e]);
        const __half2 h = __floats2half2_rn(__low2float(b), __high2float(b));
        w[e] = *reinterpret_cast<const uint32_t*>(&h);
      }
      *c = v;
    }
  }
  fence_proxy_async_smem();
  tc05_fence_before();
  __syncthreads();
  tc05_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_s = tmem, t_o = tmem + QTL * 2 * kTcTile;  // S of tile q at q 128, O at QTL 128
  bool failed = false;

  if (warp == Ly::COPY_WARP) {
    // ================================================ copies of K/V tiles
    if (lane == 0) {
      const long long rows = (long long)a.num_blocks * a.Hkv * a.bs;
      const int bs = a.bs;
      int issued = 0;
      for (int i = 0; i < ntiles; ++i) {
        const int t0 = a.k_begin + i * kTcTile;
        if constexpr (!I8) {
          const int st = i % ST;
          if (i >= ST && !mbar_wait_bounded(&kv_empty[st], ((i / ST) - 1) & 1)) {
            raise_error(err, PA_DEVERR_TIMEOUT);
            break;
          }
          mbar_arrive_expect_tx(&kv_full[st], 2 * Ly::TBYTES);
          uint8_t* kdst = smem + Ly::OFF_KV + st * 2 * Ly::TBYTES;
          uint8_t* vdst = kdst + Ly::TBYTES;
          for (int pp = 0; pp < kTcTile / bs; ++pp) {
            const int t = t0 + pp * bs;
            // pages past the range and bad block ids read as zeros (a box
            // wholly past the tensor is filled with zeros)
            int y = static_cast<int>(rows);
            if (t < a.k_end) {
              const int b = page_block(t);
              if (b >= 0 && b < a.num_blocks)
                y = (b * a.Hkv + a.g) * bs;
              else
                raise_error(err, PA_DEVERR_BLOCK_ID);
            }
#pragma unroll
            for (int j = 0; j < KB; ++j) {
              tma_load_2d(kdst + j * (kTcTile * 128) + pp * bs * 128, a.tm_k, 64 * j, y,
                          &kv_full[st]);
              tma_load_2d(vdst + j * (kTcTile * 128) + pp * bs * 128, a.tm_v, 64 * j, y,
                          &kv_full[st]);
            }
          }
        } else {
          const int rs = i % RS;
          if (i >= RS && !mbar_wait_bounded(&raw_empty[rs], ((i / RS) - 1) & 1)) {
            raise_error(err, PA_DEVERR_TIMEOUT);
            break;
          }
          // pages past the range or with a bad block id are not copied (the
          // widening writes zeros for their rows)
          uint32_t bytes = 0;
          for (int pp = 0; pp < kTcTile / bs; ++pp) {
            const int t = t0 + pp * bs;
            if (t < a.k_end) {
              const int b = page_block(t);
              if (b >= 0 && b < a.num_blocks)
                bytes += 2u * bs * (D + (ROW_SC ? 4 : 0));
              else
                raise_error(err, PA_DEVERR_BLOCK_ID);
            }
          }
          mbar_arrive_expect_tx(&raw_full[rs], bytes);
          uint8_t* raw = smem + Ly::OFF_RAW + rs * Ly::RAWB;
          for (int pp = 0; pp < kTcTile / bs; ++pp) {
            const int t = t0 + pp * bs;
            if (t >= a.k_end) break;
            const int b = page_block(t);
            if (b < 0 || b >= a.num_blocks) continue;
            const size_t row0 = ((size_t)b * a.Hkv + a.g) * bs;
            bulk_g2s(raw + pp * bs * D, a.k_codes + row0 * D, bs * D, &raw_full[rs]);
            bulk_g2s(raw + Ly::RAWT + pp * bs * D, a.v_codes + row0 * D, bs * D, &raw_full[rs]);
            if constexpr (ROW_SC) {
              bulk_g2s(raw + 2 * Ly::RAWT + pp * bs * 4, a.k_scales + row0, bs * 4,
                       &raw_full[rs]);
              bulk_g2s(raw + 2 * Ly::RAWT + kTcTile * 4 + pp * bs * 4, a.v_scales + row0, bs * 4,
                       &raw_full[rs]);
            }
          }
        }
        ++issued;
      }
      // never leave with copies in flight
      constexpr int NB_ = I8 ? RS : ST;
      uint64_t* done = I8 ? raw_full : kv_full;
      for (int k = issued > NB_ ? issued - NB_ : 0; k < issued; ++k)
        if (!mbar_wait_bounded(&done[k % NB_], (k / NB_) & 1)) raise_error(err, PA_DEVERR_TIMEOUT);
    }
    copy_idle(lane);
  } else if (warp >= Ly::CONV_WARP) {
    // ================================================ 8-bit codes: widening to f16
    if constexpr (I8) {
      const int cid = tid - Ly::CONV_WARP * 32;  // 0 .. 127
      const int row = cid & (kTcTile - 1);
      const bool is_v = cid >= kTcTile;
      for (int i = 0; i < ntiles; ++i) {
        const int rs = i % RS, st = i % ST;
        if (!mbar_wait_bounded(&raw_full[rs], (i / RS) & 1) ||
            (i >= ST && !mbar_wait_bounded(&kv_empty[st], ((i / ST) - 1) & 1))) {
          raise_error(err, PA_DEVERR_TIMEOUT);
          break;
        }
        const int t = a.k_begin + i * kTcTile + row;
        bool ok = t < a.k_end;
        if (ok) {
          const int b = page_block(t);
          ok = b >= 0 && b < a.num_blocks;
        }
        const uint8_t* raw = smem + Ly::OFF_RAW + rs * Ly::RAWB;
        const uint8_t* src = raw + (is_v ? Ly::RAWT : 0) + row * D;
        uint8_t* dst = smem + Ly::OFF_KV + st * 2 * Ly::TBYTES + (is_v ? Ly::TBYTES : 0);
#pragma unroll
        for (int k = 0; k < KB * 8; ++k) {
          const int c = (k + row) & (KB * 8 - 1);  // rotated: rows of a warp hit different banks
          uint4 out = make_uint4(0u, 0u, 0u, 0u);
          if (ok) {
            const uint2 w = *reinterpret_cast<const uint2*>(src + 8 * c);
            using Code = typename std::conditional<ROW_SC, ::pa::I8, E4M3>::type;
            widen8<Code>(w.x, out.x, out.y);
            widen8<Code>(w.y, out.z, out.w);
          }
          const int kb = c >> 3, ch = c & 7;
          *reinterpret_cast<uint4*>(dst + kb * (kTcTile * 128) + row * 128 +
                                    ((ch ^ (row & 7)) << 4)) = out;
        }
        if constexpr (ROW_SC)
          sc[(st * 2 + (is_v ? 1 : 0)) * kTcTile + row] =
              ok ? reinterpret_cast<const float*>(raw + 2 * Ly::RAWT)[(is_v ? kTcTile : 0) + row]
                 : 0.f;
        fence_proxy_async_smem();
        mbar_arrive(&conv_full[st]);
        mbar_arrive(&raw_empty[rs]);
      }
    }
  } else if (warp == Ly::MMA_WARP) {
    // ================================================ MMA issue (one thread)
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc_f16(kBf16, kTcRows, kTcTile, false);
      constexpr uint32_t idesc_o = umma_idesc_f16(kBf16, kTcRows, D, true);
      const uint32_t skv = smem_u32(smem + Ly::OFF_KV), sp = smem_u32(smem + Ly::OFF_P);
      uint64_t* ready = I8 ? conv_full : kv_full;
      auto issue_s = [&](int i) -> bool {
        const int st = i % ST;
        if (!mbar_wait_bounded(&ready[st], (i / ST) & 1)) return false;
        if (i >= 2 && !mbar_wait_bounded(&s_free[i & 1], ((i >> 1) - 1) & 1)) return false;
        tc05_fence_after();
        const uint32_t kt = skv + st * 2 * Ly::TBYTES;
#pragma unroll
        for (int q = 0; q < QTL; ++q)
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t qa = sq + q * Ly::QBYTES1 + (kk >> 2) * (kTcRows * 128) + (kk & 3) * 32;
            const uint32_t kbd = kt + (kk >> 2) * (kTcTile * 128) + (kk & 3) * 32;
            umma_f16(t_s + q * 2 * kTcTile + (i & 1) * kTcTile, umma_sdesc_sw128(qa, 16, 1024),
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
        const uint32_t vt = skv + (i % ST) * 2 * Ly::TBYTES + Ly::TBYTES;
#pragma unroll
        for (int q = 0; q < QTL; ++q) {
          const uint32_t pa = sp + ((i & 1) * QTL + q) * Ly::PBYTES;
#pragma unroll
          for (int kk = 0; kk < kTcTile / 16; ++kk)
            umma_f16(t_o + q * D, umma_sdesc_sw128(pa + kk * 32, 16, 1024),
                     umma_sdesc_sw128(vt + kk * 2048, kTcTile * 128, 1024), idesc_o,
                     i > 0 || kk > 0);
        }
        umma_commit(&pv_done[i & 1]);
        if (i + ST < ntiles) umma_commit(&kv_empty[i % ST]);  // a later tile refills it
      }
      if (!ok) raise_error(err, PA_DEVERR_TIMEOUT);
    }
  } else {
    // ================================================ softmax, one row per thread
    // (tcgen05.ld / st are warp-wide: every decision that leads to one is
    // taken by the whole warp)
    const int rr = tid;             // the CTA's row
    const int q = rr / kTcRows;     // its query tile
    const int r1 = rr % kTcRows;    // its TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_sq = t_s + q * 2 * kTcTile, t_oq = t_o + q * D;
    constexpr float kLazy = 8.f;
    const int my_pos = CAUSAL ? row_pos(rr) : 0;
    float m = -INFINITY, l = 0.f;
    uint8_t* prow = smem + Ly::OFF_P + q * Ly::PBYTES + r1 * 128;
    for (int i = 0; i < ntiles; ++i) {
      if (__any_sync(0xffffffffu, !mbar_wait_bounded(&s_full[i & 1], (i >> 1) & 1))) {
        raise_error(err, PA_DEVERR_TIMEOUT);
        failed = true;
        break;
      }
      tc05_fence_after();
      __syncwarp();
      uint32_t sr[2][32];
      tmem_ld32(t_sq + (i & 1) * kTcTile + lane_off, sr[0]);
      tmem_ld32(t_sq + (i & 1) * kTcTile + 32 + lane_off, sr[1]);
      tmem_wait_ld();
      tc05_fence_before();
      mbar_arrive(&s_free[i & 1]);
      // logits in log2 units; keys past the range (a partial last tile) and,
      // causally, past the row's position (tiles that reach the diagonal)
      // are -inf
      const int t0 = a.k_begin + i * kTcTile;
      const int valid = a.k_end - t0;  // >= 1
      const float* ksc = sc + (i % ST) * 2 * kTcTile;  // INT8: the tile's K, then V row scales
      if constexpr (I8) {
        // the scales were written by the widening threads of this slot
        if (__any_sync(0xffffffffu, !mbar_wait_bounded(&conv_full[i % ST], (i / ST) & 1))) {
          raise_error(err, PA_DEVERR_TIMEOUT);
          failed = true;
          break;
        }
      }
      float x[kTcTile];
#pragma unroll
      for (int c = 0; c < kTcTile; ++c) {
        x[c] = __uint_as_float(sr[c >> 5][c & 31]) * a.scale_log2;
        if constexpr (ROW_SC) x[c] *= ksc[c];
      }
      if (valid < kTcTile || (CAUSAL && t0 + kTcTile - 1 > a.min_pos)) {  // CTA-uniform
        const int lim = CAUSAL ? min(valid, my_pos - t0 + 1) : valid;
#pragma unroll
        for (int c = 0; c < kTcTile; ++c) x[c] = c < lim ? x[c] : -INFINITY;
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
            raise_error(err, PA_DEVERR_TIMEOUT);
            failed = true;
            break;
          }
          tc05_fence_after();
          __syncwarp();
          const float al = mn == -INFINITY ? 1.f : exp2f(m - mn);
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tmem_ld32(t_oq + c0 + lane_off, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * al);
            tmem_st32(t_oq + c0 + lane_off, o);
          }
          tmem_wait_st();
          l *= al;
        }
        m = mn;
      }
      // weights rounded to the MMA type (INT8: times the V row scale first);
      // the running sum takes the fp32 weights
      uint32_t pk[kTcTile / 2];
      float l0 = 0.f, l1 = 0.f;
#pragma unroll
      for (int c = 0; c < kTcTile; c += 2) {
        const float p0 = ex2_approx(x[c] - m), p1 = ex2_approx(x[c + 1] - m);
        l0 += p0;
        l1 += p1;
        if constexpr (ROW_SC)
          pk[c / 2] = Mma<T>::pack(p0 * ksc[kTcTile + c], p1 * ksc[kTcTile + c + 1]);
        else
          pk[c / 2] = Mma<T>::pack(p0, p1);
      }
      l += l0 + l1;
      if (i >= 2 &&
          __any_sync(0xffffffffu, !mbar_wait_bounded(&pv_done[i & 1], ((i >> 1) - 1) & 1))) {
        raise_error(err, PA_DEVERR_TIMEOUT);
        failed = true;
        break;
      }
      uint8_t* pb = prow + (i & 1) * QTL * Ly::PBYTES;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch)
        *reinterpret_cast<uint4*>(pb + ((ch ^ (r1 & 7)) << 4)) =
            make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
      if (!I8 && valid < kTcTile) {  // CTA-uniform
        // V rows past the range may hold anything (rows past a context can
        // be NaN), and a zero weight times NaN is NaN in the MMA: zero them
        // (the INT8 widening writes zeros for them already)
        uint8_t* vt = smem + Ly::OFF_KV + (i % ST) * 2 * Ly::TBYTES + Ly::TBYTES;
        for (int c = rr; c < (kTcTile - valid) * KB * 8; c += ROWS) {
          const int row = valid + c / (KB * 8), kb = (c / 8) % KB, ch = c % 8;
          *reinterpret_cast<uint4*>(vt + kb * (kTcTile * 128) + row * 128 + ch * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();
      tc05_fence_before();
      mbar_arrive(&p_full[i & 1]);
    }
    // ---- the row's output, chunk by chunk
    if (!failed && __any_sync(0xffffffffu, !mbar_wait_bounded(&pv_done[(ntiles - 1) & 1],
                                                             ((ntiles - 1) >> 1) & 1))) {
      raise_error(err, PA_DEVERR_TIMEOUT);
      failed = true;
    }
    tc05_fence_after();
    __syncwarp();
    if (!failed) {  // warp-uniform
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(t_oq + c0 + lane_off, o);
        tmem_wait_ld();
        sink(rr, c0, o, inv, m, l);
      }
    }
  }
  // every TMEM access is done before the columns are released
  tc05_fence_before();
  __syncthreads();
  tc05_fence_after();
  if (warp == Ly::MMA_WARP) {
    __syncwarp();
    tmem_dealloc(tmem, Ly::TMEM_COLS);
  }
}

// Shared-prefix attention: a CTA takes 128 query rows (all sequences' query
// heads of one kv head, row r = s G + h) and one range of the prefix (the
// prefix's block ids from row 0 of the block tables), and writes the rows'
// partials (normalised output, maximum in natural-log units, sum) to its
// slot for pa_reduce.
template <typename T, int D, int KC>
__global__ void __launch_bounds__(PrefixTcLayout<D, KC != kKc16, 1>::THREADS, 1)
    prefix_attention_kernel(const __grid_constant__ PrefixParams p) {
  using Ly = PrefixTcLayout<D, KC != kKc16, 1>;
  constexpr int NT = Ly::THREADS, ROWS = Ly::ROWS;
  static_assert(ROWS == kPrefixCtaRows, "the host's plan counts rows per CTA");
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x;
  const int qt = blockIdx.x, split = blockIdx.y, g = blockIdx.z;
  const int S = p.num_seqs, Hq = p.num_heads, G = p.group;
  const int rows_total = S * G;
  const int t_begin = split * p.tokens_per_split;
  const int t_end = min(p.prefix_tokens, t_begin + p.tokens_per_split);
  const int slot = p.slot0 + split;

  // the precondition, checked on a slice per CTA by n threads: every row's
  // first prefix_pages entries equal row 0's, and every context covers the
  // prefix (off the critical path: by the copy warp once its copies are out)
  auto check = [&](int t, int n) {
    const int cta = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
    const int nctas = gridDim.x * gridDim.y * gridDim.z;
    for (int s = 1 + cta; s < S; s += nctas)
      for (int i = t; i < p.prefix_pages; i += n)
        if (p.block_tables[(size_t)s * p.max_blocks_per_seq + i] != p.block_tables[i])
          raise_error(p.err, PA_DEVERR_BLOCK_ID);
    for (int s = cta * n + t; s < S; s += nctas * n)
      if (p.context_lens[s] < p.prefix_tokens) raise_error(p.err, PA_DEVERR_CONTEXT_LEN);
  };
  if (t_begin >= t_end) {  // a split with no prefix token: empty partials
    check(tid, NT);
    for (int i = tid; i < ROWS; i += NT) {
      const int r = qt * ROWS + i;
      if (r < rows_total) {
        const size_t row = (size_t)(r / G) * Hq + g * G + r % G;
        p.max_logits[row * p.num_slots + slot] = -INFINITY;
        p.exp_sums[row * p.num_slots + slot] = 0.f;
      }
    }
    return;
  }
  auto row_of = [&](int rr) -> long long {
    const int r = qt * ROWS + rr;
    return r < rows_total ? (long long)(r / G) * Hq + g * G + r % G : -1;
  };
  auto q_row = [&](int rr) -> const uint8_t* {
    const long long row = row_of(rr);
    return row < 0 ? nullptr : static_cast<const uint8_t*>(p.query) + row * D * 2;
  };
  auto page_block = [&](int t) -> int { return __ldg(p.block_tables + t / p.block_size); };
  auto row_pos = [&](int) -> int { return 0; };
  auto sink = [&](int rr, int c0, const uint32_t(&o)[32], float inv, float m, float l) {
    const long long row = row_of(rr);
    if (row < 0) return;
    float* dst = p.tmp_out + ((size_t)row * p.num_slots + slot) * D + c0;
    if (KC == kKcE4) inv *= p.v_scale;
#pragma unroll
    for (int e = 0; e < 32; e += 4)
      *reinterpret_cast<float4*>(dst + e) =
          make_float4(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv,
                      __uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
    if (c0 == 0) {
      constexpr float kLn2 = 0.69314718055994530942f;
      p.max_logits[(size_t)row * p.num_slots + slot] = l > 0.f ? m * kLn2 : -INFINITY;
      p.exp_sums[(size_t)row * p.num_slots + slot] = l;
    }
  };
  Tc05Args a{};
  a.tm_k = &p.tm_k;
  a.tm_v = &p.tm_v;
  a.q_base = p.query;
  a.g = g;
  a.Hkv = p.num_kv_heads;
  a.bs = p.block_size;
  a.num_blocks = p.num_blocks;
  a.k_begin = t_begin;
  a.k_end = t_end;
  a.min_pos = 0;
  a.scale_log2 = p.scale_log2;
  a.err = p.err;
  a.k_codes = p.k_cache;
  a.v_codes = p.v_cache;
  a.k_scales = p.k_scales;
  a.v_scales = p.v_scales;
  tc05_attention_cta<T, D, false, KC, 1>(smem, a, q_row, page_block, row_pos, sink,
                                            [&](int lane) { check(lane, 32); });
}

// Causal prefill over the paged cache on the tensor cores: one CTA per
// (query tile of 256 rows, 128 with an INT8 cache; kv head; sequence). The CTA's rows are (token,
// head-in-group) pairs r = i G + j of one sequence's chunk, token i at
// position n - q_len + i; it streams that sequence's pages from position 0 to
// one past its last row's position (kv_end) and masks key t for a row at
// position pos when t > pos. Every row sees position 0, so its running
// maximum is finite from the first tile on. Rows past the chunk's take the
// tile's last position (finite values that are never stored). KC: the
// cache's kind (16-bit elements, INT8 codes and row scales, or E4M3 codes).
template <typename QT, int D, int KC>
__global__ void __launch_bounds__(PrefixTcLayout<D, KC != kKc16, KC != kKc16 ? 1 : 2>::THREADS, 1)
    prefill_tc_kernel(const __grid_constant__ PrefillParams p) {
  using Ly = PrefixTcLayout<D, KC != kKc16, KC != kKc16 ? 1 : 2>;
  constexpr int NT = Ly::THREADS, ROWS = Ly::ROWS;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x;
  const int qt = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int Hq = p.num_heads, G = p.group, bs = p.block_size;
  const int MB = p.max_blocks_per_seq;
  const bool reporter = qt == 0 && g == 0 && tid == 0;  // flags a sequence's errors once

  // this sequence's query tokens [q0, q0 + q_len) and context of n tokens
  const int q0 = p.cu_q[s];
  const int q_len = p.cu_q[s + 1] - q0;
  const int n = p.context_lens[s];
  if (q_len < 0 || q0 < 0 || q0 > p.num_tokens - max(q_len, 0) || q_len > p.max_q_len) {
    if (reporter) raise_error(p.err, PA_DEVERR_SEQ);
    return;  // offsets that do not fit the batch: nothing of this sequence is written
  }
  const int rows_total = q_len * G;
  if (qt * ROWS >= rows_total) return;
  QT* out = static_cast<QT*>(p.out);
  if (n < q_len || n > MB * bs) {  // the chunk does not fit its context: zero rows
    if (reporter) raise_error(p.err, PA_DEVERR_CONTEXT_LEN);
    for (int i = tid; i < ROWS * D; i += NT) {
      const int r = qt * ROWS + i / D;
      if (r < rows_total)
        out[((size_t)(q0 + r / G) * Hq + g * G + r % G) * D + i % D] = Elem<QT>::from_f32(0.f);
    }
    return;
  }
  const int pos0 = n - q_len;  // position of the chunk's first token
  const int r_first = qt * ROWS;
  const int r_last = min(r_first + ROWS, rows_total) - 1;
  const int kv_end = pos0 + r_last / G + 1;  // keys this CTA needs: positions [0, kv_end)
  const int32_t* table = p.block_tables + (size_t)s * MB;
  auto q_row = [&](int rr) -> const uint8_t* {
    const int r = r_first + rr;
    return r < rows_total ? static_cast<const uint8_t*>(p.query) +
                                ((size_t)(q0 + r / G) * Hq + g * G + r % G) * D * 2
                          : nullptr;
  };
  auto page_block = [&](int t) -> int { return __ldg(table + t / bs); };
  auto row_pos = [&](int rr) -> int {
    const int r = r_first + rr;
    return r < rows_total ? pos0 + r / G : kv_end - 1;
  };
  auto sink = [&](int rr, int c0, const uint32_t(&o)[32], float inv, float, float) {
    const int r = r_first + rr;
    if (r >= rows_total) return;
    QT* dst = out + ((size_t)(q0 + r / G) * Hq + g * G + r % G) * D + c0;
    if (KC == kKcE4) inv *= p.v_scale;
#pragma unroll
    for (int e = 0; e < 32; e += 8) {
      uint4 v;
      v.x = Mma<QT>::pack(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
      v.y = Mma<QT>::pack(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
      v.z = Mma<QT>::pack(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
      v.w = Mma<QT>::pack(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
      *reinterpret_cast<uint4*>(dst + e) = v;
    }
  };
  Tc05Args a{};
  a.tm_k = &p.tm_k;
  a.tm_v = &p.tm_v;
  a.k_codes = p.k_cache;
  a.v_codes = p.v_cache;
  a.k_scales = p.k_scales;
  a.v_scales = p.v_scales;
  a.q_base = p.query;
  a.g = g;
  a.Hkv = p.num_kv_heads;
  a.bs = bs;
  a.num_blocks = p.num_blocks;
  a.k_begin = 0;
  a.k_end = kv_end;
  a.min_pos = pos0 + r_first / G;
  a.scale_log2 = p.scale_log2;
  a.err = p.err;
  tc05_attention_cta<QT, D, true, KC, KC != kKc16 ? 1 : 2>(smem, a, q_row, page_block, row_pos,
                                                           sink, [](int) {});
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

template <typename T, int D, int KC>
cudaError_t launch_prefix(const PrefixParams& p, cudaStream_t st) {
  using Ly = PrefixTcLayout<D, KC != kKc16, 1>;
  auto kern = prefix_attention_kernel<T, D, KC>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::SMEM);
  if (e != cudaSuccess) return e;
  const dim3 grid((p.num_seqs * p.group + Ly::ROWS - 1) / Ly::ROWS, p.num_prefix_splits,
                  p.num_kv_heads);
  return launch_pdl(kern, grid, dim3(Ly::THREADS), Ly::SMEM, st, p);
}

template <typename QT, int D, int KC>
cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t st) {
  using Ly = PrefixTcLayout<D, KC != kKc16, KC != kKc16 ? 1 : 2>;
  auto kern = prefill_tc_kernel<QT, D, KC>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::SMEM);
  if (e != cudaSuccess) return e;
  const long long tiles = ((long long)p.max_q_len * p.group + Ly::ROWS - 1) / Ly::ROWS;
  const dim3 grid(static_cast<unsigned>(tiles), p.num_kv_heads, p.num_seqs);
  return launch_pdl(kern, grid, dim3(Ly::THREADS), Ly::SMEM, st, p);
}

}  // namespace

// kind: the cache's (0 = the query's 16-bit type, 1 = INT8 codes and row
// scales, 2 = FP8 E4M3 codes); head dims 64 and 128, queries bf16 or f16.
#define PA_TC05_DISPATCH(LAUNCH, P)                                      \
  do {                                                                   \
    const int d_ = (P).head_dim;                                         \
    if (d_ != 64 && d_ != 128) return cudaErrorInvalidValue;             \
    if (dtype != PA_BF16 && dtype != PA_F16) return cudaErrorInvalidValue; \
    if (kind < 0 || kind > 2) return cudaErrorInvalidValue;              \
    const int i_ = (dtype == PA_BF16 ? 0 : 6) + (d_ == 64 ? 0 : 3) + kind; \
    switch (i_) {                                                        \
      case 0: return LAUNCH<__nv_bfloat16, 64, kKc16>(P, st);            \
      case 1: return LAUNCH<__nv_bfloat16, 64, kKcI8>(P, st);            \
      case 2: return LAUNCH<__nv_bfloat16, 64, kKcE4>(P, st);            \
      case 3: return LAUNCH<__nv_bfloat16, 128, kKc16>(P, st);           \
      case 4: return LAUNCH<__nv_bfloat16, 128, kKcI8>(P, st);           \
      case 5: return LAUNCH<__nv_bfloat16, 128, kKcE4>(P, st);           \
      case 6: return LAUNCH<__half, 64, kKc16>(P, st);                   \
      case 7: return LAUNCH<__half, 64, kKcI8>(P, st);                   \
      case 8: return LAUNCH<__half, 64, kKcE4>(P, st);                   \
      case 9: return LAUNCH<__half, 128, kKc16>(P, st);                  \
      case 10: return LAUNCH<__half, 128, kKcI8>(P, st);                 \
      default: return LAUNCH<__half, 128, kKcE4>(P, st);                 \
    }                                                                    \
  } while (0)

cudaError_t launch_prefix_attention(const PrefixParams& p, int dtype, int kind, cudaStream_t st) {
  PA_TC05_DISPATCH(launch_prefix, p);
}

cudaError_t launch_prefill_attention(const PrefillParams& p, int dtype, int kind,
                                     cudaStream_t st) {
  PA_TC05_DISPATCH(launch_prefill, p);
}
#undef PA_TC05_DISPATCH

cudaError_t launch_copy_blocks(uint8_t* k_cache, uint8_t* v_cache, const int32_t* block_pairs,
                               int num_pairs, int num_blocks, size_t block_bytes, unsigned* err,
                               cudaStream_t st) {
  if (num_pairs <= 0) return cudaSuccess;
  return launch_pdl(copy_blocks_kernel, dim3(num_pairs, 2), dim3(256), 0, st, k_cache, v_cache,
                    block_pairs, num_blocks, block_bytes, err);
}

}  // namespace pa
