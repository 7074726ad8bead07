// pa_decode.cuh -- paged decode attention kernels for sm_103a.
//
// What they compute ("PagedAttention in mistral.rs": blocked K/V pool read
// through per-sequence block tables, optional FP8 E4M3 cache; "Rolling buffer
// cache": a window of W ring slots): for sequence s, kv head g and the G query
// heads sharing it, softmax(q K^T * scale) V over the attended slots [0, L_s).
//
// Work is cut into "pieces": a run of consecutive pages of one (sequence,
// kv head) "segment". Two ways of cutting:
//  * split mode: grid (splits, kv heads, seqs); CTA (i, g, s) takes pages
//    [i*P, (i+1)*P) of segment (s, g) and writes the final output (one
//    split) or the split's partial (m, l, o) for pa_reduce.
//  * balanced mode: a persistent grid of C CTAs (the resident capacity).
//    The pages of all segments, in (sequence, kv head, page) order, are cut
//    into C equal contiguous ranges; each CTA streams its range without a
//    break, crossing segment boundaries. A segment lying wholly inside one
//    range is finished by that CTA; a segment cut by range boundaries leaves
//    a partial in each CTA it touches (at most two per CTA: its first and
//    its last piece). A CTA publishes such a partial, then adds its page
//    count to the segment's arrival counter; the CTA that completes the
//    count combines the segment's partials and writes the output. No CTA
//    waits for another, so nothing depends on the CTAs being co-resident.
//
// CTA structure (both modes):
//  * producer warp (last warp): walks the CTA's pages; per page it issues 1-D
//    bulk asynchronous copies (K page, V page: bs*D contiguous elements of the
//    head-major layout; plus the G query rows at the first page of a piece)
//    into a ring of STAGES shared-memory stages, and writes the stage's
//    descriptor (attended rows, segment, first/last-of-piece flags). Stage
//    completion is tracked by "full" mbarriers (expect-tx), reuse by "empty"
//    mbarriers.
//  * NC = bs/8 consumer warps, 8 rows of every page each, R pages per
//    iteration. A lane covers EPL elements of a row in PB-byte pieces
//    interleaved across the row's LPR lanes (each shared-memory load
//    instruction of a row reads contiguous bytes). Per iteration:
//       1. partial q.k dot products as fp32 pairs (packed FMA), reduced
//          across the row's lanes by a transposing butterfly (each level
//          halves the values a lane keeps: ~1 shuffle per (token, head));
//       2. softmax weights 2^(s - m) against a lazy running max m (log2
//          units; q pre-scaled by scale*log2(e)*k_scale): m moves, with a
//          rescale, only when a logit clears it by 2^8;
//       3. P.V into fp32 pair accumulators; rows past L_s are skipped, never
//          weighted, so stale or NaN cache rows cannot reach the output.
//     At the end of a piece the warps merge (m, l, acc) through the piece's
//     last stage (reused as scratch before it is released) and store.
//  * tensor-core consumers (16-bit cache read with queries of the same type,
//    G >= 4, head_dim 64 or 128): the pages are staged by 2-D tensor copies
//    with the 128-byte swizzle, and each consumer warp takes 16 rows of a
//    page per iteration: S = Q K^T and O += P V as m16n8k16 MMAs
//    with the G query rows of the kv head as the m16 rows (the rest zero),
//    K and V fragments read by ldmatrix (conflict-free on the swizzled
//    layout), the softmax weights P rounded to the cache type (as the MMA
//    takes them) and the running sum taken over those rounded weights.
//  * 8-bit tensor-core consumers (FP8 E4M3 or INT8 cache, 16-bit queries,
//    any G up to 8): each consumer warp takes two 16-row slices per
//    iteration; the cached rows are the m16 rows of the MMAs and the query
//    heads the n8 columns (S^T = K Q^T, O^T = V^T P^T), the codes widened
//    exactly to f16 in registers (see process_tc8).
// Every K/V byte is read from HBM once per kv head. All waits are bounded.
#pragma once

#include <cuda.h>

#include "pa_device.cuh"

namespace pa {

// Shared-memory budget for one CTA's K/V stages, and the most pages a
// consumer warp takes per iteration (build-time tunables).
#ifndef PA_STAGE_BYTES
#define PA_STAGE_BYTES 65536
#endif
#ifndef PA_PAGES_PER_ITER
#define PA_PAGES_PER_ITER 2
#endif
#ifndef PA_MAX_STAGES
#define PA_MAX_STAGES 8
#endif
// Fewest lanes a cached row is spread over, and the register budget per
// thread planned for more than two query heads per kv head (build-time
// tunables).
#ifndef PA_LPR_MIN
#define PA_LPR_MIN 4
#endif
#ifndef PA_REG_BUDGET_WIDE
#define PA_REG_BUDGET_WIDE 128
#endif

// Tensor-core consumers on or off, the smallest group they serve, and the
// shared-memory budget of their stages (build-time tunables).
#ifndef PA_DECODE_TC
#define PA_DECODE_TC 1
#endif
#ifndef PA_TC_MIN_GROUP
#define PA_TC_MIN_GROUP 4
#endif
#ifndef PA_TC_STAGE_BYTES
#define PA_TC_STAGE_BYTES 105000
#endif
// split mode (one CTA per (split, kv head, sequence), usually a few pages
// each): smaller rings, so more CTAs are resident and start at once
#ifndef PA_TC_SPLIT_STAGE_BYTES
#define PA_TC_SPLIT_STAGE_BYTES 52000
#endif
#ifndef PA_TC_WARPS
#define PA_TC_WARPS 4
#endif
// 8-bit caches (FP8 E4M3, INT8) on the tensor cores, any group size up to 8
// (off = the CUDA-core consumers), their consumer warps, the 16-row slices
// each warp takes per iteration, and their stage budgets (FP8: five CTAs per
// SM at head_dim 96; INT8, whose stages also carry row scales: four) and most
// stages (build-time tunables).
#ifndef PA_DECODE_TC8
#define PA_DECODE_TC8 1
#endif
#ifndef PA_TC8_WARPS
#define PA_TC8_WARPS 2
#endif
#ifndef PA_TC8_SLICES
#define PA_TC8_SLICES 2
#endif
#ifndef PA_TC8_STAGE_BYTES
#define PA_TC8_STAGE_BYTES 40000
#endif
#ifndef PA_TC8_I8_STAGE_BYTES
#define PA_TC8_I8_STAGE_BYTES 52000
#endif
#ifndef PA_TC8_MAX_STAGES
#define PA_TC8_MAX_STAGES 16
#endif

enum : int { kModeSplit = 0, kModeBalanced = 1 };

// Which consumers a (query type, cache type, head_dim, group bucket, block
// size) instantiation runs, asked with the C ABI's type codes so that the
// host side can ask the same questions:
//  * tc16_eligible: a 16-bit cache read with queries of the same type, head
//    dim 64 or 128, G >= PA_TC_MIN_GROUP (MMAs with the query heads as rows);
//  * tc8_eligible: an 8-bit cache (FP8 or INT8) read with 16-bit queries, any
//    G up to 8 (MMAs with the cached rows as rows);
//  * tma_staged: the pages are staged by 2-D tensor copies with the 128-byte
//    swizzle (the host builds tensor maps for exactly these): the 16-bit
//    tensor-core consumers, and the 8-bit ones at head_dim 128, where a row
//    is one 128-byte swizzle row.
constexpr bool tc16_eligible(int q_dtype, int kv_dtype, int D, int GT, int BS) {
  return PA_DECODE_TC != 0 && (q_dtype == PA_BF16 || q_dtype == PA_F16) &&
         kv_dtype == PA_KV_AUTO && (D == 64 || D == 128) && GT >= PA_TC_MIN_GROUP && BS >= 16 &&
         BS <= 64;
}
constexpr bool tc8_eligible(int q_dtype, int kv_dtype, int D, int GT, int BS) {
  return PA_DECODE_TC8 != 0 && (q_dtype == PA_BF16 || q_dtype == PA_F16) &&
         (kv_dtype == PA_KV_FP8_E4M3 || kv_dtype == PA_KV_INT8) && D % 32 == 0 && D <= 128 &&
         GT <= 8 && BS >= 16 && BS <= 64 && BS % 16 == 0;
}
constexpr bool tma_staged(int q_dtype, int kv_dtype, int D, int GT, int BS) {
  return tc16_eligible(q_dtype, kv_dtype, D, GT, BS) ||
         (tc8_eligible(q_dtype, kv_dtype, D, GT, BS) && D == 128);
}
template <typename T>
struct DtypeCode {
  static constexpr int value = -1;
};
template <>
struct DtypeCode<__nv_bfloat16> {
  static constexpr int value = PA_BF16;
};
template <>
struct DtypeCode<__half> {
  static constexpr int value = PA_F16;
};
template <typename CT>
struct KvCode {
  static constexpr int value = PA_KV_AUTO;
};
template <>
struct KvCode<E4M3> {
  static constexpr int value = PA_KV_FP8_E4M3;
};
template <>
struct KvCode<I8> {
  static constexpr int value = PA_KV_INT8;
};
template <typename QT, typename CT, int D, int GT, int BS>
constexpr bool uses_tc() {
  return std::is_same<QT, CT>::value && DtypeCode<QT>::value >= 0 &&
         tc16_eligible(DtypeCode<QT>::value, PA_KV_AUTO, D, GT, BS);
}
template <typename QT, typename CT, int D, int GT, int BS>
constexpr bool uses_tc8() {
  return DtypeCode<QT>::value >= 0 && KvCode<CT>::value != PA_KV_AUTO &&
         tc8_eligible(DtypeCode<QT>::value, KvCode<CT>::value, D, GT, BS);
}

// Stage-descriptor flags.
enum : int {
  kFirst = 1,      // first page of a piece (its stage also carries the q rows)
  kLast = 2,       // last page of a piece
  kCtaLast = 4,    // last page of the CTA's work
  kSegFirst = 8,   // the piece starts at page 0 of its segment
  kSegLast = 16,   // the piece ends at the segment's last page
  kSlot1 = 32      // balanced mode: the piece is stored in partial slot 1
};

// Balanced mode: partial slots per CTA and the most CTAs a workspace is
// sized for (152 SMs x 6 resident CTAs).
constexpr int kPieceSlots = 2;
constexpr int kMaxBalancedCtas = 152 * 6;

struct DecodeParams {
  // tensor-core consumers: the K and V caches as 2-D tensors of
  // [NB * Hkv * bs rows][D elements], boxes of 64 elements x bs rows with the
  // 128-byte swizzle (one box per 64 columns of a page)
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  // outputs
  void* out;            // [S][Hq][D] of QT
  float* tmp_out;       // split mode partials: [S][Hq][NS][D]
  float* max_logits;    // [S][Hq][NS]
  float* exp_sums;      // [S][Hq][NS]
  float* piece_o;       // balanced mode: [C][2][GT][D]
  float* piece_ml;      // [C][2][GT][2]: max logit (natural log), sum relative to it
  int* arrived;         // [C]: pages of a cut segment whose pieces are published,
                        // at the CTA holding the segment's last page (zero at launch)
  // inputs
  const void* query;    // [S][Hq][D] of QT
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const float* k_scales;        // INT8 cache: one scale per cached row, [NB][Hkv][bs]
  const float* v_scales;
  const int32_t* block_tables;  // [S][MB]
  const int32_t* context_lens;  // [S]
  unsigned* err;
  int num_seqs, num_heads, num_kv_heads, group;  // group = G (runtime, <= GT)
  int num_blocks, max_blocks_per_seq, window;
  int num_splits, pages_per_split;  // split mode
  int first_page;  // split mode: pages of every context before the splits (a shared prefix)
  // split mode: start without waiting for the previous launch on the stream
  // and wait for it at the end instead (the previous launch reads nothing
  // this one writes and has itself waited for everything before it)
  int join_at_end;
  int partials;   // split mode: 1 = write split partials, 0 = final output
  // test hook (negative = off): the producer of every CTA stops before
  // arming the stage of its page number `unarmed_page` (counted from the
  // CTA's first page), as if it had given up, so that the consumers' bounded
  // wait for that stage runs out with no copy in flight for it
  int unarmed_page;
  float q_scale;  // scale * log2(e) (* k_scale for FP8)
  float v_scale;  // FP8: v_scale, else 1 (an INT8 cache scales each row instead)
};

constexpr int cmin(int a, int b) { return a < b ? a : b; }
constexpr int cmax(int a, int b) { return a > b ? a : b; }
constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }
constexpr int round_up(int x, int m) { return (x + m - 1) / m * m; }

// Lanes per row: the fewest (>= PA_LPR_MIN) that keep q and acc at <= 32 fp32 each with
// an even number of elements per lane (they are processed as fp32 pairs);
// failing that, the most lanes that still give an even count.
constexpr int choose_lpr(int D, int GT) {
  for (int l = PA_LPR_MIN; l <= 32; l *= 2)
    if (D % l == 0 && (D / l) % 2 == 0 && (D / l) * GT <= 32) return l;
  for (int l = 32; l >= 4; l /= 2)
    if (D % l == 0 && (D / l) % 2 == 0) return l;
  return 4;
}
constexpr int choose_pb(int bytes) {
  return bytes % 16 == 0 ? 16 : bytes % 8 == 0 ? 8 : bytes % 4 == 0 ? 4 : bytes % 2 == 0 ? 2 : 1;
}

template <typename QT, typename CT, int D, int GT, int BS, int MODE = kModeBalanced>
struct Layout {
  static constexpr int EB = Elem<CT>::bytes;
  static constexpr int QB = Elem<QT>::bytes;
  static constexpr int ROWB = D * EB;      // bytes of one cached row
  static constexpr int PAGE = BS * ROWB;   // bytes of one (block, kv head) page
  static constexpr bool TC = uses_tc<QT, CT, D, GT, BS>();    // 16-bit cache on MMAs
  static constexpr bool TC8 = uses_tc8<QT, CT, D, GT, BS>();  // 8-bit cache on MMAs
  static constexpr bool SLICES = TC || TC8;  // consumer warps take 16-row slices
  static constexpr bool TMA = TC || (TC8 && ROWB == 128);  // staged by 2-D tensor copies
  static constexpr int TPW = 8;            // rows per consumer warp per page
  static constexpr int NC = TC8 ? PA_TC8_WARPS : TC ? PA_TC_WARPS : BS / TPW;  // consumer warps
  static constexpr int SW = TC8 ? PA_TC8_SLICES : 1;  // slices a consumer warp takes per iteration
  static constexpr int SPP = BS / 16;      // tensor-core consumers: 16-row slices per page
  static constexpr int THREADS = (NC + 1) * 32;
  static constexpr int LPR = choose_lpr(D, GT);
  static constexpr int EPL = D / LPR;      // elements of a row per lane
  static constexpr int PB = choose_pb(EPL * EB);
  static constexpr int EPP = PB / EB;      // elements per piece
  static constexpr int NPL = EPL / EPP;    // pieces per lane
  static constexpr int EP2 = EPP / 2;      // fp32 pairs per piece
  static constexpr int EL2 = EPL / 2;      // fp32 pairs per lane
  static constexpr int RPW = 32 / LPR;     // rows a warp covers per step
  static constexpr int NST = TPW / RPW;    // steps per page
  // pages a consumer warp takes per iteration (one weight round per R pages)
  // (tensor-core consumers: one 16-row slice of one page per warp)
  static constexpr int R = SLICES                ? cmax(1, NC * SW / cmax(SPP, 1))
                           : (2 * PAGE <= 8192)  ? 2 * PA_PAGES_PER_ITER
                           : (2 * PAGE <= 16384) ? PA_PAGES_PER_ITER
                                                 : 1;
  static constexpr int TPI = TPW * R;      // rows per warp per iteration
  static constexpr int NSTI = NST * R;     // steps per iteration
  static constexpr int SG = cmin(NSTI, cmax(1, 8 / GT));   // steps per reduction group
  static constexpr int NV = SG * GT;       // partial dot products per group
  static constexpr int NFIN = cmax(NV / LPR, 1);       // reduced values a lane holds
  static constexpr int RED = NV < LPR ? LPR / NV : 1;  // lanes holding the same value
  static constexpr int NG = NSTI / SG;                 // reduction groups per iteration
  // After the reduction lane c (of a row) holds value index (c*NV)/LPR + kk,
  // head = index % GT. Lane bits [HB0, HB0 + NHB) of c select the head; the
  // other lane bits only select tokens (or redundant copies).
  static constexpr int HB0 = NV >= LPR ? 0 : ilog2(RED);
  static constexpr int NHB = NV >= LPR ? ilog2(cmax(GT / NFIN, 1)) : ilog2(GT);
  static constexpr int HEAD_MASK = ((1 << NHB) - 1) << HB0;
  static constexpr int QSLOT = round_up(GT * D * QB, 16);        // q rows of a piece
  // an INT8 cache stages its pages' row scales too (BS floats each for K and V)
  static constexpr bool ROW_SCALES = std::is_same<CT, I8>::value;
  static constexpr int SCB = ROW_SCALES ? BS * 4 : 0;
  static constexpr int OFF_Q = 2 * PAGE + 2 * SCB;
  // K page | V page | (K row scales | V row scales) | q rows; the swizzled
  // boxes of the tensor-core layout start on 1024-byte boundaries
  static constexpr int STAGE = round_up(OFF_Q + QSLOT, TMA ? 1024 : 128);
  static constexpr int STAGES =
      TC8      ? cmax(2 * R, cmin(PA_TC8_MAX_STAGES,
                                   (ROW_SCALES ? PA_TC8_I8_STAGE_BYTES : PA_TC8_STAGE_BYTES) /
                                       STAGE))
      : SLICES ? cmax(2 * R, cmin(PA_MAX_STAGES, (MODE == kModeSplit ? PA_TC_SPLIT_STAGE_BYTES
                                                                   : PA_TC_STAGE_BYTES) /
                                                    STAGE))
          : cmax(2 * R, cmin(PA_MAX_STAGES, PA_STAGE_BYTES / (2 * PAGE)));
  static constexpr int BOXB = BS * 128;     // bytes of one 128-byte-wide box of a page
  static constexpr int BOXES = ROWB / 128;  // boxes per page (tensor-copy layouts)
  static constexpr int SCR = SLICES ? 0 : round_up(TPI * GT, 4);  // per-warp weights
  static constexpr int MACC = NC * GT * D * 4;                   // merge accumulators
  static constexpr bool MERGE_IN_STAGE = MACC <= STAGE;
  // dynamic shared memory layout
  static constexpr int OFF_BAR = STAGES * STAGE;
  static constexpr int OFF_DESC = round_up(OFF_BAR + (2 * STAGES + 1) * 8, 16);
  static constexpr int OFF_SCR = round_up(OFF_DESC + STAGES * 16, 16);
  static constexpr int OFF_MSTAT = OFF_SCR + NC * SCR * 4;  // [3][NC][GT]
  static constexpr int OFF_MACC = round_up(OFF_MSTAT + 3 * NC * GT * 4, 16);
  static constexpr int OFF_MISC = OFF_MACC + (MERGE_IN_STAGE ? 0 : MACC);
  // misc: 4 ints, 2 int64 (range start, total pages), 2 cut-piece records
  static constexpr int SMEM_USED = OFF_MISC + 32 + 2 * 24;
  // the tensor-core layout rounds the dynamic shared memory's base up to
  // 1024 bytes itself (it may start anywhere 16-byte aligned)
  static constexpr int ALIGN_PAD = TMA ? 1024 : 0;
  static constexpr int SMEM = SMEM_USED + ALIGN_PAD;
  // CTAs per SM to plan registers for: what the shared memory allows (228 KB
  // per SM, 1 KB reserved per CTA), at most 4, and no more than keeps a
  // register budget per thread (96 for one or two heads per kv head, else
  // 128); __launch_bounds__ makes ptxas fit that many.
  static constexpr int REG_BUDGET = GT <= 2 ? 96 : PA_REG_BUDGET_WIDE;
  static constexpr int MIN_CTAS =
      cmax(1, cmin(cmin(4, (228 * 1024) / (SMEM + 1024)), 65536 / (THREADS * REG_BUDGET)));
  static_assert(NST >= 1, "lanes per row too small for 8 rows per warp");
  static_assert(NSTI % SG == 0, "reduction groups must tile the steps");
  static_assert(STAGES >= R, "a consumer iteration holds R stages");
  static_assert(EPL * LPR == D && NPL * EPP == EPL, "row split");
  static_assert(EPP % 2 == 0, "pieces hold whole fp32 pairs");
  static_assert(PAGE % 16 == 0 && SCB % 16 == 0, "bulk copies move multiples of 16 bytes");
  static_assert(STAGE % 128 == 0 && OFF_BAR % 8 == 0, "stage and mbarrier alignment");
  static_assert(!TMA || (ROWB % 128 == 0 && PAGE % 1024 == 0 && BOXB % 1024 == 0),
                "tensor-copy layout: whole 128-byte boxes");
  static_assert(!SLICES || (BS % 16 == 0 && (NC * SW) % SPP == 0),
                "tensor-core layout: 16-row slices, whole pages per iteration");
  static_assert(!TC8 || D % 32 == 0, "8-bit tensor-core layout: 32-dim blocks");
  static_assert(OFF_DESC % 16 == 0 && OFF_SCR % 16 == 0 && OFF_MSTAT % 16 == 0 &&
                    OFF_MACC % 16 == 0 && OFF_MISC % 16 == 0 && (SCR * 4) % 16 == 0,
                "16-byte vector accesses need 16-byte aligned shared-memory regions");
};

// Transposing butterfly reduction of N per-lane values over lane offsets
// OFF, OFF/2, ..., 1: while a lane holds >= 2 values, each level halves them
// (the lane keeps the half selected by its lane bit and adds its partner's
// copy of that half); below 2 values it is a plain butterfly.
template <int N, int OFF>
struct TransposeReduce {
  __device__ __forceinline__ static void run(float* v, int lane) {
    if constexpr (OFF >= 1) {
      if constexpr (N >= 2) {
        constexpr int H = N / 2;
        const bool upper = (lane & OFF) != 0;
#pragma unroll
        for (int i = 0; i < H; ++i) {
          const float send = upper ? v[i] : v[i + H];
          const float keep = upper ? v[i + H] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
        }
        TransposeReduce<H, OFF / 2>::run(v, lane);
      } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], OFF);
        TransposeReduce<1, OFF / 2>::run(v, lane);
      }
    }
  }
};

// N consecutive floats from shared memory (vector loads where aligned).
template <int N>
__device__ __forceinline__ void load_row(const float* src, float* dst) {
  if constexpr (N % 4 == 0) {
#pragma unroll
    for (int i = 0; i < N; i += 4) {
      const float4 v = *reinterpret_cast<const float4*>(src + i);
      dst[i] = v.x; dst[i + 1] = v.y; dst[i + 2] = v.z; dst[i + 3] = v.w;
    }
  } else if constexpr (N == 2) {
    const float2 v = *reinterpret_cast<const float2*>(src);
    dst[0] = v.x; dst[1] = v.y;
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) dst[i] = src[i];
  }
}

// acc[h][:] += p[h] * V_row[this lane's elements] for one row.
template <typename CT, typename Ly, int GT, int EL2>
__device__ __forceinline__ void pv_row(const float* pw_src, const uint8_t* vr, int c,
                                       float2 (&acc)[GT][EL2]) {
  float pw[GT];
  load_row<GT>(pw_src, pw);
#pragma unroll
  for (int kk = 0; kk < Ly::NPL; ++kk) {
    float2 vf[Ly::EP2];
    load_piece2<CT, Ly::PB>(vr + (kk * Ly::LPR + c) * Ly::PB, vf);
#pragma unroll
    for (int h = 0; h < GT; ++h) {
      const float2 pp = make_float2(pw[h], pw[h]);
#pragma unroll
      for (int j2 = 0; j2 < Ly::EP2; ++j2)
        acc[h][kk * Ly::EP2 + j2] = __ffma2_rn(pp, vf[j2], acc[h][kk * Ly::EP2 + j2]);
    }
  }
}

// Per-lane state of one piece's online softmax.
template <typename Ly, int GT>
struct PieceState {
  float2 qf[GT][Ly::EL2];   // q (pre-scaled), consecutive pairs of this lane's elements
  float2 acc[GT][Ly::EL2];  // un-normalised output, same layout
  float m_run[Ly::NFIN];    // running (lazy) max of the head of reduced value kk
  float l_run[Ly::NFIN];    // this lane's share of the running sum
  float s_top[Ly::NFIN];    // largest logit seen
};

// Start a piece: q rows (G of them, row-major [G][D] of QT in shared memory).
template <typename QT, typename Ly, int GT, int D>
__device__ __forceinline__ void begin_piece(PieceState<Ly, GT>& st, const uint8_t* qrows, int G,
                                            int c, float q_scale) {
  const QT* q = reinterpret_cast<const QT*>(qrows);
#pragma unroll
  for (int h = 0; h < GT; ++h) {
#pragma unroll
    for (int kk = 0; kk < Ly::NPL; ++kk) {
#pragma unroll
      for (int j2 = 0; j2 < Ly::EP2; ++j2) {
        const int d = (kk * Ly::LPR + c) * Ly::EPP + 2 * j2;
        st.qf[h][kk * Ly::EP2 + j2] =
            h < G ? make_float2(Elem<QT>::to_f32(q[h * D + d]) * q_scale,
                                Elem<QT>::to_f32(q[h * D + d + 1]) * q_scale)
                  : make_float2(0.f, 0.f);
        st.acc[h][kk * Ly::EP2 + j2] = make_float2(0.f, 0.f);
      }
    }
  }
#pragma unroll
  for (int kk = 0; kk < Ly::NFIN; ++kk) {
    st.m_run[kk] = -INFINITY;
    st.l_run[kk] = 0.f;
    st.s_top[kk] = -INFINITY;
  }
}

// One consumer iteration over R pages of the current piece (a page with
// lim[r] <= 0 contributes nothing). Token t of the warp's TPI rows is row
// warp*TPW + t%TPW of page t/TPW; rows t%TPW < lim[t/TPW] are attended.
// With an INT8 cache, Ks / Vs point at the pages' staged row scales: a
// token's logit is multiplied by its K row's scale, and its softmax weight
// by its V row's scale before P.V (the running sum takes the bare weight).
template <typename CT, typename Ly, int GT>
__device__ __forceinline__ void process_pages(PieceState<Ly, GT>& st,
                                              const uint8_t* const (&Kp)[Ly::R],
                                              const uint8_t* const (&Vp)[Ly::R],
                                              const float* const (&Ks)[Ly::R],
                                              const float* const (&Vs)[Ly::R],
                                              const int (&lim)[Ly::R], float* wscr, int warp,
                                              int lane, int c, int rg) {
  constexpr int R = Ly::R, TPW = Ly::TPW, RPW = Ly::RPW, LPR = Ly::LPR, NV = Ly::NV;
  constexpr int NG = Ly::NG, NFIN = Ly::NFIN, RED = Ly::RED, EP2 = Ly::EP2, EL2 = Ly::EL2;
  constexpr float kLazy = 8.f;  // weights stay <= 2^kLazy
  const bool writer = (c % RED) == 0;  // one lane per distinct reduced value

  // ---- 1. logits, reduced across the row's lanes; invalid rows become -inf
  float sl[NG][NFIN];
#pragma unroll
  for (int sg = 0; sg < NG; ++sg) {
    float part[NV];
    {
      float2 part2[NV];
#pragma unroll
      for (int i = 0; i < NV; ++i) part2[i] = make_float2(0.f, 0.f);
#pragma unroll
      for (int stl = 0; stl < Ly::SG; ++stl) {
        const int stp = sg * Ly::SG + stl;
        const int row = warp * TPW + (stp % Ly::NST) * RPW + rg;
        const uint8_t* kr = Kp[stp / Ly::NST] + row * Ly::ROWB;
#pragma unroll
        for (int kk = 0; kk < Ly::NPL; ++kk) {
          float2 kf[EP2];
          load_piece2<CT, Ly::PB>(kr + (kk * LPR + c) * Ly::PB, kf);
#pragma unroll
          for (int h = 0; h < GT; ++h)
#pragma unroll
            for (int j2 = 0; j2 < EP2; ++j2)
              part2[stl * GT + h] = __ffma2_rn(st.qf[h][kk * EP2 + j2], kf[j2], part2[stl * GT + h]);
        }
      }
#pragma unroll
      for (int i = 0; i < NV; ++i) part[i] = part2[i].x + part2[i].y;
    }
    TransposeReduce<NV, LPR / 2>::run(part, lane);
#pragma unroll
    for (int kk = 0; kk < NFIN; ++kk) {
      const int t = (sg * Ly::SG + ((c * NV) / LPR + kk) / GT) * RPW + rg;
      int lim_t = lim[0];  // lim of token t's page, without dynamic indexing
#pragma unroll
      for (int r = 1; r < R; ++r) lim_t = t >= r * TPW ? lim[r] : lim_t;
      float logit = part[kk];
      if constexpr (Ly::ROW_SCALES) {
        const float* ks = Ks[0];
#pragma unroll
        for (int r = 1; r < R; ++r) ks = t >= r * TPW ? Ks[r] : ks;
        logit *= ks[warp * TPW + t % TPW];
      }
      sl[sg][kk] = (writer && (t % TPW) < lim_t) ? logit : -INFINITY;
    }
  }

  // ---- 2. lazy max: move m only when a logit clears it by kLazy
  bool raise = false;
#pragma unroll
  for (int kk = 0; kk < NFIN; ++kk) {
    float top = sl[0][kk];
#pragma unroll
    for (int sg = 1; sg < NG; ++sg) top = fmaxf(top, sl[sg][kk]);
    st.s_top[kk] = fmaxf(st.s_top[kk], top);
    raise |= top > st.m_run[kk] + kLazy;
  }
  if (__any_sync(0xffffffffu, raise)) {
    float alpha[NFIN];
#pragma unroll
    for (int kk = 0; kk < NFIN; ++kk) {
      float top = sl[0][kk];
#pragma unroll
      for (int sg = 1; sg < NG; ++sg) top = fmaxf(top, sl[sg][kk]);
#pragma unroll
      for (int off = 1; off < 32; off *= 2)  // over every lane bit but the head bits
        if ((off & Ly::HEAD_MASK) == 0) top = fmaxf(top, __shfl_xor_sync(0xffffffffu, top, off));
      const float m_new = fmaxf(st.m_run[kk], top);
      alpha[kk] = m_new == -INFINITY ? 1.f : exp2f(st.m_run[kk] - m_new);
      st.m_run[kk] = m_new;
      st.l_run[kk] *= alpha[kk];
    }
    float al[GT];  // every head's factor, from a lane that holds that head
#pragma unroll
    for (int h = 0; h < GT; ++h)
      al[h] = __shfl_sync(0xffffffffu, alpha[h % NFIN], NV >= LPR ? h / NFIN : h * RED);
#pragma unroll
    for (int h = 0; h < GT; ++h)
#pragma unroll
      for (int e = 0; e < EL2; ++e) st.acc[h][e] = __fmul2_rn(st.acc[h][e], make_float2(al[h], al[h]));
  }

  // ---- 3. weights 2^(s - m) to shared memory, then P.V
#pragma unroll
  for (int sg = 0; sg < NG; ++sg)
#pragma unroll
    for (int kk = 0; kk < NFIN; ++kk) {
      const float pw = sl[sg][kk] == -INFINITY ? 0.f : exp2f(sl[sg][kk] - st.m_run[kk]);
      st.l_run[kk] += pw;
      if (writer) {
        const int idx = (c * NV) / LPR + kk;
        const int t = (sg * Ly::SG + idx / GT) * RPW + rg;
        float w = pw;
        if constexpr (Ly::ROW_SCALES) {
          const float* vs = Vs[0];
#pragma unroll
          for (int r = 1; r < R; ++r) vs = t >= r * TPW ? Vs[r] : vs;
          // rows past the context have weight 0 and may hold any scale
          w = pw == 0.f ? 0.f : pw * vs[warp * TPW + t % TPW];
        }
        wscr[t * GT + idx % GT] = w;
      }
    }
  __syncwarp();
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (lim[r] >= TPW) {  // every row of this warp in page r is attended
#pragma unroll
      for (int stp = 0; stp < Ly::NST; ++stp) {
        const int tr = stp * RPW + rg;
        pv_row<CT, Ly>(wscr + (r * TPW + tr) * GT, Vp[r] + (warp * TPW + tr) * Ly::ROWB, c, st.acc);
      }
    } else if (lim[r] > 0) {
#pragma unroll
      for (int stp = 0; stp < Ly::NST; ++stp) {
        const int tr = stp * RPW + rg;
        if (tr < lim[r])
          pv_row<CT, Ly>(wscr + (r * TPW + tr) * GT, Vp[r] + (warp * TPW + tr) * Ly::ROWB, c,
                         st.acc);
      }
    }
  }
  __syncwarp();
}

// ------------------------------------------------------ tensor-core consumers
// Lane l of a consumer warp is (g = l / 4, t = l % 4) in the m16n8k16
// fragments: it owns query head g of the group (m16 rows g >= G and 8..15
// are zero padding), logits of tokens 2t, 2t+1, 8+2t, 9+2t of the warp's
// 16-row slice, and output elements 8j + 2t, 8j + 2t + 1 of head g.
template <int D>
struct TcState {
  uint32_t qa[D / 16][2];  // A fragments of q: head g, dims 16kk + 2t (+1) and 16kk + 8 + 2t (+1)
  float o[D / 8][4];       // C fragments of P V: [0..1] head g, [2..3] padding rows
  float m_run;             // running (lazy) max of head g, log2 units
  float l_run;             // this lane's share of head g's running sum
  float s_top;             // largest logit of head g seen
};

// Start a piece: q rows (G of them, row-major [G][D] of QT in shared memory).
template <typename QT, int D>
__device__ __forceinline__ void begin_piece_tc(TcState<D>& st, const uint8_t* qrows, int G,
                                               int lane) {
  const int g = lane >> 2, t = lane & 3;
  const uint32_t* q = reinterpret_cast<const uint32_t*>(qrows) + g * (D / 2);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    st.qa[kk][0] = g < G ? q[8 * kk + t] : 0u;
    st.qa[kk][1] = g < G ? q[8 * kk + 4 + t] : 0u;
  }
#pragma unroll
  for (int j = 0; j < D / 8; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) st.o[j][e] = 0.f;
  st.m_run = -INFINITY;
  st.l_run = 0.f;
  st.s_top = -INFINITY;
}

// Shared-memory address of 16-byte chunk `ch` (8 elements) of row `row` of a
// page staged as D/64 boxes of BS rows x 128 bytes with the 128-byte swizzle
// (the chunk index is XORed with the row index mod 8).
template <typename Ly>
__device__ __forceinline__ uint32_t tc_chunk(uint32_t page, int row, int ch) {
  return page + (ch >> 3) * Ly::BOXB + row * 128 + (((ch & 7) ^ (row & 7)) << 4);
}

// One consumer iteration: the warp takes rows [r0, r0 + 16) of page
// pr = warp / SPP of the R staged pages (r0 = 16 (warp mod SPP)); rows[r] is
// the number of attended rows of page r (0 for pages not in this iteration).
template <typename QT, typename Ly, int D>
__device__ __forceinline__ void process_tc(TcState<D>& st, const uint8_t* const (&Kp)[Ly::R],
                                           const uint8_t* const (&Vp)[Ly::R],
                                           const int (&rows)[Ly::R], int warp, int lane,
                                           float q_scale, int G) {
  constexpr int R = Ly::R, SPP = Ly::SPP;
  constexpr float kLazy = 8.f;  // weights stay <= 2^kLazy
  using M = Mma<QT>;
  const int pr = warp / SPP, r0 = 16 * (warp % SPP);
  const uint8_t* kp = Kp[0];
  const uint8_t* vp = Vp[0];
  int n = rows[0];
#pragma unroll
  for (int r = 1; r < R; ++r)
    if (pr == r) {
      kp = Kp[r];
      vp = Vp[r];
      n = rows[r];
    }
  const int lim = n - r0;  // attended rows of the slice (warp-uniform)
  if (lim <= 0) return;
  const int g = lane >> 2, t = lane & 3, mi = lane >> 3;
  const bool real = g < G;

  // ---- S = Q K^T over the slice's 16 tokens (two n8 tiles)
  float sacc[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
  {
    // matrix mi of an x4 load: tokens r0 + 8 (mi / 2) .. + 7, chunk 2 kk + mi % 2
    const uint32_t kb = smem_u32(kp);
    const int krow = r0 + ((mi >> 1) << 3) + (lane & 7);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(tc_chunk<Ly>(kb, krow, 2 * kk + (mi & 1)), b0, b1, b2, b3);
      const uint32_t a[4] = {st.qa[kk][0], 0u, st.qa[kk][1], 0u};
      M::run(sacc[0], a, b0, b1);
      M::run(sacc[1], a, b2, b3);
    }
  }

  // ---- logits of head g (log2 units), masked past the context; lazy max
  float x[4] = {sacc[0][0] * q_scale, sacc[0][1] * q_scale, sacc[1][0] * q_scale,
                sacc[1][1] * q_scale};
  const int tok[4] = {2 * t, 2 * t + 1, 8 + 2 * t, 9 + 2 * t};
#pragma unroll
  for (int j = 0; j < 4; ++j) x[j] = (real && tok[j] < lim) ? x[j] : -INFINITY;
  float tm = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
  tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 1));
  tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 2));
  st.s_top = fmaxf(st.s_top, tm);
  if (__any_sync(0xffffffffu, tm > st.m_run + kLazy)) {
    const float mn = fmaxf(st.m_run, tm);
    const float al = mn == -INFINITY ? 1.f : exp2f(st.m_run - mn);
    st.m_run = mn;
    st.l_run *= al;
#pragma unroll
    for (int j = 0; j < D / 8; ++j) {
      st.o[j][0] *= al;
      st.o[j][1] *= al;
    }
  }

  // ---- weights 2^(s - m), rounded to the cache type as the MMA takes them
  uint32_t pa0 = M::pack(exp2f(x[0] - st.m_run), exp2f(x[1] - st.m_run));
  uint32_t pa2 = M::pack(exp2f(x[2] - st.m_run), exp2f(x[3] - st.m_run));
  if (!real) pa0 = pa2 = 0u;  // padding rows: m_run stays -inf, weights would be NaN
  st.l_run += M::sum2(pa0) + M::sum2(pa2);
  const uint32_t a[4] = {pa0, 0u, pa2, 0u};

  // ---- O += P V (16 n8 tiles of head_dim for D 128); rows past the
  // context are zeroed in the fragments (they may hold anything, NaN too)
  const uint32_t vb = smem_u32(vp);
  // matrix mi of an x4.trans load: tokens r0 + 8 (mi % 2) .. + 7, chunk 2 jj + mi / 2
  const int vrow = r0 + ((mi & 1) << 3) + (lane & 7);
  if (lim >= 16) {
#pragma unroll
    for (int jj = 0; jj < D / 16; ++jj) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(tc_chunk<Ly>(vb, vrow, 2 * jj + (mi >> 1)), b0, b1, b2, b3);
      M::run(st.o[2 * jj], a, b0, b1);
      M::run(st.o[2 * jj + 1], a, b2, b3);
    }
  } else {
    const uint32_t mk0 = (tok[0] < lim ? 0x0000FFFFu : 0u) | (tok[1] < lim ? 0xFFFF0000u : 0u);
    const uint32_t mk1 = (tok[2] < lim ? 0x0000FFFFu : 0u) | (tok[3] < lim ? 0xFFFF0000u : 0u);
#pragma unroll
    for (int jj = 0; jj < D / 16; ++jj) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(tc_chunk<Ly>(vb, vrow, 2 * jj + (mi >> 1)), b0, b1, b2, b3);
      M::run(st.o[2 * jj], a, b0 & mk0, b1 & mk1);
      M::run(st.o[2 * jj + 1], a, b2 & mk0, b3 & mk1);
    }
  }
}

// ------------------------------------------------ tensor-core consumers, 8-bit
// An 8-bit cache (FP8 E4M3 with per-tensor scales, or INT8 with a scale per
// cached row) read with 16-bit queries, any group size up to 8 and head_dim
// 64 / 96 / 128, on m16n8k16 f16 MMAs with the roles turned round: the 16
// cached rows of a slice are the m16 rows and the (up to 8) query heads of
// the kv head the n8 columns, so S^T = K Q^T and O^T = V^T P^T and no MMA
// row is padding whatever G is. Codes widen exactly to f16: E4M3 two per cvt
// (every E4M3 value is an f16 value); INT8 by a byte permute that makes
// 1024 + (c + 128) an f16 bit pattern and one packed subtract of 1152. q is
// carried in f16 (exact for a bf16 query inside f16's range); the scales
// multiply the fp32 logits; the weights are rounded to f16 for the MMA.
// FP8: the running sum takes the rounded weights, v_scale is applied at the
// end. INT8: a row's K scale multiplies its logits, its V scale its weight
// before the rounding, and the running sum takes the bare weights.
// Staging: at head_dim 128 a row is one 128-byte swizzle row and the pages
// come by 2-D tensor copies (chunk c of row r at chunk c ^ (r mod 8)); else
// by 1-D bulk copies, rows of D bytes. The loads below are bank-conflict free
// on both (D = 96 unswizzled, D = 128 swizzled) because of a fixed
// permutation of a slice's rows: MMA row i < 8 reads cached row pi(i), row
// 8 + i reads 8 + pi(i), pi = (0 1 2 3 5 4 7 6).
//  * K: lane (g, t) reads bytes [D/4 t, D/4 (t + 1)) of rows pi(g) and
//    8 + pi(g); its four codes of step kk (dims D/4 t + 4 kk .. +3) are the
//    step's k indices (2t, 2t+1, 2t+8, 2t+9), and q's B fragments follow the
//    same permutation of dims.
//  * P: the C fragment of S^T (row = cached row, column = head) becomes P^T's
//    B fragment by movmatrix (an 8 x 8 transpose in registers).
//  * V: lane (g, t) reads 4-code words at dims 4x .. 4x + 3, x = g + 8j, of
//    rows pi(2t), pi(2t+1), 8 + pi(2t), 8 + pi(2t+1); a byte permute pairs
//    the two rows' codes of a dim, which is one A register of V^T. Tile 2j
//    takes dims 4x (MMA row g) and 4x + 1 (row g + 8), tile 2j + 1 dims 4x + 2
//    and 4x + 3; the output is put back in dim order when it is stored.
template <int D>
struct Tc8State {
  uint32_t qb[D / 16][2];  // B fragments of q^T: head g, dims D/4 t + 4 kk (+1) / (+2, +3)
  float o[D / 16][4];      // C fragments of O^T: tile 2j + u, rows dims, columns heads
  float m_run[2], l_run[2], s_top[2];  // heads 2t and 2t + 1
};

__device__ __forceinline__ int tc8_row(int i) { return i < 4 ? i : i ^ 1; }

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

template <typename QT>
__device__ __forceinline__ uint32_t q_pair_f16(const QT* q) {
  const __half2 h = __floats2half2_rn(Elem<QT>::to_f32(q[0]), Elem<QT>::to_f32(q[1]));
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Byte `b` of row `r` of a staged page (swizzled rows of 128 bytes when the
// layout is staged by tensor copies).
template <typename Ly>
__device__ __forceinline__ const uint8_t* tc8_at(const uint8_t* page, int r, int b) {
  if constexpr (Ly::TMA)
    return page + r * 128 + ((((b >> 4) ^ r) & 7) << 4) + (b & 15);
  else
    return page + r * Ly::ROWB + b;
}

template <typename QT, int D>
__device__ __forceinline__ void begin_piece_tc8(Tc8State<D>& st, const uint8_t* qrows, int G,
                                                int lane) {
  const int g = lane >> 2, t = lane & 3;
  const QT* q = reinterpret_cast<const QT*>(qrows) + g * D + (D / 4) * t;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    st.qb[kk][0] = g < G ? q_pair_f16(q + 4 * kk) : 0u;
    st.qb[kk][1] = g < G ? q_pair_f16(q + 4 * kk + 2) : 0u;
  }
#pragma unroll
  for (int j = 0; j < D / 16; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) st.o[j][e] = 0.f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    st.m_run[h] = -INFINITY;
    st.l_run[h] = 0.f;
    st.s_top[h] = -INFINITY;
  }
}

// S^T = K Q^T over the slice of rows [r0, r0 + 16) of a staged K page: the
// log2-unit logits of heads 2t (x[0], x[2]) and 2t + 1 (x[1], x[3]) for rows
// r0 + kr (x[0], x[1]) and r0 + 8 + kr (x[2], x[3]); rows at or past r0 + lim
// are masked. ks: the page's K row scales (INT8), else unused.
template <typename Ly, typename CT, int D>
__device__ __forceinline__ void tc8_logits(const Tc8State<D>& st, const uint8_t* kpage,
                                           const float* ks, int r0, int kr, int t, int lim,
                                           float q_scale, float (&x)[4]) {
  using M = Mma<__half>;
  float sacc[4] = {0.f, 0.f, 0.f, 0.f};
  uint32_t w0[D / 16], w1[D / 16];
  const int ra = r0 + kr, rb = r0 + 8 + kr;
  if constexpr ((D / 4) % 16 == 0) {
#pragma unroll
    for (int i = 0; i < D / 64; ++i) {
      const uint4 a = *reinterpret_cast<const uint4*>(tc8_at<Ly>(kpage, ra, (D / 4) * t + 16 * i));
      const uint4 b = *reinterpret_cast<const uint4*>(tc8_at<Ly>(kpage, rb, (D / 4) * t + 16 * i));
      w0[4 * i] = a.x; w0[4 * i + 1] = a.y; w0[4 * i + 2] = a.z; w0[4 * i + 3] = a.w;
      w1[4 * i] = b.x; w1[4 * i + 1] = b.y; w1[4 * i + 2] = b.z; w1[4 * i + 3] = b.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < D / 32; ++i) {
      const uint2 a = *reinterpret_cast<const uint2*>(tc8_at<Ly>(kpage, ra, (D / 4) * t + 8 * i));
      const uint2 b = *reinterpret_cast<const uint2*>(tc8_at<Ly>(kpage, rb, (D / 4) * t + 8 * i));
      w0[2 * i] = a.x; w0[2 * i + 1] = a.y;
      w1[2 * i] = b.x; w1[2 * i + 1] = b.y;
    }
  }
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    uint32_t a[4];
    widen8<CT>(w0[kk], a[0], a[2]);
    widen8<CT>(w1[kk], a[1], a[3]);
    M::run(sacc, a, st.qb[kk][0], st.qb[kk][1]);
  }
  float sa = q_scale, sb = q_scale;
  if constexpr (Ly::ROW_SCALES) {
    sa *= ks[ra];
    sb *= ks[rb];
  }
  const bool ok0 = kr < lim, ok1 = kr + 8 < lim;
  x[0] = ok0 ? sacc[0] * sa : -INFINITY;
  x[1] = ok0 ? sacc[1] * sa : -INFINITY;
  x[2] = ok1 ? sacc[2] * sb : -INFINITY;
  x[3] = ok1 ? sacc[3] * sb : -INFINITY;
}

// O^T += V^T P^T over the slice of rows [r0, r0 + 16) of a staged V page;
// with MASK, the codes of rows at or past r0 + lim are zeroed first (they
// may hold anything, NaN codes too).
template <typename Ly, typename CT, int D, bool MASK>
__device__ __forceinline__ void tc8_pv(Tc8State<D>& st, const uint8_t* vpage, int r0,
                                       uint32_t pb0, uint32_t pb1, int g, int t, int lim) {
  using M = Mma<__half>;
  const int ra = tc8_row(2 * t), rb = tc8_row(2 * t + 1);
  const bool oka = ra < lim, okb = rb < lim, okc = ra + 8 < lim, okd = rb + 8 < lim;
#pragma unroll
  for (int j = 0; j < D / 32; ++j) {
    const int b = 4 * g + 32 * j;
    uint32_t wa = *reinterpret_cast<const uint32_t*>(tc8_at<Ly>(vpage, r0 + ra, b));
    uint32_t wb = *reinterpret_cast<const uint32_t*>(tc8_at<Ly>(vpage, r0 + rb, b));
    uint32_t wc = *reinterpret_cast<const uint32_t*>(tc8_at<Ly>(vpage, r0 + 8 + ra, b));
    uint32_t wd = *reinterpret_cast<const uint32_t*>(tc8_at<Ly>(vpage, r0 + 8 + rb, b));
    if constexpr (MASK) {
      // an INT8 zero code is the byte 0; an E4M3 zero too
      wa = oka ? wa : 0u;
      wb = okb ? wb : 0u;
      wc = okc ? wc : 0u;
      wd = okd ? wd : 0u;
    }
    uint32_t a0[4], a1[4];
    widen8<CT>(__byte_perm(wa, wb, 0x5140), a0[0], a0[1]);  // dims 4x, 4x+1; rows a, b
    widen8<CT>(__byte_perm(wc, wd, 0x5140), a0[2], a0[3]);  // rows 8+a, 8+b
    widen8<CT>(__byte_perm(wa, wb, 0x7362), a1[0], a1[1]);  // dims 4x+2, 4x+3
    widen8<CT>(__byte_perm(wc, wd, 0x7362), a1[2], a1[3]);
    M::run(st.o[2 * j], a0, pb0, pb1);
    M::run(st.o[2 * j + 1], a1, pb0, pb1);
  }
}

// One consumer iteration of the 8-bit tensor-core path: the warp takes SW
// slices, slice warp * SW + j being rows [r0, r0 + 16) of page pr of the R
// staged pages (pr = slice / SPP, r0 = 16 (slice mod SPP)); rows[r] is the
// number of attended rows of page r (0 for pages not in this iteration); Ks
// and Vs hold the pages' row scales (INT8). The slices share one
// running-max update.
template <typename Ly, typename CT, int D>
__device__ __forceinline__ void process_tc8(Tc8State<D>& st, const uint8_t* const (&Kp)[Ly::R],
                                            const uint8_t* const (&Vp)[Ly::R],
                                            const float* const (&Ks)[Ly::R],
                                            const float* const (&Vs)[Ly::R],
                                            const int (&rows)[Ly::R], int warp, int lane,
                                            float q_scale) {
  constexpr int R = Ly::R, SPP = Ly::SPP, SW = Ly::SW;
  constexpr float kLazy = 8.f;
  const int g = lane >> 2, t = lane & 3;
  const int kr = tc8_row(g);
  const uint8_t* kp[SW];
  const uint8_t* vp[SW];
  const float* ksc[SW];
  const float* vsc[SW];
  int r0[SW], lim[SW];
#pragma unroll
  for (int j = 0; j < SW; ++j) {
    const int si = warp * SW + j, pr = si / SPP;
    kp[j] = Kp[0];
    vp[j] = Vp[0];
    ksc[j] = Ks[0];
    vsc[j] = Vs[0];
    int n = rows[0];
#pragma unroll
    for (int r = 1; r < R; ++r)
      if (pr == r) {
        kp[j] = Kp[r];
        vp[j] = Vp[r];
        ksc[j] = Ks[r];
        vsc[j] = Vs[r];
        n = rows[r];
      }
    r0[j] = 16 * (si % SPP);
    lim[j] = n - r0[j];  // warp-uniform
  }
  // the slices run in row order, so an empty first slice means no work
  if (lim[0] <= 0) return;

  // ---- logits of every slice; one lazy running-max update for all of them
  float x[SW][4];
#pragma unroll
  for (int j = 0; j < SW; ++j) {
    if (j == 0 || lim[j] > 0) {
      tc8_logits<Ly, CT, D>(st, kp[j], ksc[j], r0[j], kr, t, lim[j], q_scale, x[j]);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) x[j][e] = -INFINITY;
    }
  }
  float tm0 = fmaxf(x[0][0], x[0][2]), tm1 = fmaxf(x[0][1], x[0][3]);
#pragma unroll
  for (int j = 1; j < SW; ++j) {
    tm0 = fmaxf(tm0, fmaxf(x[j][0], x[j][2]));
    tm1 = fmaxf(tm1, fmaxf(x[j][1], x[j][3]));
  }
#pragma unroll
  for (int off = 4; off < 32; off *= 2) {
    tm0 = fmaxf(tm0, __shfl_xor_sync(0xffffffffu, tm0, off));
    tm1 = fmaxf(tm1, __shfl_xor_sync(0xffffffffu, tm1, off));
  }
  st.s_top[0] = fmaxf(st.s_top[0], tm0);
  st.s_top[1] = fmaxf(st.s_top[1], tm1);
  if (__any_sync(0xffffffffu, tm0 > st.m_run[0] + kLazy || tm1 > st.m_run[1] + kLazy)) {
    const float mn0 = fmaxf(st.m_run[0], tm0), mn1 = fmaxf(st.m_run[1], tm1);
    const float al0 = mn0 == -INFINITY ? 1.f : exp2f(st.m_run[0] - mn0);
    const float al1 = mn1 == -INFINITY ? 1.f : exp2f(st.m_run[1] - mn1);
    st.m_run[0] = mn0;
    st.m_run[1] = mn1;
    st.l_run[0] *= al0;
    st.l_run[1] *= al1;
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      st.o[i][0] *= al0;
      st.o[i][2] *= al0;
      st.o[i][1] *= al1;
      st.o[i][3] *= al1;
    }
  }

  // ---- weights 2^(s - m) rounded to f16, P^T's B fragments by transposes,
  // then O^T += V^T P^T slice by slice
#pragma unroll
  for (int j = 0; j < SW; ++j) {
    if (j > 0 && lim[j] <= 0) continue;
    float pw[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      pw[e] = x[j][e] == -INFINITY ? 0.f : exp2f(x[j][e] - st.m_run[e & 1]);
    __half2 p01, p23;
    if constexpr (Ly::ROW_SCALES) {
      // masked rows keep a zero weight, whatever their scale holds
      const float va = vsc[j][r0[j] + kr], vb = vsc[j][r0[j] + 8 + kr];
      st.l_run[0] += pw[0] + pw[2];
      st.l_run[1] += pw[1] + pw[3];
      p01 = __floats2half2_rn(pw[0] == 0.f ? 0.f : pw[0] * va, pw[1] == 0.f ? 0.f : pw[1] * va);
      p23 = __floats2half2_rn(pw[2] == 0.f ? 0.f : pw[2] * vb, pw[3] == 0.f ? 0.f : pw[3] * vb);
    } else {
      p01 = __floats2half2_rn(pw[0], pw[1]);
      p23 = __floats2half2_rn(pw[2], pw[3]);
      const float2 f01 = __half22float2(p01), f23 = __half22float2(p23);
      st.l_run[0] += f01.x + f23.x;
      st.l_run[1] += f01.y + f23.y;
    }
    const uint32_t pb0 = movmatrix_trans(*reinterpret_cast<const uint32_t*>(&p01));
    const uint32_t pb1 = movmatrix_trans(*reinterpret_cast<const uint32_t*>(&p23));
    if (lim[j] >= 16)
      tc8_pv<Ly, CT, D, false>(st, vp[j], r0[j], pb0, pb1, g, t, lim[j]);
    else
      tc8_pv<Ly, CT, D, true>(st, vp[j], r0[j], pb0, pb1, g, t, lim[j]);
  }
}

// Bounded barrier among the NC consumer warps (an mbarrier with one arrival
// per warp), so a consumer that gave up on a wait can never hang the others.
__device__ __forceinline__ void consumer_sync(uint64_t* bar, uint32_t& phase, int lane,
                                              unsigned* err) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
  if (!mbar_wait_bounded(bar, phase & 1)) raise_error(err, PA_DEVERR_TIMEOUT);
  ++phase;
}

template <typename Ly, int GT, int D, typename Sink>
__device__ __forceinline__ void merge_warps(const float* mstat, const float* macc, uint64_t* cbar,
                                            uint32_t& cphase, int G, int warp, int lane,
                                            float v_scale, unsigned* err, Sink&& sink);

// End of a piece: reduce each warp's state, merge the NC warps through shared
// memory, and hand every (head, element) result to `sink`:
//   sink(h, d, o, m_nat, l) with o the normalised output (v_scale applied),
//   m_nat the piece's largest logit in natural-log units and l the sum of
//   exp(logit - m_nat) (m_nat = -inf, l = 0 when no slot was attended).
template <typename Ly, int GT, int D, typename Sink>
__device__ __forceinline__ void finish_piece(PieceState<Ly, GT>& st, float* mstat, float* macc,
                                             uint64_t* cbar, uint32_t& cphase, int G, int warp,
                                             int lane, int c, int rg, float v_scale, unsigned* err,
                                             Sink&& sink) {
  constexpr int NC = Ly::NC, LPR = Ly::LPR, NFIN = Ly::NFIN, EL2 = Ly::EL2, EP2 = Ly::EP2;
  float mh[GT], lh[GT], th[GT];
  {
    float lsum[NFIN], tmax[NFIN];
#pragma unroll
    for (int kk = 0; kk < NFIN; ++kk) {
      lsum[kk] = st.l_run[kk];
      tmax[kk] = st.s_top[kk];
#pragma unroll
      for (int off = 1; off < 32; off *= 2)
        if ((off & Ly::HEAD_MASK) == 0) {
          lsum[kk] += __shfl_xor_sync(0xffffffffu, lsum[kk], off);
          tmax[kk] = fmaxf(tmax[kk], __shfl_xor_sync(0xffffffffu, tmax[kk], off));
        }
    }
#pragma unroll
    for (int h = 0; h < GT; ++h) {
      const int src = Ly::NV >= LPR ? h / NFIN : h * Ly::RED;
      mh[h] = __shfl_sync(0xffffffffu, st.m_run[h % NFIN], src);
      lh[h] = __shfl_sync(0xffffffffu, lsum[h % NFIN], src);
      th[h] = __shfl_sync(0xffffffffu, tmax[h % NFIN], src);
    }
  }
#pragma unroll
  for (int off = LPR; off < 32; off *= 2)
#pragma unroll
    for (int h = 0; h < GT; ++h)
#pragma unroll
      for (int e = 0; e < EL2; ++e) {
        st.acc[h][e].x += __shfl_xor_sync(0xffffffffu, st.acc[h][e].x, off);
        st.acc[h][e].y += __shfl_xor_sync(0xffffffffu, st.acc[h][e].y, off);
      }

  consumer_sync(cbar, cphase, lane, err);  // every warp is done with the stage
  float* mm = mstat;                // [NC][GT] running max (log2 units)
  float* ml = mstat + NC * GT;      // [NC][GT] running sum relative to mm
  float* mt = mstat + 2 * NC * GT;  // [NC][GT] largest logit
#pragma unroll
  for (int h = 0; h < GT; ++h)  // static indices keep mh/lh/th in registers
    if (lane == h) {
      mm[warp * GT + h] = mh[h];
      ml[warp * GT + h] = lh[h];
      mt[warp * GT + h] = th[h];
    }
  if (rg == 0) {
#pragma unroll
    for (int h = 0; h < GT; ++h)
#pragma unroll
      for (int kk = 0; kk < Ly::NPL; ++kk)
#pragma unroll
        for (int j2 = 0; j2 < EP2; ++j2)
          *reinterpret_cast<float2*>(&macc[(warp * GT + h) * D + (kk * LPR + c) * Ly::EPP + 2 * j2]) =
              st.acc[h][kk * EP2 + j2];
  }
  consumer_sync(cbar, cphase, lane, err);
  merge_warps<Ly, GT, D>(mstat, macc, cbar, cphase, G, warp, lane, v_scale, err, sink);
}

// The second half of a piece's end, shared by both consumer kinds: every warp
// has stored its running max, sum and largest logit per head (mstat) and its
// un-normalised output rows (macc); merge the NC warps and hand every (head,
// element) result to `sink`, then release the stage memory used as scratch.
template <typename Ly, int GT, int D, typename Sink>
__device__ __forceinline__ void merge_warps(const float* mstat, const float* macc, uint64_t* cbar,
                                            uint32_t& cphase, int G, int warp, int lane,
                                            float v_scale, unsigned* err, Sink&& sink) {
  constexpr int NC = Ly::NC;
  constexpr float kLn2 = 0.69314718055994530942f;
  const float* mm = mstat;
  const float* ml = mstat + NC * GT;
  const float* mt = mstat + 2 * NC * GT;
  for (int i = warp * 32 + lane; i < G * D; i += NC * 32) {
    const int h = i / D, d = i % D;
    float M = -INFINITY, T = -INFINITY;
#pragma unroll
    for (int w = 0; w < NC; ++w) {
      M = fmaxf(M, mm[w * GT + h]);
      T = fmaxf(T, mt[w * GT + h]);
    }
    float o = 0.f, lsum = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < NC; ++w) {
        const float lw = ml[w * GT + h];
        if (lw > 0.f) {
          const float f = exp2f(mm[w * GT + h] - M);
          lsum += lw * f;
          o += macc[(w * GT + h) * D + d] * f;
        }
      }
    }
    const bool any = M != -INFINITY && lsum > 0.f;
    sink(h, d, any ? o / lsum * v_scale : 0.f, any ? T * kLn2 : -INFINITY,
         any ? lsum * exp2f(M - T) : 0.f);
  }
  // the merge wrote the stage with ordinary stores; order them before the
  // bulk copies that will refill it
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  consumer_sync(cbar, cphase, lane, err);
}

// End of a piece on the tensor-core path: each warp stores its state per
// head (the running sum reduced over the 4 lanes of a head), then the warps
// are merged as on the CUDA-core path.
template <typename Ly, int GT, int D, typename Sink>
__device__ __forceinline__ void finish_piece_tc(TcState<D>& st, float* mstat, float* macc,
                                                uint64_t* cbar, uint32_t& cphase, int G,
                                                int warp, int lane, float v_scale, unsigned* err,
                                                Sink&& sink) {
  constexpr int NC = Ly::NC;
  const int g = lane >> 2, t = lane & 3;
  float l = st.l_run;
  l += __shfl_xor_sync(0xffffffffu, l, 1);
  l += __shfl_xor_sync(0xffffffffu, l, 2);
  consumer_sync(cbar, cphase, lane, err);  // every warp is done with the stage
  if (g < GT) {
    if (t == 0) {
      mstat[warp * GT + g] = st.m_run;
      mstat[NC * GT + warp * GT + g] = l;
      mstat[2 * NC * GT + warp * GT + g] = st.s_top;
    }
#pragma unroll
    for (int j = 0; j < D / 8; ++j)
      *reinterpret_cast<float2*>(&macc[(warp * GT + g) * D + 8 * j + 2 * t]) =
          make_float2(st.o[j][0], st.o[j][1]);
  }
  consumer_sync(cbar, cphase, lane, err);
  merge_warps<Ly, GT, D>(mstat, macc, cbar, cphase, G, warp, lane, v_scale, err, sink);
}

// End of a piece on the 8-bit tensor-core path: lane (g, t) holds heads 2t and
// 2t + 1; the running sums are reduced over the 8 lanes of a head, and the
// output is stored back in dim order (dims 4x .. 4x + 3 from tiles 2j, 2j+1).
template <typename Ly, int GT, int D, typename Sink>
__device__ __forceinline__ void finish_piece_tc8(Tc8State<D>& st, float* mstat, float* macc,
                                                 uint64_t* cbar, uint32_t& cphase, int G,
                                                 int warp, int lane, float v_scale, unsigned* err,
                                                 Sink&& sink) {
  constexpr int NC = Ly::NC;
  const int g = lane >> 2, t = lane & 3;
  float l[2] = {st.l_run[0], st.l_run[1]};
#pragma unroll
  for (int off = 4; off < 32; off *= 2) {
    l[0] += __shfl_xor_sync(0xffffffffu, l[0], off);
    l[1] += __shfl_xor_sync(0xffffffffu, l[1], off);
  }
  consumer_sync(cbar, cphase, lane, err);  // every warp is done with the stage
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int h = 2 * t + hh;
    if (h < GT) {
      if (g == 0) {
        mstat[warp * GT + h] = st.m_run[hh];
        mstat[NC * GT + warp * GT + h] = l[hh];
        mstat[2 * NC * GT + warp * GT + h] = st.s_top[hh];
      }
#pragma unroll
      for (int j = 0; j < D / 32; ++j)
        *reinterpret_cast<float4*>(&macc[(warp * GT + h) * D + 4 * (g + 8 * j)]) =
            make_float4(st.o[2 * j][hh], st.o[2 * j][2 + hh], st.o[2 * j + 1][hh],
                        st.o[2 * j + 1][2 + hh]);
    }
  }
  consumer_sync(cbar, cphase, lane, err);
  merge_warps<Ly, GT, D>(mstat, macc, cbar, cphase, G, warp, lane, v_scale, err, sink);
}

// Attended slots of sequence s (window- and table-limited); flags bad lengths.
__device__ __forceinline__ int attended_len(const DecodeParams& p, int s, int bs, bool flag) {
  const int n = p.context_lens[s];
  const int cap = p.max_blocks_per_seq * bs;
  if (n < 0) {
    if (flag) raise_error(p.err, PA_DEVERR_CONTEXT_LEN);
    return 0;
  }
  if (p.window > 0) return n < p.window ? n : p.window;
  if (n > cap) {
    if (flag) raise_error(p.err, PA_DEVERR_CONTEXT_LEN);
    return cap;
  }
  return n;
}

__device__ __forceinline__ int warp_sum_int(int v) {
#pragma unroll
  for (int off = 16; off >= 1; off /= 2) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Balanced mode. The work is the flattened (sequence, kv head, page) order of
// P pages; CTA c of C streams pages [lo(c), lo(c+1)) with lo(c) = c*P/C.
// cta_of(x) is the CTA whose range holds flattened page x.
__device__ __forceinline__ long long range_lo(int c, long long P, int C) {
  return (long long)c * P / C;
}
__device__ __forceinline__ int cta_of(long long x, long long P, int C) {
  return static_cast<int>(((x + 1) * C - 1) / P);
}

// Partial slot (cta * 2 + slot) of the j-th piece of the cut segment that
// covers flattened pages [seg0, seg0 + pages); c_first = cta_of(seg0). With
// P >= C every CTA holds at least one page, so the pieces sit in CTAs
// c_first, c_first + 1, ...; with P < C every CTA holds at most one page and
// piece j sits in cta_of(seg0 + j). Only the first piece can be a CTA's
// second piece (its range began with the end of another segment).
__device__ __forceinline__ int piece_index(int j, long long seg0, long long P, int C,
                                           int c_first, bool first_in_slot1) {
  const int cc = P >= C ? c_first + j : cta_of(seg0 + j, P, C);
  return cc * kPieceSlots + ((j == 0 && first_in_slot1) ? 1 : 0);
}

// Log-sum-exp combination of a cut segment's pieces into its G output rows,
// run by `nwarps` warps of the CTA whose piece arrived last (warp w takes
// heads w, w + nwarps, ...; a lane takes D / 32 elements of the row). Each
// piece holds its normalised output o_j, its largest logit m_j and the sum
// l_j of exp(logit - m_j); the segment's output is
//   sum_j l_j exp(m_j - M) o_j / sum_j l_j exp(m_j - M),  M = max_j m_j,
// accumulated here with a running maximum, four pieces per round of loads.
// The pieces were written by other CTAs of this launch: they are read
// through L2 (ld.global.cg), after the acquire of the caller.
template <typename QT, typename Ly, int GT, int D>
__device__ __forceinline__ void combine_segment(const DecodeParams& p, QT* out, long long seg0,
                                                int pages, long long P, int C, int G, int warp,
                                                int nwarps, int lane) {
  constexpr int DPL = D / 32, U = 4;
  static_assert(D % 32 == 0, "a lane takes D / 32 elements of a row");
  const int c_first = cta_of(seg0, P, C);
  const bool first_in_slot1 = seg0 != range_lo(c_first, P, C);
  const int n = P >= C ? cta_of(seg0 + pages - 1, P, C) - c_first + 1 : pages;
  const float2* mlp = reinterpret_cast<const float2*>(p.piece_ml);
  for (int h = warp; h < G; h += nwarps) {
    float M = -INFINITY, lsum = 0.f, acc[DPL];
#pragma unroll
    for (int t = 0; t < DPL; ++t) acc[t] = 0.f;
    for (int j0 = 0; j0 < n; j0 += U) {
      float2 ml[U];
      float o[U][DPL];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        ml[u] = make_float2(-INFINITY, 0.f);
#pragma unroll
        for (int t = 0; t < DPL; ++t) o[u][t] = 0.f;
        if (j0 + u < n) {
          const size_t b =
              (size_t)piece_index(j0 + u, seg0, P, C, c_first, first_in_slot1) * GT + h;
          ml[u] = __ldcg(mlp + b);
#pragma unroll
          for (int t = 0; t < DPL; ++t) o[u][t] = __ldcg(p.piece_o + b * D + lane + 32 * t);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (ml[u].y > 0.f) {
          if (ml[u].x > M) {
            const float f = expf(M - ml[u].x);
            lsum *= f;
#pragma unroll
            for (int t = 0; t < DPL; ++t) acc[t] *= f;
            M = ml[u].x;
          }
          const float w = ml[u].y * expf(ml[u].x - M);
          lsum += w;
#pragma unroll
          for (int t = 0; t < DPL; ++t) acc[t] = fmaf(w, o[u][t], acc[t]);
        }
      }
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
#pragma unroll
    for (int t = 0; t < DPL; ++t) out[h * D + lane + 32 * t] = Elem<QT>::from_f32(acc[t] * inv);
  }
}

// A cut piece the producer still has to count (balanced mode), kept in
// shared memory while the CTA streams on.
struct CutPiece {
  long long seg0;  // flattened index of its segment's first page
  int pages;       // pages of the segment
  int len;         // pages of the piece
  int row;         // first output row of the segment (s * Hq + g * G)
  int pad;
};
static_assert(sizeof(CutPiece) == 24, "two records fit the misc area");

// Balanced mode, producer warp: count a finished cut piece (cp.len pages of
// the segment at flattened pages [cp.seg0, cp.seg0 + cp.pages), output rows
// from cp.row) and combine the segment if this piece completes it. The consumers' stores
// of the piece are ordered before this through the stage's empty barrier
// (release/acquire, CTA scope); lane 0's fence then makes them visible at
// device scope before the count, and after a completing count orders the
// other pieces' stores before the combine's loads.
template <typename QT, typename Ly, int GT, int D>
__device__ __forceinline__ void publish_piece(const DecodeParams& p, const CutPiece& cp,
                                              long long P, int C, int G, int lane) {
  const long long seg0 = cp.seg0;
  const int pages = cp.pages, len = cp.len, row = cp.row;
  int last = 0;
  if (lane == 0) {
    int* cnt = p.arrived + cta_of(seg0 + pages - 1, P, C);
    fence_acq_rel_gpu();
    const int before = atomicAdd(cnt, len);
    last = before + len == pages ? 1 : 0;
    if (last) {
      *cnt = 0;  // nobody else touches it in this launch: leave it zero
      fence_acq_rel_gpu();
    }
  }
  __syncwarp();
  last = __shfl_sync(0xffffffffu, last, 0);
  if (last)
    combine_segment<QT, Ly, GT, D>(p, reinterpret_cast<QT*>(p.out) + (size_t)row * D, seg0, pages,
                                   P, C, G, 0, 1, lane);
}

template <typename QT, typename CT, int D, int GT, int BS, int MODE>
__device__ __forceinline__ void decode_body(const DecodeParams& p) {
  using Ly = Layout<QT, CT, D, GT, BS, MODE>;
  constexpr int NC = Ly::NC, STAGES = Ly::STAGES, R = Ly::R, TPW = Ly::TPW;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // the tensor-core layout's swizzled boxes need 1024-byte aligned stages
  uint8_t* smem = smem_raw;
  if constexpr (Ly::TMA)
    smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hq = p.num_heads, Hkv = p.num_kv_heads, G = p.group;
  const int MB = p.max_blocks_per_seq;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Ly::OFF_BAR);
  uint64_t* empty = full + STAGES;
  uint64_t* cbar = empty + STAGES;  // consumer-to-consumer barrier
  int4* desc = reinterpret_cast<int4*>(smem + Ly::OFF_DESC);
  int* misc = reinterpret_cast<int*>(smem + Ly::OFF_MISC);
  long long* misc64 = reinterpret_cast<long long*>(smem + Ly::OFF_MISC + 16);

  // ---------------------------------------------------------- work of this CTA
  // Both modes end up with: start segment (s0, g0), start page pg0 in it, and
  // npages pages to stream (crossing segments only in balanced mode).
  int s0, g0, pg0, npages;
  if constexpr (MODE == kModeSplit) {
    const int split = blockIdx.x;
    g0 = blockIdx.y;
    s0 = blockIdx.z;
    const int L = attended_len(p, s0, BS, threadIdx.x == 0 && split == 0 && g0 == 0);
    const int total = (L + BS - 1) / BS;
    pg0 = p.first_page + split * p.pages_per_split;
    npages = min(total, pg0 + p.pages_per_split) - pg0;
    if (npages <= 0) {  // nothing attended in this split (uniform for the CTA)
      for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
        const int h = i / D, d = i % D;
        const size_t row = (size_t)s0 * Hq + (size_t)g0 * G + h;
        if (p.partials) {
          if (d == 0) {
            p.max_logits[row * p.num_splits + split] = -INFINITY;
            p.exp_sums[row * p.num_splits + split] = 0.f;
          }
        } else {
          reinterpret_cast<QT*>(p.out)[row * D + d] = Elem<QT>::from_f32(0.f);
        }
      }
      return;
    }
  } else {
    const int cta = blockIdx.x, C = gridDim.x, S = p.num_seqs;
    if (warp < NC) {
      // sequences with nothing to attend get zero rows (CTA c takes c, c + C,
      // ...); impossible lengths are flagged here, once per sequence
      for (int s = cta; s < S; s += C)
        if (attended_len(p, s, BS, threadIdx.x == 0) == 0) {
          QT* o = reinterpret_cast<QT*>(p.out) + (size_t)s * Hq * D;
          for (int i = threadIdx.x; i < Hq * D; i += NC * 32) o[i] = Elem<QT>::from_f32(0.f);
        }
    } else {
      // total pages, then this CTA's equal share [lo, hi) of the flattened
      // (sequence, kv head, page) order, then where lo falls
      long long total = 0;
      for (int b = 0; b < S; b += 32) {
        const int s = b + lane;
        const int pg = s < S ? (attended_len(p, s, BS, false) + BS - 1) / BS : 0;
        total += warp_sum_int(pg);
      }
      const long long P = total * Hkv;
      const long long lo = range_lo(cta, P, C), hi = range_lo(cta + 1, P, C);
      int ls0 = 0, lg0 = 0, lpg0 = 0;
      if (lo < hi) {
        long long run = 0;  // pages of the sequences before this chunk
        for (int b = 0; b < S; b += 32) {
          const int s = b + lane;
          const int pg = s < S ? (attended_len(p, s, BS, false) + BS - 1) / BS : 0;
          int incl = pg;  // inclusive prefix within the chunk
#pragma unroll
          for (int off = 1; off < 32; off *= 2) {
            const int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
          }
          const unsigned hit = __ballot_sync(0xffffffffu, s < S && (run + incl) * Hkv > lo);
          if (hit) {
            const int src = __ffs(hit) - 1;
            const int pgs = __shfl_sync(0xffffffffu, pg, src);
            const long long before = run + __shfl_sync(0xffffffffu, incl, src) - pgs;
            const long long rem = lo - before * Hkv;
            ls0 = b + src;
            lg0 = static_cast<int>(rem / pgs);
            lpg0 = static_cast<int>(rem % pgs);
            break;
          }
          run += __shfl_sync(0xffffffffu, incl, 31);
        }
      }
      if (lane == 0) {
        misc[0] = ls0;
        misc[1] = lg0;
        misc[2] = lpg0;
        misc[3] = static_cast<int>(hi - lo);
        misc64[0] = lo;
        misc64[1] = P;
      }
    }
    __syncthreads();
    s0 = misc[0];
    g0 = misc[1];
    pg0 = misc[2];
    npages = misc[3];
    if (npages <= 0) return;
  }

  if (threadIdx.x == 0) {
#pragma unroll
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], NC);
    }
    mbar_init(cbar, NC);
    fence_mbar_init();
  }
  __syncthreads();

  // ======================================================== producer warp
  if (warp == NC) {
    const size_t blk_stride = (size_t)Hkv * Ly::PAGE;
    const uint32_t qbytes = static_cast<uint32_t>(G) * D * Ly::QB;
    int s = s0, g = g0, pg = pg0;
    int L = attended_len(p, s, BS, false);
    int pages = (L + BS - 1) / BS;
    int tb_s = -1, tb_base = 0, tbl = -1;  // 32 table entries cached across lanes
    bool piece_start = true;
    int piece_flags = 0, piece_end = 0, issued = 0;
    bool aborted = false;
    // balanced mode: the CTA's range start and the total page count, and the
    // CTA's cut pieces: the head piece (the range starts inside its segment
    // and goes on past it), counted here once the consumers have finished
    // it, and the tail piece (the range ends inside its segment), recorded
    // for the consumers, who count it themselves at the end
    long long lo = 0, P = 1;
    if constexpr (MODE == kModeBalanced) {
      lo = misc64[0];
      P = misc64[1];
    }
    CutPiece* cut = reinterpret_cast<CutPiece*>(smem + Ly::OFF_MISC + 32);  // head, tail
    bool h_on = false;
    int h_k = 0;
    for (int k = 0; k < npages; ++k) {
      if (s != tb_s || pg < tb_base || pg >= tb_base + 32) {
        tb_s = s;
        tb_base = pg;
        const int idx = pg + lane;
        tbl = idx < pages ? __ldg(p.block_tables + (size_t)s * MB + idx) : -1;
      }
      const int bid = __shfl_sync(0xffffffffu, tbl, pg - tb_base);
      if (piece_start) {
        const int len = min(pages - pg, npages - k);
        piece_end = k + len - 1;
        piece_flags = (pg == 0 ? kSegFirst : 0) | (pg + len == pages ? kSegLast : 0) |
                      (k > 0 ? kSlot1 : 0);
        if constexpr (MODE == kModeBalanced) {
          if (pg != 0 || pg + len != pages) {  // cut
            const bool tail = k + len == npages;
            if (!tail) {
              h_on = true;
              h_k = len - 1;
            }
            // the consumers read the tail record after the piece's full
            // barriers, which this write precedes
            if (lane == 0) cut[tail ? 1 : 0] = CutPiece{lo + k - pg, pages, len, s * Hq + g * G, 0};
            __syncwarp();
          }
        }
      }
      const int slot = k % STAGES;
      if (lane == 0) {
        if (k >= STAGES && !mbar_wait_bounded(&empty[slot], ((k / STAGES) - 1) & 1)) {
          raise_error(p.err, PA_DEVERR_TIMEOUT);
          aborted = true;
        }
        if (k == p.unarmed_page) aborted = true;  // test hook: issue nothing more
        if (!aborted) {
          const bool ok = bid >= 0 && bid < p.num_blocks;
          if (!ok) raise_error(p.err, PA_DEVERR_BLOCK_ID);
          const int rows = ok ? min(BS, L - pg * BS) : 0;
          const int flags = piece_flags | (piece_start ? kFirst : 0) | (k == piece_end ? kLast : 0) |
                            (k == npages - 1 ? kCtaLast : 0);
          desc[slot] = make_int4(rows, s * Hkv + g, flags, 0);
          uint8_t* stage = smem + slot * Ly::STAGE;
          const uint32_t bytes =
              (ok ? 2u * (Ly::PAGE + Ly::SCB) : 0u) + (piece_start ? qbytes : 0u);
          if (bytes) {
            mbar_arrive_expect_tx(&full[slot], bytes);
            if (ok && Ly::TMA) {
              // one tensor copy per 128-byte-wide box of the K page and of the V page
              const int y = (bid * Hkv + g) * BS;
#pragma unroll
              for (int j = 0; j < Ly::BOXES; ++j) {
                tma_load_2d(stage + j * Ly::BOXB, &p.tm_k, (128 / Ly::EB) * j, y, &full[slot]);
                tma_load_2d(stage + Ly::PAGE + j * Ly::BOXB, &p.tm_v, (128 / Ly::EB) * j, y,
                            &full[slot]);
              }
            } else if (ok) {
              const size_t off = (size_t)bid * blk_stride + (size_t)g * Ly::PAGE;
              bulk_g2s(stage, p.k_cache + off, Ly::PAGE, &full[slot]);
              bulk_g2s(stage + Ly::PAGE, p.v_cache + off, Ly::PAGE, &full[slot]);
            }
            if constexpr (Ly::ROW_SCALES) {
              if (ok) {
                const size_t so = ((size_t)bid * Hkv + g) * BS;
                bulk_g2s(stage + 2 * Ly::PAGE, p.k_scales + so, Ly::SCB, &full[slot]);
                bulk_g2s(stage + 2 * Ly::PAGE + Ly::SCB, p.v_scales + so, Ly::SCB, &full[slot]);
              }
            }
            if (piece_start)
              bulk_g2s(stage + Ly::OFF_Q,
                       static_cast<const uint8_t*>(p.query) +
                           ((size_t)s * Hq + (size_t)g * G) * D * Ly::QB,
                       qbytes, &full[slot]);
          } else {
            mbar_arrive(&full[slot]);
          }
          ++issued;
        }
      }
      if (__shfl_sync(0xffffffffu, aborted ? 1 : 0, 0)) break;
      if constexpr (MODE == kModeBalanced) {
        // the wait above saw the head piece's last stage released: count it
        // now, with this iteration's copies already in flight
        if (h_on && k == h_k + STAGES) {
          publish_piece<QT, Ly, GT, D>(p, cut[0], P, gridDim.x, G, lane);
          h_on = false;
        }
      }
      // advance to the next page of the walk
      piece_start = false;
      ++pg;
      if (k == piece_end) {
        piece_start = true;
        if constexpr (MODE == kModeBalanced) {
          if (pg == pages && k + 1 < npages) {
            pg = 0;
            if (++g == Hkv) {
              g = 0;
              do {
                ++s;
                L = attended_len(p, s, BS, false);
                pages = (L + BS - 1) / BS;
              } while (pages == 0 && s + 1 < p.num_seqs);
            }
          }
        }
      }
    }
    // never leave the CTA with copies in flight: wait for the last fill of
    // every stage (already complete in the normal case)
    if (lane == 0) {
      for (int k = issued > STAGES ? issued - STAGES : 0; k < issued; ++k)
        if (!mbar_wait_bounded(&full[k % STAGES], (k / STAGES) & 1))
          raise_error(p.err, PA_DEVERR_TIMEOUT);
    }
    if constexpr (MODE == kModeBalanced) {
      // a head piece whose last stage was not reused: wait for the consumers
      // to release it, then count it (skipped after any timeout)
      if (h_on && __shfl_sync(0xffffffffu, aborted ? 0 : 1, 0)) {
        int got = 1;
        if (lane == 0 && !mbar_wait_bounded(&empty[h_k % STAGES], (h_k / STAGES) & 1)) {
          raise_error(p.err, PA_DEVERR_TIMEOUT);
          got = 0;
        }
        if (__shfl_sync(0xffffffffu, got, 0))
          publish_piece<QT, Ly, GT, D>(p, cut[0], P, gridDim.x, G, lane);
      }
    }
    return;
  }

  // ======================================================== consumer warps
  const int c = lane % Ly::LPR;   // piece column of the row
  const int rg = lane / Ly::LPR;  // row within a warp step
  float* wscr = reinterpret_cast<float*>(smem + Ly::OFF_SCR) + warp * Ly::SCR;
  float* mstat = reinterpret_cast<float*>(smem + Ly::OFF_MSTAT);
  uint32_t cphase = 0;
  typename std::conditional<
      Ly::TC, TcState<D>,
      typename std::conditional<Ly::TC8, Tc8State<D>, PieceState<Ly, GT>>::type>::type st;
  // end of a piece: the consumer kind's own reduction, then the shared merge
  auto finish = [&](float* macc, auto&& sink) {
    if constexpr (Ly::TC)
      finish_piece_tc<Ly, GT, D>(st, mstat, macc, cbar, cphase, G, warp, lane, p.v_scale, p.err,
                                 sink);
    else if constexpr (Ly::TC8)
      finish_piece_tc8<Ly, GT, D>(st, mstat, macc, cbar, cphase, G, warp, lane, p.v_scale,
                                  p.err, sink);
    else
      finish_piece<Ly, GT, D>(st, mstat, macc, cbar, cphase, G, warp, lane, c, rg, p.v_scale,
                              p.err, sink);
  };

  int k = 0;
  bool aborted = false, tail_cut = false;
  while (true) {
    // up to R pages of the current piece
    const uint8_t* Kp[R];
    const uint8_t* Vp[R];
    const float* Ks[R];
    const float* Vs[R];
    int lim[R], rows[R];
    int n_here = 0, last_flags = 0, seg = 0, last_slot = 0;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      lim[r] = 0;
      rows[r] = 0;
      Kp[r] = smem;
      Vp[r] = smem;
      Ks[r] = reinterpret_cast<const float*>(smem);
      Vs[r] = reinterpret_cast<const float*>(smem);
      if (aborted || (r > 0 && (last_flags & kLast))) continue;
      const int slot = (k + r) % STAGES;
      if (!mbar_wait_bounded(&full[slot], ((k + r) / STAGES) & 1)) {
        raise_error(p.err, PA_DEVERR_TIMEOUT);
        aborted = true;
        continue;
      }
      const int4 d = desc[slot];
      uint8_t* stage = smem + slot * Ly::STAGE;
      if (r == 0) {
        seg = d.y;
        if (d.z & kFirst) {
          if constexpr (Ly::TC)
            begin_piece_tc<QT, D>(st, stage + Ly::OFF_Q, G, lane);
          else if constexpr (Ly::TC8)
            begin_piece_tc8<QT, D>(st, stage + Ly::OFF_Q, G, lane);
          else
            begin_piece<QT, Ly, GT, D>(st, stage + Ly::OFF_Q, G, c, p.q_scale);
        }
      }
      Kp[r] = stage;
      Vp[r] = stage + Ly::PAGE;
      Ks[r] = reinterpret_cast<const float*>(stage + 2 * Ly::PAGE);
      Vs[r] = reinterpret_cast<const float*>(stage + 2 * Ly::PAGE + Ly::SCB);
      lim[r] = d.x - warp * TPW;
      rows[r] = d.x;
      last_flags = d.z;
      last_slot = slot;
      n_here = r + 1;
    }
    if (__any_sync(0xffffffffu, aborted)) break;

    if constexpr (Ly::TC)
      process_tc<QT, Ly, D>(st, Kp, Vp, rows, warp, lane, p.q_scale, G);
    else if constexpr (Ly::TC8)
      process_tc8<Ly, CT, D>(st, Kp, Vp, Ks, Vs, rows, warp, lane, p.q_scale);
    else
      process_pages<CT, Ly, GT>(st, Kp, Vp, Ks, Vs, lim, wscr, warp, lane, c, rg);

    const bool ends_piece = (last_flags & kLast) != 0;
    if (lane == 0) {
      for (int r = 0; r < n_here - (ends_piece ? 1 : 0); ++r) mbar_arrive(&empty[(k + r) % STAGES]);
    }
    if (ends_piece) {
      float* macc = Ly::MERGE_IN_STAGE
                        ? reinterpret_cast<float*>(smem + last_slot * Ly::STAGE)
                        : reinterpret_cast<float*>(smem + Ly::OFF_MACC);
      const int s = seg / Hkv, g = seg % Hkv;
      if constexpr (MODE == kModeSplit) {
        const int split = blockIdx.x, nsplit = p.num_splits;
        const bool partials = p.partials != 0;
        QT* out = reinterpret_cast<QT*>(p.out);
        float* tmp_out = p.tmp_out;
        float* max_logits = p.max_logits;
        float* exp_sums = p.exp_sums;
        const size_t row0 = (size_t)s * Hq + (size_t)g * G;
        finish(macc, [=](int h, int d, float o, float m_nat, float l) {
              const size_t row = row0 + h;
              if (partials) {
                const size_t pi = row * nsplit + split;
                if (l > 0.f) tmp_out[pi * D + d] = o;
                if (d == 0) {
                  max_logits[pi] = m_nat;
                  exp_sums[pi] = l;
                }
              } else {
                out[row * D + d] = Elem<QT>::from_f32(o);
              }
            });
        if (lane == 0) mbar_arrive(&empty[last_slot]);
      } else {
        const bool whole = (last_flags & kSegFirst) && (last_flags & kSegLast);
        const int pslot = (last_flags & kSlot1) ? 1 : 0;
        const size_t base = (size_t)blockIdx.x * kPieceSlots + pslot;
        QT* out = reinterpret_cast<QT*>(p.out) + ((size_t)s * Hq + (size_t)g * G) * D;
        float* piece_o = p.piece_o + base * GT * D;
        float* piece_ml = p.piece_ml + base * GT * 2;
        finish(macc, [=](int h, int d, float o, float m_nat, float l) {
              if (whole) {
                out[h * D + d] = Elem<QT>::from_f32(o);
              } else {
                piece_o[h * D + d] = o;
                if (d == 0) {
                  piece_ml[h * 2 + 0] = m_nat;
                  piece_ml[h * 2 + 1] = l;
                }
              }
            });
        // the merge is done with the stage; for a head piece this release also
        // tells the producer that the piece's rows are stored
        if (lane == 0) mbar_arrive(&empty[last_slot]);
        tail_cut = !whole && (last_flags & kCtaLast);
      }
    }
    k += n_here;
    if (last_flags & kCtaLast) break;
  }
  if constexpr (MODE == kModeBalanced) {
    if (tail_cut) {
      // The tail piece, counted here. If every other piece of its segment
      // has been counted already, it completes the segment and needs no
      // counting; otherwise count it (the consumer barrier that ended
      // finish_piece ordered every thread's rows before lane 0's fence).
      const CutPiece cp = *reinterpret_cast<const CutPiece*>(smem + Ly::OFF_MISC + 32 + 24);
      const long long P = misc64[1];
      if (warp == 0 && lane == 0) {
        int* cnt = p.arrived + cta_of(cp.seg0 + cp.pages - 1, P, gridDim.x);
        int last = ld_acquire_gpu(cnt) + cp.len == cp.pages ? 1 : 0;
        // completing without counting: this CTA's own rows of the piece still
        // have to reach device scope, since the combine reads them (like every
        // other piece) through L2
        if (last) fence_acq_rel_gpu();
        if (!last) {
          fence_acq_rel_gpu();
          last = atomicAdd(cnt, cp.len) + cp.len == cp.pages ? 1 : 0;
          if (last) fence_acq_rel_gpu();
        }
        if (last) *cnt = 0;  // leave it zero for the next launch
        misc[8] = last;
      }
      consumer_sync(cbar, cphase, lane, p.err);
      if (misc[8])
        combine_segment<QT, Ly, GT, D>(p, reinterpret_cast<QT*>(p.out) + (size_t)cp.row * D,
                                       cp.seg0, cp.pages, P, gridDim.x, G, warp, NC, lane);
    }
  }
}

template <typename QT, typename CT, int D, int GT, int BS, int MODE>
__global__ void __launch_bounds__(Layout<QT, CT, D, GT, BS, MODE>::THREADS,
                                  Layout<QT, CT, D, GT, BS, MODE>::MIN_CTAS)
    paged_decode_kernel(const __grid_constant__ DecodeParams p) {
  if constexpr (MODE == kModeSplit) {
    if (!p.join_at_end) pdl_wait();
    pdl_trigger();
    decode_body<QT, CT, D, GT, BS, MODE>(p);
    if (p.join_at_end) pdl_wait();
  } else {
    pdl_wait();
    pdl_trigger();
    decode_body<QT, CT, D, GT, BS, MODE>(p);
  }
}

// Host side: launch one instantiation in the given mode. In balanced mode a
// grid.x of 0 asks for the kernel's resident capacity (SMs x CTAs per SM,
// at most kMaxBalancedCtas); the grid size used is returned in *ctas.
template <typename QT, typename CT, int D, int GT, int BS, int MODE>
cudaError_t launch_decode(const DecodeParams& prm, dim3 grid, int* ctas, cudaStream_t stream) {
  using Ly = Layout<QT, CT, D, GT, BS, MODE>;
  auto kern = paged_decode_kernel<QT, CT, D, GT, BS, MODE>;
  static int configured_devices = 0;  // bit per device id < 32
  static int capacity[32] = {};       // resident CTAs per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 32 || !(__atomic_load_n(&configured_devices, __ATOMIC_ACQUIRE) & (1 << dev))) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::SMEM);
    if (e != cudaSuccess) return e;
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, Ly::THREADS, Ly::SMEM);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long long C = (long long)sms * (per_sm > 0 ? per_sm : 1);
    if (dev < 32) {
      capacity[dev] = static_cast<int>(C < kMaxBalancedCtas ? C : kMaxBalancedCtas);
      __atomic_fetch_or(&configured_devices, 1 << dev, __ATOMIC_RELEASE);
    }
  }
  if (MODE == kModeBalanced && grid.x == 0)
    grid.x = dev < 32 && capacity[dev] > 0 ? capacity[dev] : kMaxBalancedCtas;
  if (ctas) *ctas = static_cast<int>(grid.x);
  return launch_pdl(kern, grid, dim3(Ly::THREADS), Ly::SMEM, stream, prm);
}

// Dispatch over (head_dim, group bucket, block size) for one (QT, CT) pair.
template <typename QT, typename CT>
cudaError_t dispatch_decode(const DecodeParams& prm, dim3 grid, int D, int GT, int BS, int mode,
                            int* ctas, cudaStream_t stream) {
#define PA_CASE_BS(D_, GT_)                                                                     \
  switch (BS) {                                                                                 \
    case 16:                                                                                    \
      return mode == kModeSplit                                                                 \
                 ? launch_decode<QT, CT, D_, GT_, 16, kModeSplit>(prm, grid, ctas, stream)      \
                 : launch_decode<QT, CT, D_, GT_, 16, kModeBalanced>(prm, grid, ctas, stream);  \
    case 32:                                                                                    \
      return mode == kModeSplit                                                                 \
                 ? launch_decode<QT, CT, D_, GT_, 32, kModeSplit>(prm, grid, ctas, stream)      \
                 : launch_decode<QT, CT, D_, GT_, 32, kModeBalanced>(prm, grid, ctas, stream);  \
    case 64:                                                                                    \
      return mode == kModeSplit                                                                 \
                 ? launch_decode<QT, CT, D_, GT_, 64, kModeSplit>(prm, grid, ctas, stream)      \
                 : launch_decode<QT, CT, D_, GT_, 64, kModeBalanced>(prm, grid, ctas, stream);  \
    default:                                                                                    \
      return cudaErrorInvalidValue;                                                             \
  }
#define PA_CASE_GT(D_)                     \
  switch (GT) {                            \
    case 1: PA_CASE_BS(D_, 1)              \
    case 2: PA_CASE_BS(D_, 2)              \
    case 4: PA_CASE_BS(D_, 4)              \
    case 8: PA_CASE_BS(D_, 8)              \
    default: return cudaErrorInvalidValue; \
  }
  switch (D) {
    case 64: PA_CASE_GT(64)
    case 96: PA_CASE_GT(96)
    case 128: PA_CASE_GT(128)
    default: return cudaErrorInvalidValue;
  }
#undef PA_CASE_GT
#undef PA_CASE_BS
}

}  // namespace pa

// One translation unit per (query dtype, cache dtype) pair defines these.
#define PA_DECLARE_DISPATCH(NAME)                                                       \
  cudaError_t NAME(const pa::DecodeParams& prm, dim3 grid, int D, int GT, int BS,      \
                   int mode, int* ctas, cudaStream_t stream)
PA_DECLARE_DISPATCH(pa_dispatch_decode_f32_f32);
PA_DECLARE_DISPATCH(pa_dispatch_decode_bf16_bf16);
PA_DECLARE_DISPATCH(pa_dispatch_decode_f16_f16);
PA_DECLARE_DISPATCH(pa_dispatch_decode_f32_e4m3);
PA_DECLARE_DISPATCH(pa_dispatch_decode_bf16_e4m3);
PA_DECLARE_DISPATCH(pa_dispatch_decode_f16_e4m3);
PA_DECLARE_DISPATCH(pa_dispatch_decode_bf16_i8);
PA_DECLARE_DISPATCH(pa_dispatch_decode_f16_i8);
