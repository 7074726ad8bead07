// pa_decode.cuh -- split-context paged decode attention kernel for sm_103a.
//
// What it computes ("PagedAttention in mistral.rs": blocked K/V pool read
// through per-sequence block tables, optional FP8 E4M3 cache; "Rolling buffer
// cache": a window of W slots): for sequence s, kv head g and the G query
// heads sharing it, softmax(q K^T * scale) V over the attended slots
// [0, L_s), restricted to this CTA's split of pages.
//
// One CTA = one (split, kv head, sequence). Warp roles:
//   * producer warp (last warp): reads the split's block-table entries and,
//     per page, issues two 1-D bulk asynchronous copies (K page, V page; each
//     bs*D contiguous elements of the head-major layout) into a ring of
//     STAGES shared-memory stages, completion tracked by "full" mbarriers;
//     waits on "empty" mbarriers before reusing a stage.
//   * NC = bs/8 consumer warps: each owns 8 rows (tokens) of every page.
//     A lane covers LPR-th of a row (EPL elements of D, in PB-byte pieces
//     interleaved across the LPR lanes of the row, so every shared-memory
//     load instruction of a row reads contiguous bytes). Per page:
//       1. partial dot products q.k for (token, head) pairs, then a
//          transposing butterfly reduction across the LPR lanes (each level
//          halves the values a lane keeps, so a warp spends ~1 shuffle per
//          (token, head) instead of log2(LPR));
//       2. online softmax per head over the warp's 8 tokens (running max and
//          sum in log2 units; q is pre-scaled by scale*log2(e)*k_scale);
//       3. P.V accumulation into per-lane fp32 accumulators, skipping rows
//          past L_s (never multiplying a weight by a stale or NaN value).
//     At the end the NC warps' (m, l, acc) are merged through shared memory
//     and written either as the final output (one split) or as a split
//     partial (m in natural-log units, l, acc / l) for the LSE reduction.
// Each K/V byte of the split is read from HBM exactly once per kv head.
#pragma once

#include "pa_device.cuh"

namespace pa {

struct DecodeParams {
  void* out;           // [S][Hq][D] of QT (final mode)
  float* tmp_out;      // [S][Hq][NS][D]  (partials mode)
  float* max_logits;   // [S][Hq][NS]
  float* exp_sums;     // [S][Hq][NS]
  const void* query;   // [S][Hq][D] of QT
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const int32_t* block_tables;  // [S][MB]
  const int32_t* context_lens;  // [S]
  unsigned* err;
  int num_heads, num_kv_heads, group;  // group = G (runtime, <= template GT)
  int num_blocks, max_blocks_per_seq, window;
  int num_splits, pages_per_split;
  int partials;   // 1: split partials, 0: final output
  float q_scale;  // scale * log2(e) (* k_scale for FP8)
  float v_scale;  // FP8: v_scale, else 1
};

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

constexpr int cmin(int a, int b) { return a < b ? a : b; }
constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }
constexpr int cmax(int a, int b) { return a > b ? a : b; }

// Lanes per row: the fewest (>= 4) that keep q and acc at <= 32 fp32 each with
// an even number of elements per lane (they are processed as fp32 pairs);
// failing that, the most lanes that still give an even count.
constexpr int choose_lpr(int D, int GT) {
  for (int l = 4; l <= 32; l *= 2)
    if (D % l == 0 && (D / l) % 2 == 0 && (D / l) * GT <= 32) return l;
  for (int l = 32; l >= 4; l /= 2)
    if (D % l == 0 && (D / l) % 2 == 0) return l;
  return 4;
}
constexpr int choose_pb(int bytes) {
  return bytes % 16 == 0 ? 16 : bytes % 8 == 0 ? 8 : bytes % 4 == 0 ? 4 : bytes % 2 == 0 ? 2 : 1;
}

template <typename CT, int D, int GT, int BS>
struct Layout {
  static constexpr int EB = Elem<CT>::bytes;
  static constexpr int ROWB = D * EB;      // bytes of one cached row
  static constexpr int PAGE = BS * ROWB;   // bytes of one (block, kv head) page
  static constexpr int TPW = 8;            // rows per consumer warp per page
  static constexpr int NC = BS / TPW;      // consumer warps
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
  // pages a consumer warp takes per iteration (one softmax round per R pages)
  static constexpr int R = (2 * PAGE <= 16384) ? PA_PAGES_PER_ITER : 1;
  static constexpr int TPI = TPW * R;      // rows per warp per iteration
  static constexpr int NSTI = NST * R;     // steps per iteration
  static constexpr int SG = cmin(NSTI, cmax(1, 16 / GT));  // steps per reduction group
  static constexpr int NV = SG * GT;       // partial dot products per group
  static constexpr int NFIN = cmax(NV / LPR, 1);   // reduced values a lane holds
  static constexpr int RED = NV < LPR ? LPR / NV : 1;  // lanes holding the same value
  static constexpr int NG = NSTI / SG;               // reduction groups per iteration
  // After the reduction lane c (of a row) holds value index (c*NV)/LPR + kk,
  // head = index % GT. Lane bits [HB0, HB0 + NHB) of c select the head;
  // the other lane bits only select tokens (or redundant copies).
  static constexpr int HB0 = NV >= LPR ? 0 : ilog2(RED);
  static constexpr int NHB = NV >= LPR ? ilog2(cmax(GT / NFIN, 1)) : ilog2(GT);
  static constexpr int HEAD_MASK = ((1 << NHB) - 1) << HB0;
  static constexpr int STAGES = cmax(2 * R, cmin(PA_MAX_STAGES, PA_STAGE_BYTES / (2 * PAGE)));
  static constexpr int SCR = (TPI * GT + GT + 3) / 4 * 4;  // per-warp scratch floats
  // dynamic shared memory layout
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = STAGES * PAGE;
  static constexpr int OFF_BAR = 2 * STAGES * PAGE;
  static constexpr int OFF_OK = OFF_BAR + 2 * STAGES * 8;
  static constexpr int OFF_SCR = (OFF_OK + STAGES * 4 + 15) / 16 * 16;
  static constexpr int SMEM = OFF_SCR + NC * SCR * 4;
  // end-of-split merge area (reuses the K/V stages)
  static constexpr int MERGE = NC * GT * (D + 3) * 4;
  static_assert(NST >= 1, "lanes per row too small for 8 rows per warp");
  static_assert(NSTI % SG == 0, "reduction groups must tile the steps");
  static_assert(STAGES >= R, "a consumer iteration holds R stages");
  static_assert(EPL * LPR == D && NPL * EPP == EPL, "row split");
  static_assert(EPP % 2 == 0, "pieces hold whole fp32 pairs");
  static_assert(MERGE <= 2 * STAGES * PAGE, "merge area");
  static_assert(PAGE % 16 == 0, "bulk copies move multiples of 16 bytes");
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
__device__ __forceinline__ void pv_row_impl(const float* pw_src, const uint8_t* vr, int c,
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
template <typename CT, typename Ly, int GT, int EL2>
__device__ __forceinline__ void pv_row(const float* pw_src, const uint8_t* vr, int c,
                                       float2 (&acc)[GT][EL2]) {
  pv_row_impl<CT, Ly, GT, EL2>(pw_src, vr, c, acc);
}

template <typename QT, typename CT, int D, int GT, int BS>
__global__ void __launch_bounds__(Layout<CT, D, GT, BS>::THREADS)
    paged_decode_kernel(const __grid_constant__ DecodeParams p) {
  using Ly = Layout<CT, D, GT, BS>;
  constexpr int NC = Ly::NC, STAGES = Ly::STAGES, LPR = Ly::LPR, EPP = Ly::EPP;
  constexpr int NPL = Ly::NPL, EPL = Ly::EPL, RPW = Ly::RPW, TPW = Ly::TPW;
  constexpr float kLn2 = 0.69314718055994530942f;
  extern __shared__ __align__(128) uint8_t smem[];

  const int split = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hq = p.num_heads, G = p.group;
  pdl_wait();
  pdl_trigger();

  // ---- attended slots of this sequence and this split's pages
  int n = p.context_lens[s];
  const int cap = p.max_blocks_per_seq * BS;
  int L;
  if (n < 0) {
    L = 0;
    if (threadIdx.x == 0 && split == 0 && g == 0) raise_error(p.err, PA_DEVERR_CONTEXT_LEN);
  } else if (p.window > 0) {
    L = n < p.window ? n : p.window;
  } else if (n > cap) {
    L = cap;
    if (threadIdx.x == 0 && split == 0 && g == 0) raise_error(p.err, PA_DEVERR_CONTEXT_LEN);
  } else {
    L = n;
  }
  const int total_pages = (L + BS - 1) / BS;
  const int pg0 = split * p.pages_per_split;
  const int pg1 = min(total_pages, pg0 + p.pages_per_split);
  const int npg = pg1 - pg0;

  if (npg <= 0) {  // nothing to attend in this split (uniform for the CTA)
    for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
      const int h = i / D, d = i % D;
      const size_t row = (size_t)s * Hq + (size_t)g * G + h;
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

  uint8_t* sK = smem + Ly::OFF_K;
  uint8_t* sV = smem + Ly::OFF_V;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Ly::OFF_BAR);
  uint64_t* empty = full + STAGES;
  volatile int* stage_ok = reinterpret_cast<volatile int*>(smem + Ly::OFF_OK);

  if (threadIdx.x == 0) {
#pragma unroll
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], NC);
    }
    fence_mbar_init();
  }
  __syncthreads();

  // ======================================================== producer warp
  if (warp == NC) {
    const int32_t* bt = p.block_tables + (size_t)s * p.max_blocks_per_seq + pg0;
    const size_t head_off = (size_t)g * Ly::PAGE;
    const size_t blk_stride = (size_t)p.num_kv_heads * Ly::PAGE;
    int tbl = -1;
    int issued = 0;
    bool aborted = false;
    for (int k = 0; k < npg; ++k) {
      if ((k & 31) == 0) {
        const int idx = k + lane;
        tbl = idx < npg ? __ldg(bt + idx) : -1;
      }
      const int bid = __shfl_sync(0xffffffffu, tbl, k & 31);
      const int slot = k % STAGES;
      if (lane == 0) {
        if (k >= STAGES && !mbar_wait_bounded(&empty[slot], ((k / STAGES) - 1) & 1)) {
          raise_error(p.err, PA_DEVERR_TIMEOUT);
          aborted = true;
        }
        if (!aborted) {
          const bool ok = bid >= 0 && bid < p.num_blocks;
          stage_ok[slot] = ok ? 1 : 0;
          if (ok) {
            const size_t off = (size_t)bid * blk_stride + head_off;
            mbar_arrive_expect_tx(&full[slot], 2u * Ly::PAGE);
            bulk_g2s(sK + slot * Ly::PAGE, p.k_cache + off, Ly::PAGE, &full[slot]);
            bulk_g2s(sV + slot * Ly::PAGE, p.v_cache + off, Ly::PAGE, &full[slot]);
          } else {
            raise_error(p.err, PA_DEVERR_BLOCK_ID);
            mbar_arrive(&full[slot]);
          }
          ++issued;
        }
      }
      if (__shfl_sync(0xffffffffu, aborted ? 1 : 0, 0)) break;
    }
    // never leave the CTA with copies in flight: wait for the last fill of
    // every stage (already complete in the normal case)
    if (lane == 0) {
      for (int k = issued > STAGES ? issued - STAGES : 0; k < issued; ++k)
        if (!mbar_wait_bounded(&full[k % STAGES], (k / STAGES) & 1))
          raise_error(p.err, PA_DEVERR_TIMEOUT);
    }
    return;
  }

  // ======================================================== consumer warps
  const int c = lane % LPR;   // piece column of the row
  const int rg = lane / LPR;  // row within a warp step
  float* wscr = reinterpret_cast<float*>(smem + Ly::OFF_SCR) + warp * Ly::SCR;

  constexpr int EP2 = Ly::EP2, EL2 = Ly::EL2;
  float2 qf[GT][EL2];   // q (pre-scaled), as consecutive pairs of this lane's elements
  float2 acc[GT][EL2];  // un-normalised output, same layout
  {
    const QT* q = reinterpret_cast<const QT*>(p.query);
#pragma unroll
    for (int h = 0; h < GT; ++h) {
      const bool live = h < G;
      const QT* qh = q + ((size_t)s * Hq + (size_t)g * G + (live ? h : 0)) * D;
#pragma unroll
      for (int kk = 0; kk < NPL; ++kk) {
#pragma unroll
        for (int j2 = 0; j2 < EP2; ++j2) {
          const int d = (kk * LPR + c) * EPP + 2 * j2;
          qf[h][kk * EP2 + j2] =
              live ? make_float2(Elem<QT>::to_f32(qh[d]) * p.q_scale,
                                 Elem<QT>::to_f32(qh[d + 1]) * p.q_scale)
                   : make_float2(0.f, 0.f);
          acc[h][kk * EP2 + j2] = make_float2(0.f, 0.f);
        }
      }
    }
  }

  // Online softmax with a lazy running max (log2 units). For the reduced
  // values it holds (index kk: head hd[kk]) a lane keeps the running max m of
  // that head, its own share of the running sum l and the largest logit seen.
  // Weights are 2^(s - m); m only moves (and acc/l are rescaled) when a logit
  // exceeds it by more than kLazy, so the weights stay <= 2^kLazy.
  constexpr float kLazy = 8.f;
  constexpr int NFIN = Ly::NFIN, RED = Ly::RED, NG = Ly::NG, NV = Ly::NV;
  constexpr int TPI = Ly::TPI, R = Ly::R;
  const bool writer = (c % RED) == 0;  // one lane per distinct reduced value
  int hd[NFIN];
#pragma unroll
  for (int kk = 0; kk < NFIN; ++kk) hd[kk] = ((c * NV) / LPR + kk) % GT;
  float m_run[NFIN], l_run[NFIN], s_top[NFIN];
#pragma unroll
  for (int kk = 0; kk < NFIN; ++kk) {
    m_run[kk] = -INFINITY;
    l_run[kk] = 0.f;
    s_top[kk] = -INFINITY;
  }

  bool aborted = false;
  for (int k0 = 0; k0 < npg; k0 += R) {
    // this iteration's R pages; token t of the warp's TPI rows is row
    // warp*TPW + t%TPW of page k0 + t/TPW
    const uint8_t* Kp[R];
    const uint8_t* Vp[R];
    int lim[R];  // rows t%TPW < lim[r] of page r hold attended slots
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int k = k0 + r;
      const int slot = (k < npg ? k : k0) % STAGES;
      Kp[r] = sK + slot * Ly::PAGE;
      Vp[r] = sV + slot * Ly::PAGE;
      lim[r] = 0;
      if (k < npg) {
        if (!mbar_wait_bounded(&full[slot], (k / STAGES) & 1)) {
          raise_error(p.err, PA_DEVERR_TIMEOUT);
          aborted = true;
        }
        if (stage_ok[slot] != 0) lim[r] = L - (pg0 + k) * BS - warp * TPW;
      }
    }
    if (__any_sync(0xffffffffu, aborted)) break;

    // ---- 1. logits of this warp's rows for the GT heads (fp32 pair FMAs),
    //         reduced across the row's lanes; invalid rows become -inf
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
          const int st = sg * Ly::SG + stl;
          const int row = warp * TPW + (st % Ly::NST) * RPW + rg;
          const uint8_t* kr = Kp[st / Ly::NST] + row * Ly::ROWB;
#pragma unroll
          for (int kk = 0; kk < NPL; ++kk) {
            float2 kf[EP2];
            load_piece2<CT, Ly::PB>(kr + (kk * LPR + c) * Ly::PB, kf);
#pragma unroll
            for (int h = 0; h < GT; ++h)
#pragma unroll
              for (int j2 = 0; j2 < EP2; ++j2)
                part2[stl * GT + h] = __ffma2_rn(qf[h][kk * EP2 + j2], kf[j2], part2[stl * GT + h]);
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
        sl[sg][kk] = (writer && (t % TPW) < lim_t) ? part[kk] : -INFINITY;
      }
    }

    // ---- 2. lazy max: move m only when a logit clears it by kLazy
    bool raise = false;
#pragma unroll
    for (int kk = 0; kk < NFIN; ++kk) {
      float top = sl[0][kk];
#pragma unroll
      for (int sg = 1; sg < NG; ++sg) top = fmaxf(top, sl[sg][kk]);
      s_top[kk] = fmaxf(s_top[kk], top);
      raise |= top > m_run[kk] + kLazy;
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
        const float m_new = fmaxf(m_run[kk], top);
        alpha[kk] = m_new == -INFINITY ? 1.f : exp2f(m_run[kk] - m_new);
        m_run[kk] = m_new;
        l_run[kk] *= alpha[kk];
      }
      float al[GT];  // every head's factor, from a lane that holds that head
#pragma unroll
      for (int h = 0; h < GT; ++h)
        al[h] = __shfl_sync(0xffffffffu, alpha[h % NFIN], Ly::NV >= LPR ? h / NFIN : h * RED);
#pragma unroll
      for (int h = 0; h < GT; ++h)
#pragma unroll
        for (int e = 0; e < EL2; ++e) acc[h][e] = __fmul2_rn(acc[h][e], make_float2(al[h], al[h]));
    }

    // ---- 3. weights 2^(s - m) to shared memory, then P.V (fp32 pair FMAs)
#pragma unroll
    for (int sg = 0; sg < NG; ++sg)
#pragma unroll
      for (int kk = 0; kk < NFIN; ++kk) {
        const float pw = sl[sg][kk] == -INFINITY ? 0.f : exp2f(sl[sg][kk] - m_run[kk]);
        l_run[kk] += pw;
        if (writer) {
          const int idx = (c * NV) / LPR + kk;
          const int t = (sg * Ly::SG + idx / GT) * RPW + rg;
          wscr[t * GT + idx % GT] = pw;
        }
      }
    __syncwarp();
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (lim[r] >= TPW) {  // every row of this warp in page r is attended
#pragma unroll
        for (int st = 0; st < Ly::NST; ++st) {
          const int tr = st * RPW + rg;
          pv_row<CT, Ly>(wscr + (r * TPW + tr) * GT, Vp[r] + (warp * TPW + tr) * Ly::ROWB, c, acc);
        }
      } else if (lim[r] > 0) {
#pragma unroll
        for (int st = 0; st < Ly::NST; ++st) {
          const int tr = st * RPW + rg;
          if (tr < lim[r])
            pv_row<CT, Ly>(wscr + (r * TPW + tr) * GT, Vp[r] + (warp * TPW + tr) * Ly::ROWB, c,
                           acc);
        }
      }
    }
    __syncwarp();
    if (lane == 0) {
#pragma unroll
      for (int r = 0; r < R; ++r)
        if (k0 + r < npg) mbar_arrive(&empty[(k0 + r) % STAGES]);
    }
  }

  // ---- per-head (m, l, top) of this warp, then merge row groups and warps
  float mh[GT], lh[GT], th[GT];
  {
    float lsum[NFIN], tmax[NFIN];
#pragma unroll
    for (int kk = 0; kk < NFIN; ++kk) {
      lsum[kk] = l_run[kk];
      tmax[kk] = s_top[kk];
#pragma unroll
      for (int off = 1; off < 32; off *= 2)
        if ((off & Ly::HEAD_MASK) == 0) {
          lsum[kk] += __shfl_xor_sync(0xffffffffu, lsum[kk], off);
          tmax[kk] = fmaxf(tmax[kk], __shfl_xor_sync(0xffffffffu, tmax[kk], off));
        }
    }
#pragma unroll
    for (int h = 0; h < GT; ++h) {
      const int src = Ly::NV >= LPR ? h / NFIN : h * RED;
      mh[h] = __shfl_sync(0xffffffffu, m_run[h % NFIN], src);
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
        acc[h][e].x += __shfl_xor_sync(0xffffffffu, acc[h][e].x, off);
        acc[h][e].y += __shfl_xor_sync(0xffffffffu, acc[h][e].y, off);
      }

  named_bar_sync(1, NC * 32);  // every consumer is done with the stages
  float* mm = reinterpret_cast<float*>(smem);   // [NC][GT] running max
  float* ml = mm + NC * GT;                     // [NC][GT] running sum (relative to mm)
  float* mt = ml + NC * GT;                     // [NC][GT] largest logit
  float* ma = mt + NC * GT;                     // [NC][GT][D] accumulators
  if (lane < GT) {
    mm[warp * GT + lane] = aborted ? -INFINITY : mh[lane];
    ml[warp * GT + lane] = aborted ? 0.f : lh[lane];
    mt[warp * GT + lane] = aborted ? -INFINITY : th[lane];
  }
  if (rg == 0) {
#pragma unroll
    for (int h = 0; h < GT; ++h)
#pragma unroll
      for (int kk = 0; kk < NPL; ++kk)
#pragma unroll
        for (int j2 = 0; j2 < EP2; ++j2) {
          const float2 a = aborted ? make_float2(0.f, 0.f) : acc[h][kk * EP2 + j2];
          *reinterpret_cast<float2*>(&ma[(warp * GT + h) * D + (kk * LPR + c) * EPP + 2 * j2]) = a;
        }
  }
  named_bar_sync(1, NC * 32);

  for (int i = threadIdx.x; i < G * D; i += NC * 32) {
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
          o += ma[(w * GT + h) * D + d] * f;
        }
      }
      o = o / lsum * p.v_scale;
    }
    const size_t row = (size_t)s * Hq + (size_t)g * G + h;
    if (p.partials) {
      const size_t pi = row * p.num_splits + split;
      const bool any = M != -INFINITY && lsum > 0.f;
      if (any) p.tmp_out[pi * D + d] = o;
      if (d == 0) {
        // report the split's largest logit and the sum relative to it
        p.max_logits[pi] = any ? T * kLn2 : -INFINITY;
        p.exp_sums[pi] = any ? lsum * exp2f(M - T) : 0.f;
      }
    } else {
      reinterpret_cast<QT*>(p.out)[row * D + d] = Elem<QT>::from_f32(o);
    }
  }
}

// Host-side launcher for one instantiation.
template <typename QT, typename CT, int D, int GT, int BS>
cudaError_t launch_decode(const DecodeParams& prm, int num_seqs, cudaStream_t stream) {
  using Ly = Layout<CT, D, GT, BS>;
  auto kern = paged_decode_kernel<QT, CT, D, GT, BS>;
  static int configured_devices = 0;  // bit per device id < 32
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 32 || !(__atomic_load_n(&configured_devices, __ATOMIC_ACQUIRE) & (1 << dev))) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::SMEM);
    if (e != cudaSuccess) return e;
    if (dev < 32) __atomic_fetch_or(&configured_devices, 1 << dev, __ATOMIC_RELEASE);
  }
  dim3 grid(prm.num_splits, prm.num_kv_heads, num_seqs);
  return launch_pdl(kern, grid, dim3(Ly::THREADS), Ly::SMEM, stream, prm);
}

// Dispatch over (head_dim, group bucket, block size) for one (QT, CT) pair.
template <typename QT, typename CT>
cudaError_t dispatch_decode(const DecodeParams& prm, int num_seqs, int D, int GT, int BS,
                            cudaStream_t stream) {
#define PA_CASE_BS(D_, GT_)                                                               \
  switch (BS) {                                                                           \
    case 16: return launch_decode<QT, CT, D_, GT_, 16>(prm, num_seqs, stream);            \
    case 32: return launch_decode<QT, CT, D_, GT_, 32>(prm, num_seqs, stream);            \
    case 64: return launch_decode<QT, CT, D_, GT_, 64>(prm, num_seqs, stream);            \
    default: return cudaErrorInvalidValue;                                                \
  }
#define PA_CASE_GT(D_)                  \
  switch (GT) {                         \
    case 1: PA_CASE_BS(D_, 1)           \
    case 2: PA_CASE_BS(D_, 2)           \
    case 4: PA_CASE_BS(D_, 4)           \
    case 8: PA_CASE_BS(D_, 8)           \
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
  cudaError_t NAME(const pa::DecodeParams& prm, int num_seqs, int D, int GT, int BS,   \
                   cudaStream_t stream)
PA_DECLARE_DISPATCH(pa_dispatch_decode_f32_f32);
PA_DECLARE_DISPATCH(pa_dispatch_decode_bf16_bf16);
PA_DECLARE_DISPATCH(pa_dispatch_decode_f16_f16);
PA_DECLARE_DISPATCH(pa_dispatch_decode_f32_e4m3);
PA_DECLARE_DISPATCH(pa_dispatch_decode_bf16_e4m3);
PA_DECLARE_DISPATCH(pa_dispatch_decode_f16_e4m3);
