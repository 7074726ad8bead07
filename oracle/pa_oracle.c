/*
 * pa_oracle.c -- CPU oracle for paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow, obviously correct
 * statement of what the paged decode path computes. It is used by the tests,
 * by the smoke check and by the benchmark's CPU-baseline leg; the product
 * path never links, loads or calls it. It shares no code, header, table or
 * constant with the CUDA library: element codes, the FP8 E4M3 encoder and
 * decoder, bf16/f16 widening and the attention itself are all written out
 * here from their definitions.
 *
 * Passages followed (web pages on the subject):
 *  - "PagedAttention in mistral.rs" (engine/docs/PAGED_ATTENTION.md), intro
 *    and "Using the CLI": the K/V cache is a pool of blocks; block size is the
 *    number of tokens per block (default 32).
 *  - same page, "KV Cache Quantization": the cache may be held as FP8 in the
 *    E4M3 format instead of the native dtype ("auto").
 *  - "Optimization plans" (mistral.rs discussion #46): reshape_and_cache
 *    writes each new token's K/V into the cache.
 *  - "Rolling buffer cache" (llama.cpp discussion #3581), opening post: with a
 *    fixed span W, timestep i is stored in slot i mod W and overwrites the
 *    older value there.
 *  - same page, "FlashAttention V2/V3 + PagedAttention" and its feature list
 *    (speculative decoding): a prefill phase runs several query tokens of a
 *    sequence against the paged cache at once; each attends causally.
 *  - "libmir-metal trace/kv.rs", model summary strings: a KV cache of type
 *    "INT8 per token/head" keeps packed INT8 pages with one FP32 scale per
 *    token and head, dequantised inside the paged attention.
 * Readings where the pages are silent (layout [NB][Hkv][bs][D], kv head
 * h / G, FP8 divide-then-round-to-nearest-even with saturation at 448, NaN to
 * 0x7F|sign, attending exactly the last W positions, context_len including the
 * new token, empty context giving 0) are the ones listed in the design notes.
 *
 * Everything is computed in double precision except where the stored format
 * fixes the precision (FP8 quantisation divides in binary32; dequantisation
 * multiplies in binary32), exactly as the method states it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Host threads of the parallel loops below (n > 0 sets it); returns the
 * previous setting, 1 when built without OpenMP. Timing only: the results do
 * not depend on it (every row is computed by one thread in a fixed order). */
int oracle_set_threads(int n)
{
#ifdef _OPENMP
    int prev = omp_get_max_threads();
    if (n > 0)
        omp_set_num_threads(n);
    return prev;
#else
    (void)n;
    return 1;
#endif
}

/* Element codes of this oracle's own interface. */
#define OR_F32 0
#define OR_BF16 1
#define OR_F16 2
#define OR_E4M3 3 /* only as a cache element type */
#define OR_I8 4   /* only as a cache element type: INT8 with per-row scales */

/* ------------------------------------------------------------------ */
/* scalar formats                                                      */
/* ------------------------------------------------------------------ */

/* bfloat16 is the upper half of a binary32: widening appends 16 zero bits. */
static float or_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static float or_f16_to_f32(uint16_t h)
{
    int s = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 31)
        v = m ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)m, -24); /* subnormal: m * 2^-14 * 2^-10 */
    else
        v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
    return (float)(s ? -v : v);
}

/* Load element i of an array of the given element code, widened to float. */
static float or_load(const void* base, int code, size_t i)
{
    switch (code) {
    case OR_F32: return ((const float*)base)[i];
    case OR_BF16: return or_bf16_to_f32(((const uint16_t*)base)[i]);
    case OR_F16: return or_f16_to_f32(((const uint16_t*)base)[i]);
    default: return NAN;
    }
}

static size_t or_elem_bytes(int code)
{
    return code == OR_F32 ? 4 : (code == OR_E4M3 || code == OR_I8) ? 1 : 2;
}

/*
 * FP8 E4M3 (the "F8E4M3" cache type of "KV Cache Quantization"), written from
 * the format: 1 sign bit, 4 exponent bits with bias 7, 3 fraction bits; no
 * infinities; S.1111.111 is NaN. Normal values (1 + m/8) * 2^(e-7) for
 * e = 1..15 (largest 1.75 * 2^8 = 448), subnormals m * 2^-9 for m = 1..7.
 */
float oracle_e4m3_decode(uint8_t b)
{
    int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7)
        return s ? -NAN : NAN; /* S.1111.111: NaN, sign kept */
    v = (e == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return (float)(s ? -v : v);
}

/*
 * Round |y| to the nearest E4M3 value (ties to the even code) with an
 * unbounded exponent, then saturate anything above 448 to 448.
 */
uint8_t oracle_e4m3_encode(float y)
{
    uint32_t u;
    uint8_t sign;
    double a, quantum, n, fl, frac, k, v;
    int e, E, qexp, mant;

    memcpy(&u, &y, 4);
    sign = (u >> 31) ? 0x80 : 0x00;
    if (isnan(y))
        return (uint8_t)(0x7F | sign);
    if (isinf(y))
        return (uint8_t)(0x7E | sign);
    a = fabs((double)y);
    if (a == 0.0)
        return sign;

    /* binade: a in [2^E, 2^(E+1)) */
    frexp(a, &e);
    E = e - 1;
    /* spacing of the E4M3 grid in that binade: 8 steps per binade for normal
       values (E >= -6), fixed 2^-9 below the smallest normal 2^-6 */
    qexp = (E >= -6) ? E - 3 : -9;
    quantum = ldexp(1.0, qexp);
    n = a / quantum; /* exact: division by a power of two */
    fl = floor(n);
    frac = n - fl;
    if (frac > 0.5)
        k = fl + 1.0;
    else if (frac < 0.5)
        k = fl;
    else /* tie: pick the even multiple (even code) */
        k = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    v = k * quantum;
    if (v > 448.0)
        v = 448.0;
    if (v == 0.0)
        return sign;
    if (v < ldexp(1.0, -6)) /* subnormal: v = m * 2^-9 */
        return (uint8_t)(sign | (uint8_t)(v / ldexp(1.0, -9)));
    frexp(v, &e);
    E = e - 1;
    mant = (int)(v / ldexp(1.0, E - 3)) - 8; /* v = (8 + mant) * 2^(E-3) */
    return (uint8_t)(sign | ((E + 7) << 3) | mant);
}

/*
 * Code stored for input x with per-tensor scale: E4M3(x / scale) with a
 * binary32 division. A NaN input keeps its own sign (0x7F | sign of x): the
 * sign of a NaN quotient is not fixed by IEEE 754, so it is not taken from it.
 */
static uint8_t or_quantise(float x, float scale)
{
    uint32_t u;
    if (isnan(x)) {
        memcpy(&u, &x, 4);
        return (uint8_t)(0x7F | ((u >> 31) ? 0x80 : 0x00));
    }
    return oracle_e4m3_encode(x / scale);
}

/* Bulk helpers so the tests can sweep every binary32 bit pattern. */
void oracle_e4m3_encode_array(const float* x, uint8_t* out, int64_t n)
{
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < n; ++i)
        out[i] = oracle_e4m3_encode(x[i]);
}

void oracle_e4m3_decode_array(const uint8_t* b, float* out, int64_t n)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = oracle_e4m3_decode(b[i]);
}

/*
 * INT8 per token/head ("libmir-metal trace/kv.rs": packed INT8 pages, one
 * FP32 scale per token and head). Symmetric quantisation of one row of n
 * values (one token of one kv head, K or V separately), all in binary32:
 *   amax  = max |x_i|
 *   scale = amax / 127
 *   q_i   = round-to-nearest-even(x_i / scale), clamped to [-127, 127]
 * and q_i = 0 for every i when scale is 0 (an all-zero row, or one so small
 * that amax / 127 underflows). The stored value is q_i * scale (one binary32
 * multiply). Inputs are finite; NaN or infinity give codes with no meaning.
 */
void oracle_int8_quantise_row(const float* x, int n, int8_t* codes, float* scale_out)
{
    float amax = 0.0f, scale;
    int i;
    for (i = 0; i < n; ++i)
        amax = fmaxf(amax, fabsf(x[i]));
    scale = amax / 127.0f;
    *scale_out = scale;
    for (i = 0; i < n; ++i) {
        float r;
        if (scale == 0.0f) {
            codes[i] = 0;
            continue;
        }
        r = rintf(x[i] / scale);
        r = fminf(fmaxf(r, -127.0f), 127.0f);
        codes[i] = (int8_t)r;
    }
}

/* ------------------------------------------------------------------ */
/* slot mapping (ring-aware)                                           */
/* ------------------------------------------------------------------ */

/*
 * Slot of token t: its position r in the sequence's slot space (the position
 * itself, or position mod W for a rolling buffer of W slots), then block
 * table entry r / bs, row r % bs. Returns the number of tokens whose sequence
 * index or page index was out of range (their slot is -1).
 */
int64_t oracle_slot_mapping(int64_t* slot_mapping, const int32_t* block_tables,
                            const int32_t* seq_idx, const int32_t* positions,
                            int64_t num_tokens, int num_seqs, int max_blocks_per_seq,
                            int block_size, int window)
{
    int64_t t, bad = 0;
    for (t = 0; t < num_tokens; ++t) {
        int64_t s = seq_idx ? seq_idx[t] : t;
        int64_t pos = positions[t];
        int64_t r, page;
        if (pos < 0) {
            slot_mapping[t] = -1;
            continue;
        }
        r = (window > 0) ? pos % window : pos;
        page = r / block_size;
        if (s < 0 || s >= num_seqs || page >= max_blocks_per_seq) {
            slot_mapping[t] = -1;
            ++bad;
            continue;
        }
        slot_mapping[t] = (int64_t)block_tables[s * (int64_t)max_blocks_per_seq + page] * block_size
                          + r % block_size;
    }
    return bad;
}

/* ------------------------------------------------------------------ */
/* reshape_and_cache                                                   */
/* ------------------------------------------------------------------ */

/*
 * Copy (AUTO) or quantise (E4M3) row [t][h][:] of key/value into
 * cache[slot / bs][h][slot % bs][:]. Negative slots are padding. Returns the
 * number of tokens whose slot was beyond the pool (not written).
 *
 * in_code   : element code of key/value (OR_F32 / OR_BF16 / OR_F16)
 * cache_code: in_code (AUTO) or OR_E4M3
 */
int64_t oracle_reshape_and_cache(const void* key, const void* value, void* k_cache,
                                 void* v_cache, const int64_t* slot_mapping,
                                 int64_t num_tokens, int num_kv_heads, int head_dim,
                                 int block_size, int64_t num_blocks, int in_code,
                                 int cache_code, float k_scale, float v_scale)
{
    int64_t t, bad = 0;
    size_t in_b = or_elem_bytes(in_code);
    for (t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        int64_t blk, off;
        int h, d;
        if (slot < 0)
            continue;
        if (slot >= num_blocks * (int64_t)block_size) {
            ++bad;
            continue;
        }
        blk = slot / block_size;
        off = slot % block_size;
        for (h = 0; h < num_kv_heads; ++h) {
            size_t src = ((size_t)t * num_kv_heads + h) * head_dim;
            size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + off) * head_dim;
            if (cache_code != OR_E4M3) {
                memcpy((char*)k_cache + dst * in_b, (const char*)key + src * in_b, head_dim * in_b);
                memcpy((char*)v_cache + dst * in_b, (const char*)value + src * in_b, head_dim * in_b);
                continue;
            }
            for (d = 0; d < head_dim; ++d) {
                /* binary32 division, correctly rounded (no contraction/fast-math) */
                ((uint8_t*)k_cache)[dst + d] = or_quantise(or_load(key, in_code, src + d), k_scale);
                ((uint8_t*)v_cache)[dst + d] = or_quantise(or_load(value, in_code, src + d), v_scale);
            }
        }
    }
    return bad;
}

/*
 * INT8 write: row [t][h][:] of key (and of value) quantised as one row, codes
 * to cache[slot / bs][h][slot % bs][:], its scale to
 * scales[slot / bs][h][slot % bs]. Negative slots are padding. Returns the
 * number of tokens whose slot was beyond the pool (not written).
 */
int64_t oracle_reshape_and_cache_int8(const void* key, const void* value, int8_t* k_cache,
                                      int8_t* v_cache, float* k_scales, float* v_scales,
                                      const int64_t* slot_mapping, int64_t num_tokens,
                                      int num_kv_heads, int head_dim, int block_size,
                                      int64_t num_blocks, int in_code)
{
    int64_t t, bad = 0;
    float* row = (float*)malloc(sizeof(float) * (size_t)head_dim);
    for (t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        int64_t blk, off;
        int h, d, pass;
        if (slot < 0)
            continue;
        if (slot >= num_blocks * (int64_t)block_size) {
            ++bad;
            continue;
        }
        blk = slot / block_size;
        off = slot % block_size;
        for (h = 0; h < num_kv_heads; ++h) {
            size_t src = ((size_t)t * num_kv_heads + h) * head_dim;
            size_t dst_row = ((size_t)blk * num_kv_heads + h) * block_size + off;
            for (pass = 0; pass < 2; ++pass) {
                const void* in = pass ? value : key;
                for (d = 0; d < head_dim; ++d)
                    row[d] = or_load(in, in_code, src + d);
                oracle_int8_quantise_row(row, head_dim,
                                         (pass ? v_cache : k_cache) + dst_row * head_dim,
                                         (pass ? v_scales : k_scales) + dst_row);
            }
        }
    }
    free(row);
    return bad;
}

/* ------------------------------------------------------------------ */
/* decode: gather through the block table, then dense softmax attention */
/* ------------------------------------------------------------------ */

/* Cache element as the method defines it: native value, E4M3 value times the
   per-tensor scale, or INT8 code times its row's scale (row = i / head_dim);
   each a single binary32 multiply. */
static double or_cache_value(const void* cache, int cache_code, size_t i, float cscale,
                             const float* row_scales, int head_dim)
{
    if (cache_code == OR_I8) {
        float q = (float)((const int8_t*)cache)[i] * row_scales[i / (size_t)head_dim];
        return (double)q;
    }
    if (cache_code == OR_E4M3) {
        float q = oracle_e4m3_decode(((const uint8_t*)cache)[i]) * cscale;
        return (double)q;
    }
    return (double)or_load(cache, cache_code, i);
}

/*
 * Attention of one query row q[D] (fp64) of sequence s, kv head g, over the
 * slots [b0, b1) of its block table (0 <= b0, b1 <= MB * bs):
 *   m = max logit, l = sum exp(logit - m), o = sum exp(logit - m) V / l,
 *   logit_j = scale * q . K_j.
 * Empty range: m = -inf, l = 0, o = 0. Returns -1 if a needed block id is
 * outside [0, num_blocks), else 0. k_scales / v_scales ([NB][Hkv][bs] fp32)
 * are read only for an INT8 cache (cache_code OR_I8).
 */
static int or_attend(double* o, double* m_out, double* l_out, const double* q, int s, int g,
                     const void* k_cache, const void* v_cache, const int32_t* block_tables,
                     int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                     int max_blocks_per_seq, double scale, int cache_code, float k_scale,
                     float v_scale, const float* k_scales, const float* v_scales, int64_t b0,
                     int64_t b1)
{
    int64_t j, cnt;
    int d, rc = 0;
    double *K, *V, *logit, m, l;

    for (d = 0; d < head_dim; ++d)
        o[d] = 0.0;
    *m_out = -INFINITY;
    *l_out = 0.0;
    if (b1 <= b0)
        return 0;
    cnt = b1 - b0;

    /* 1. gather the attended rows into contiguous K[cnt][D], V[cnt][D] */
    K = (double*)malloc(sizeof(double) * (size_t)cnt * head_dim);
    V = (double*)malloc(sizeof(double) * (size_t)cnt * head_dim);
    logit = (double*)malloc(sizeof(double) * (size_t)cnt);
    for (j = 0; j < cnt; ++j) {
        int64_t slot = b0 + j;
        int64_t blk = block_tables[(int64_t)s * max_blocks_per_seq + slot / block_size];
        int64_t row = slot % block_size;
        size_t base = (((size_t)blk * num_kv_heads + g) * block_size + row) * head_dim;
        if (blk < 0 || blk >= num_blocks) {
            rc = -1;
            for (d = 0; d < head_dim; ++d)
                K[j * head_dim + d] = V[j * head_dim + d] = NAN;
            continue;
        }
        for (d = 0; d < head_dim; ++d) {
            K[j * head_dim + d] =
                or_cache_value(k_cache, cache_code, base + d, k_scale, k_scales, head_dim);
            V[j * head_dim + d] =
                or_cache_value(v_cache, cache_code, base + d, v_scale, v_scales, head_dim);
        }
    }

    /* 2. logits = scale * q . K_j */
    m = -INFINITY;
    for (j = 0; j < cnt; ++j) {
        double acc = 0.0;
        for (d = 0; d < head_dim; ++d)
            acc += q[d] * K[j * head_dim + d];
        logit[j] = scale * acc;
        if (logit[j] > m)
            m = logit[j];
    }

    /* 3. softmax weights relative to the max, and the weighted sum of V */
    l = 0.0;
    for (j = 0; j < cnt; ++j) {
        double p = exp(logit[j] - m);
        l += p;
        for (d = 0; d < head_dim; ++d)
            o[d] += p * V[j * head_dim + d];
    }
    for (d = 0; d < head_dim; ++d)
        o[d] /= l;
    *m_out = m;
    *l_out = l;
    free(K);
    free(V);
    free(logit);
    return rc;
}

/*
 * Partial attention of query head h of sequence s over its slots
 * [tok_begin, tok_end) intersected with [0, L_s) (see or_attend for the
 * outputs and the return value).
 */
int oracle_decode_partial(double* o, double* m_out, double* l_out, const void* query,
                          const void* k_cache, const void* v_cache,
                          const int32_t* block_tables, const int32_t* context_lens,
                          int s, int h, int num_heads, int num_kv_heads, int head_dim,
                          int block_size, int64_t num_blocks, int max_blocks_per_seq,
                          double scale, int window, int q_code, int cache_code,
                          float k_scale, float v_scale, const float* k_scales,
                          const float* v_scales, int64_t tok_begin, int64_t tok_end)
{
    int G = num_heads / num_kv_heads;
    int g = h / G; /* contiguous groups of query heads share one kv head */
    int64_t n = context_lens[s];
    int64_t L = (window > 0 && n > window) ? window : n;
    int64_t b0, b1;
    int d, rc;
    double* q;

    if (n < 0)
        L = 0;
    b0 = tok_begin < 0 ? 0 : tok_begin;
    b1 = tok_end < L ? tok_end : L;
    q = (double*)malloc(sizeof(double) * (size_t)head_dim);
    for (d = 0; d < head_dim; ++d)
        q[d] = (double)or_load(query, q_code, ((size_t)s * num_heads + h) * head_dim + d);
    rc = or_attend(o, m_out, l_out, q, s, g, k_cache, v_cache, block_tables, num_kv_heads,
                   head_dim, block_size, num_blocks, max_blocks_per_seq, scale, cache_code,
                   k_scale, v_scale, k_scales, v_scales, b0, b1);
    free(q);
    return rc;
}

/*
 * Full decode for the (s, h) pairs listed in rows[] (row = s * num_heads + h),
 * or for every pair when rows == NULL (nrows ignored). out is
 * [S][Hq][D] double; only the listed rows are written. Returns the number of
 * rows that met an out-of-range block id.
 */
int64_t oracle_decode_rows(double* out, const void* query, const void* k_cache,
                           const void* v_cache, const int32_t* block_tables,
                           const int32_t* context_lens, int num_seqs, int num_heads,
                           int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                           int max_blocks_per_seq, double scale, int window, int q_code,
                           int cache_code, float k_scale, float v_scale,
                           const float* k_scales, const float* v_scales,
                           const int64_t* rows, int64_t nrows)
{
    int64_t i, bad = 0;
    int64_t total = rows ? nrows : (int64_t)num_seqs * num_heads;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
    for (i = 0; i < total; ++i) {
        int64_t r = rows ? rows[i] : i;
        int s = (int)(r / num_heads), h = (int)(r % num_heads);
        double m, l;
        if (oracle_decode_partial(out + (size_t)r * head_dim, &m, &l, query, k_cache, v_cache,
                                  block_tables, context_lens, s, h, num_heads, num_kv_heads,
                                  head_dim, block_size, num_blocks, max_blocks_per_seq, scale,
                                  window, q_code, cache_code, k_scale, v_scale, k_scales,
                                  v_scales, 0, (int64_t)1 << 62) != 0)
            ++bad;
    }
    return bad;
}

/*
 * Multi-query (prefill) attention over the paged cache: query token t belongs
 * to sequence q_seq[t] at absolute position q_pos[t] and attends causally to
 * the positions 0 .. q_pos[t] of that sequence, read through its block table
 * (slot = position; no window). Its own K/V and those of the tokens before it
 * are expected in the cache already. query / out are [T][Hq][D] (out fp64).
 * A token with q_pos < 0 is padding (its rows of out are 0). Returns the
 * number of (token, head) rows that met an out-of-range sequence, position or
 * block id (their rows are NaN).
 */
int64_t oracle_prefill_rows(double* out, const void* query, const int32_t* q_seq,
                            const int32_t* q_pos, int64_t num_tokens, const void* k_cache,
                            const void* v_cache, const int32_t* block_tables, int num_seqs,
                            int num_heads, int num_kv_heads, int head_dim, int block_size,
                            int64_t num_blocks, int max_blocks_per_seq, double scale,
                            int q_code, int cache_code, float k_scale, float v_scale,
                            const float* k_scales, const float* v_scales)
{
    int64_t i, bad = 0;
    int G = num_heads / num_kv_heads;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
    for (i = 0; i < num_tokens * num_heads; ++i) {
        int64_t t = i / num_heads;
        int h = (int)(i % num_heads), d;
        int s = q_seq[t];
        int64_t p = q_pos[t];
        double* o = out + (size_t)i * head_dim;
        double m, l, q[512];
        if (p < 0) {
            for (d = 0; d < head_dim; ++d)
                o[d] = 0.0;
            continue;
        }
        if (s < 0 || s >= num_seqs || p >= (int64_t)max_blocks_per_seq * block_size ||
            head_dim > 512) {
            for (d = 0; d < head_dim; ++d)
                o[d] = NAN;
            ++bad;
            continue;
        }
        for (d = 0; d < head_dim; ++d)
            q[d] = (double)or_load(query, q_code, (size_t)i * head_dim + d);
        if (or_attend(o, &m, &l, q, s, h / G, k_cache, v_cache, block_tables, num_kv_heads,
                      head_dim, block_size, num_blocks, max_blocks_per_seq, scale, cache_code,
                      k_scale, v_scale, k_scales, v_scales, 0, p + 1) != 0)
            ++bad;
    }
    return bad;
}

/* ------------------------------------------------------------------ */
/* log-sum-exp combination of split partials                           */
/* ------------------------------------------------------------------ */

/*
 * out[r][:] = sum_i w_i o_i / sum_i w_i with w_i = l_i exp(m_i - M),
 * M = max m_i over non-empty splits (l_i > 0); all empty -> 0.
 * tmp_out [R][NS][D], max_logits/exp_sums [R][NS], R = rows.
 */
void oracle_reduce(double* out, const double* tmp_out, const double* max_logits,
                   const double* exp_sums, int64_t rows, int head_dim, int num_splits)
{
    int64_t r;
    for (r = 0; r < rows; ++r) {
        double M = -INFINITY, wsum = 0.0;
        int i, d;
        for (d = 0; d < head_dim; ++d)
            out[r * head_dim + d] = 0.0;
        for (i = 0; i < num_splits; ++i)
            if (exp_sums[r * num_splits + i] > 0.0 && max_logits[r * num_splits + i] > M)
                M = max_logits[r * num_splits + i];
        if (M == -INFINITY)
            continue;
        for (i = 0; i < num_splits; ++i) {
            double l = exp_sums[r * num_splits + i], w;
            if (!(l > 0.0))
                continue;
            w = l * exp(max_logits[r * num_splits + i] - M);
            wsum += w;
            for (d = 0; d < head_dim; ++d)
                out[r * head_dim + d] += w * tmp_out[((size_t)r * num_splits + i) * head_dim + d];
        }
        for (d = 0; d < head_dim; ++d)
            out[r * head_dim + d] /= wsum;
    }
}
