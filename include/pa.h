/*
 * pa.h -- C ABI of the GB300 (sm_103a) PagedAttention decode library.
 *
 * The library computes softmax attention of ONE new query token per sequence
 * over a key/value cache that is stored in fixed-size blocks ("pages") of
 * block_size tokens and addressed through a per-sequence block table.
 *
 * Sources of the operations (web pages this library restates):
 *  - "PagedAttention in mistral.rs" (engine/docs/PAGED_ATTENTION.md), opening
 *    section and "Using the CLI": the cache is a pool of blocks sized by a GPU
 *    memory budget; block size = tokens per block, default 32.
 *  - same page, "KV Cache Quantization": the cache may be stored as FP8 E4M3
 *    instead of the model's native dtype ("auto"), about half the bytes of FP16.
 *  - "Optimization plans" (mistral.rs discussion #46), the update that traces
 *    junk output to reshape_and_cache: the write that scatters each new token's
 *    K/V into its cache slot.
 *  - "Rolling buffer cache" (llama.cpp discussion #3581), the opening post
 *    quoting Mistral 7B: a fixed-size cache of W slots where the K/V of
 *    timestep i live in slot i mod W and overwrite older entries.
 *
 * Conventions for every call below
 *  - All tensor arguments are DEVICE pointers to dense, row-major (C order)
 *    arrays owned by the caller. The library never allocates device memory and
 *    never frees caller memory.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). Kernels are
 *    enqueued asynchronously on it; a call returns as soon as they are queued.
 *  - Argument errors are detected on the host BEFORE anything is enqueued and
 *    are returned as a negative pa_status; nothing is written in that case.
 *  - Data-dependent errors that only the GPU can see (a slot or block id out of
 *    range, a context length beyond the table) never fault: the offending
 *    element is skipped, a bit is set in a per-device error word, and
 *    pa_get_device_error() reports it later.
 *  - Notation: T = num_tokens, S = num_seqs, Hq = num_heads,
 *    Hkv = num_kv_heads, G = Hq / Hkv, D = head_dim, bs = block_size,
 *    NB = num_blocks, MB = max_blocks_per_seq, n_s = context_lens[s]
 *    (INCLUDING the new token), W = window (0 = no window),
 *    L_s = n_s if W == 0 else min(n_s, W) (tokens attended by sequence s).
 *  - Cache layout (both K and V): [NB][Hkv][bs][D]. The page of one
 *    (block, kv head) is bs*D contiguous elements ("head-major pages").
 *    Element type: the input dtype for PA_KV_AUTO, one byte (E4M3) for
 *    PA_KV_FP8_E4M3, one signed byte for PA_KV_INT8 (whose calls take, beside
 *    each cache, fp32 row scales [NB][Hkv][bs]: one per token and kv head).
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so this header needs no CUDA headers. */
typedef struct CUstream_st* pa_stream_t;

typedef enum {
    PA_OK = 0,
    PA_ERR_NULL = -1,        /* a required pointer is NULL                          */
    PA_ERR_DTYPE = -2,       /* unsupported element type or combination             */
    PA_ERR_SHAPE = -3,       /* a size is negative/zero where it may not be, or
                                num_heads % num_kv_heads != 0, or G > 8            */
    PA_ERR_HEAD_DIM = -4,    /* head_dim not in {64, 96, 128}                       */
    PA_ERR_BLOCK_SIZE = -5,  /* block_size not supported                            */
    PA_ERR_WINDOW = -6,      /* window < 0, window % block_size != 0, or
                                window / block_size > max_blocks_per_seq           */
    PA_ERR_WORKSPACE = -7,   /* workspace smaller than the requested split plan     */
    PA_ERR_CUDA = -8,        /* a CUDA runtime call failed (bad stream, launch)     */
    PA_ERR_DEVICE = -9,      /* pa_get_device_error(): a kernel flagged bad data    */
    PA_ERR_ALIGN = -10,      /* a pointer is not 16-byte aligned                    */
    PA_ERR_SCALE = -11       /* an FP8 scale is not finite and > 0                  */
} pa_status;

/* Element type of query / key / value / output (and of an AUTO cache). */
typedef enum { PA_F32 = 0, PA_BF16 = 1, PA_F16 = 2 } pa_dtype;

/* Cache storage type ("auto" and "f8e4m3" of "KV Cache Quantization"). */
typedef enum { PA_KV_AUTO = 0, PA_KV_FP8_E4M3 = 1, PA_KV_INT8 = 2 } pa_kv_dtype;

/* Bits of the per-device error word (see pa_get_device_error). */
enum {
    PA_DEVERR_SLOT = 1u,        /* slot_mapping entry >= NB*bs: that token was not written   */
    PA_DEVERR_BLOCK_ID = 2u,    /* a block-table entry needed by a sequence is outside
                                   [0, NB): that page was treated as holding no tokens     */
    PA_DEVERR_CONTEXT_LEN = 4u, /* context_lens[s] < 0 or L_s > MB*bs: clamped to the range */
    PA_DEVERR_TIMEOUT = 8u,     /* a bounded wait for an asynchronous copy gave up          */
    PA_DEVERR_SEQ = 16u         /* pa_slot_mapping: seq index out of range or page index
                                   >= MB: slot set to -1                                   */
};

/*
 * pa_slot_mapping -- cache slot of each token to be written (ring-aware).
 *
 * Source: "Rolling buffer cache" (opening post): timestep i goes to slot
 * i mod W of a fixed cache of W entries, overwriting older values; and the
 * paged store of "PagedAttention in mistral.rs" (block = block_size tokens).
 *
 *   r = (window > 0) ? positions[t] mod window : positions[t]
 *   s = seq_idx ? seq_idx[t] : t
 *   slot_mapping[t] = block_tables[s][r / bs] * bs + r % bs
 *
 * slot_mapping : out, int64 [T].  positions : int32 [T] (absolute position of
 * the token in its sequence, < 0 = padding -> slot -1).  seq_idx : int32 [T]
 * or NULL (token t belongs to sequence t).  block_tables : int32 [S][MB].
 * A seq index outside [0, S) or r/bs >= MB gives slot -1 and sets
 * PA_DEVERR_SEQ.  T == 0 is a no-op.
 */
pa_status pa_slot_mapping(int64_t* slot_mapping, const int32_t* block_tables,
                          const int32_t* seq_idx, const int32_t* positions,
                          int num_tokens, int num_seqs, int max_blocks_per_seq,
                          int block_size, int window, pa_stream_t stream);

/*
 * pa_reshape_and_cache -- scatter the K/V of new tokens into their cache slots.
 *
 * Source: "Optimization plans" (reshape_and_cache, the write whose bug gave
 * junk output) and "KV Cache Quantization" (F8E4M3 cache).
 *
 * key, value   : in, [T][Hkv][D] of in_dtype.
 * k_cache,
 * v_cache      : in/out, [NB][Hkv][bs][D] of in_dtype (AUTO) or uint8 (FP8).
 * slot_mapping : in, int64 [T]; slot < 0 = padding (skipped); block
 *                slot / bs, row slot % bs. Duplicate slots within one call
 *                leave that slot's value unspecified (one of the writers).
 * AUTO  : the element bits are copied unchanged.
 * FP8   : code = E4M3(x / k_scale) (IEEE fp32 divide; bf16/f16 inputs widened
 *         exactly), round to nearest even, finite overflow and +-inf saturate
 *         to +-448 (code 0x7E / 0xFE), a NaN input -> 0x7F | (sign of the
 *         input), -0 -> 0x80.
 *         Same for V with v_scale. Scales must be finite and > 0.
 * Only the rows named by slot_mapping are written; every other byte of the
 * cache is left untouched. Pointers must be 16-byte aligned.
 */
pa_status pa_reshape_and_cache(const void* key, const void* value,
                               void* k_cache, void* v_cache,
                               const int64_t* slot_mapping,
                               int num_tokens, int num_kv_heads, int head_dim,
                               int block_size, int num_blocks,
                               pa_dtype in_dtype, pa_kv_dtype kv_dtype,
                               float k_scale, float v_scale, pa_stream_t stream);

/*
 * pa_decode -- paged decode attention, one query token per sequence.
 *
 * Source: "PagedAttention in mistral.rs" (blocked cache read through block
 * tables; FP8 cache); "Rolling buffer cache" (window W: attend to the last W
 * positions, held in ring slots 0 .. L_s-1).
 *
 * For every sequence s and query head h (kv head g = h / G):
 *   slot j in [0, L_s) lives at block block_tables[s][j / bs], row j % bs
 *   logit_j = scale * sum_d q[s][h][d] * K_j[d]          (K_j dequantised)
 *   out[s][h][:] = sum_j softmax(logit)_j * V_j[:]       (0 when L_s == 0)
 * With FP8, K_j[d] = E4M3value(byte) * k_scale and V_j likewise with v_scale.
 * Accumulation is fp32. Where the products run on the tensor cores the
 * operands are rounded as the MMAs take them: a 16-bit cache with G >= 4
 * (head_dim 64 or 128) rounds the softmax weights to the cache type; an FP8
 * or INT8 cache read with 16-bit queries carries q in f16 (exact for a bf16
 * query inside f16's range, |q| < 65520) and rounds the weights to f16.
 * Bytes of the cache outside the L_s attended slots
 * (tail rows of the last block, unused blocks) are never used, whatever they
 * hold (NaN included).
 *
 * out          : out, [S][Hq][D] of q_dtype.     query : in, [S][Hq][D] q_dtype.
 * k_cache,
 * v_cache      : in, [NB][Hkv][bs][D] (q_dtype for AUTO, uint8 for FP8).
 * block_tables : in, int32 [S][MB].  context_lens : in, int32 [S].
 * window       : 0 = none; else W > 0, W % bs == 0, W / bs <= MB (ring of
 *                W / bs blocks per sequence in block_tables[s][0 .. W/bs-1]).
 * workspace    : device scratch of workspace_bytes (may be NULL / 0). With
 *                at least pa_decode_workspace_size() bytes the call runs the
 *                balanced path (pa_decode_workspace_clear, then one launch of
 *                pa_decode_balanced): one persistent CTA per resident slot,
 *                each streaming an equal share of all sequences' pages;
 *                otherwise one CTA per (sequence, kv head) does that whole
 *                context. Contents on entry do not matter; on exit undefined.
 * Supported: D in {64, 96, 128}; bs in {16, 32, 64}; G = Hq/Hkv in 1..8;
 * q_dtype F32/BF16/F16; AUTO caches hold q_dtype. Pointers 16-byte aligned.
 * Calls whose pages are staged by tensor copies (16-bit queries with a
 * 16-bit cache at G >= 4, or with an 8-bit cache at head_dim 128) need
 * NB * Hkv * bs <= 2^31 - 1 cache rows (else PA_ERR_SHAPE).
 * kv_dtype PA_KV_INT8 is refused with PA_ERR_DTYPE here (its row scales go
 * through pa_decode_int8).
 */
pa_status pa_decode(void* out, const void* query,
                    const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, const int32_t* context_lens,
                    int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                    int block_size, int num_blocks, int max_blocks_per_seq,
                    float scale, int window, pa_dtype q_dtype, pa_kv_dtype kv_dtype,
                    float k_scale, float v_scale,
                    void* workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_reshape_and_cache_int8 -- scatter the K/V of new tokens into an INT8
 * cache with one fp32 scale per token and kv head.
 *
 * Source: "libmir-metal trace/kv.rs" (model summary strings: packed INT8 pages
 * with per-token/head FP32 scales, dequantised inside the paged attention).
 * Each row x = key[t][h][:] (and value[t][h][:]) is quantised on its own, in
 * binary32 (bf16/f16 inputs widened exactly):
 *   scale = max_d |x[d]| / 127 (IEEE divide)
 *   code[d] = round-to-nearest-even(x[d] / scale) clamped to [-127, 127]
 *   (every code 0 when scale == 0)
 * and stored as k_cache[blk][h][off][:] = code, k_scales[blk][h][off] = scale
 * (blk = slot / bs, off = slot % bs). Inputs are expected finite; a NaN or an
 * infinity gives codes with no meaning but is never a fault.
 *
 * key, value   : in, [T][Hkv][D] of in_dtype (F32, BF16 or F16).
 * k_cache,
 * v_cache      : in/out, int8 [NB][Hkv][bs][D].
 * k_scales,
 * v_scales     : in/out, fp32 [NB][Hkv][bs].
 * slot_mapping : in, int64 [T]; < 0 = padding (skipped); a slot >= NB*bs is
 *                skipped and sets PA_DEVERR_SLOT.
 * Supported: D a multiple of 8 up to 256 (else PA_ERR_HEAD_DIM); bs 1..1024
 * (else PA_ERR_BLOCK_SIZE). Pointers 16-byte aligned (PA_ERR_ALIGN); NULL ->
 * PA_ERR_NULL; T == 0 is a no-op.
 */
pa_status pa_reshape_and_cache_int8(const void* key, const void* value,
                                    int8_t* k_cache, int8_t* v_cache,
                                    float* k_scales, float* v_scales,
                                    const int64_t* slot_mapping, int num_tokens,
                                    int num_kv_heads, int head_dim, int block_size,
                                    int num_blocks, pa_dtype in_dtype, pa_stream_t stream);

/*
 * pa_decode_int8 -- pa_decode over an INT8 cache with per-row scales.
 *
 * Source: "libmir-metal trace/kv.rs" (INT8 per-token/head pages, fused
 * dequantisation in the paged attention) on top of the decode of
 * "PagedAttention in mistral.rs". Same computation, arguments, workspace and
 * error behaviour as pa_decode, with
 *   K_j[d] = k_cache[blk][g][row][d] * k_scales[blk][g][row]
 * and V_j likewise (one binary32 multiply each; the kernel applies the K scale
 * to the dot product and the V scale to the softmax weight, which is the same
 * value up to fp32 rounding). k_scales / v_scales : in, fp32 [NB][Hkv][bs].
 * Supported: q_dtype BF16 or F16 (else PA_ERR_DTYPE); D, bs, G and window as
 * pa_decode. Pointers 16-byte aligned.
 */
pa_status pa_decode_int8(void* out, const void* query,
                         const int8_t* k_cache, const int8_t* v_cache,
                         const float* k_scales, const float* v_scales,
                         const int32_t* block_tables, const int32_t* context_lens,
                         int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                         int block_size, int num_blocks, int max_blocks_per_seq,
                         float scale, int window, pa_dtype q_dtype,
                         void* workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_prefill -- causal multi-query attention over the paged cache.
 *
 * Source: "PagedAttention in mistral.rs" (a prefill phase runs beside the
 * paged decode, "FlashAttention V2/V3 + PagedAttention"; speculative
 * decoding in the feature list): several query tokens of a sequence attend
 * to its paged K/V at once. Sequence s owns query tokens [cu_q[s], cu_q[s+1])
 * (q_len_s of them, q_len_s <= max_q_len); they are the LAST q_len_s
 * positions of its context of n_s = context_lens[s] tokens, whose K and V
 * are already in the cache (written by pa_reshape_and_cache). Token i of the
 * chunk is at position p = n_s - q_len_s + i and
 *   out[cu_q[s] + i][h][:] = softmax_j<=p(scale * q . K_j) V_j,
 * kv head h / G, fp32 accumulation, P rounded to the input type before P.V
 * (tensor cores), output rounded to q_dtype. No window.
 *
 * out, query   : [T][Hq][D] of q_dtype (BF16 or F16, else PA_ERR_DTYPE).
 * k_cache,
 * v_cache      : [NB][Hkv][bs][D] of q_dtype.
 * block_tables : int32 [S][MB].  cu_q : int32 [S + 1].  context_lens :
 *                int32 [S].
 * Supported: D in {64, 128} (PA_ERR_HEAD_DIM); bs in {16, 32, 64}
 * (PA_ERR_BLOCK_SIZE); G in 1..8; 1 <= max_q_len <= T and
 * NB * Hkv * bs <= 2^31 - 1 cache rows (pages are staged by tensor copies)
 * (PA_ERR_SHAPE).
 * Device-side checks: offsets that do not fit [0, T] or a q_len above
 * max_q_len set PA_DEVERR_SEQ and that sequence is not written; n_s < q_len_s
 * or n_s > MB * bs sets PA_DEVERR_CONTEXT_LEN and its rows are zero; a block
 * id outside [0, NB) sets PA_DEVERR_BLOCK_ID and reads as zeros. Pointers
 * 16-byte aligned. T == 0 or S == 0 is a no-op.
 */
pa_status pa_prefill(void* out, const void* query,
                     const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, const int32_t* cu_q,
                     const int32_t* context_lens, int num_tokens, int num_seqs,
                     int num_heads, int num_kv_heads, int head_dim, int block_size,
                     int num_blocks, int max_blocks_per_seq, int max_q_len, float scale,
                     pa_dtype q_dtype, pa_stream_t stream);

/*
 * pa_prefill_int8 -- pa_prefill over an INT8 cache with per-row scales.
 *
 * Source: "libmir-metal trace/kv.rs" (INT8 per-token/head pages, dequantised
 * inside the paged attention) with the prefill of "PagedAttention in
 * mistral.rs". Same computation, arguments and errors as pa_prefill, with
 *   K_j[d] = k_cache[blk][g][row][d] * k_scales[blk][g][row]
 * and V_j likewise (the caches and scales written by
 * pa_reshape_and_cache_int8). k_cache, v_cache: int8 [NB][Hkv][bs][D];
 * k_scales, v_scales: fp32 [NB][Hkv][bs]. On the tensor cores the codes are
 * widened exactly to f16, q is carried in f16 (exact for a bf16 query inside
 * f16's range), the K row scale multiplies the logit and the V row scale the
 * softmax weight before it is rounded to f16; fp32 accumulation. Pages are
 * moved by 1-D bulk copies (no limit on the cache's rows). NULL scales ->
 * PA_ERR_NULL; scales not 16-byte aligned -> PA_ERR_ALIGN.
 */
pa_status pa_prefill_int8(void* out, const void* query,
                          const int8_t* k_cache, const int8_t* v_cache,
                          const float* k_scales, const float* v_scales,
                          const int32_t* block_tables, const int32_t* cu_q,
                          const int32_t* context_lens, int num_tokens, int num_seqs,
                          int num_heads, int num_kv_heads, int head_dim, int block_size,
                          int num_blocks, int max_blocks_per_seq, int max_q_len, float scale,
                          pa_dtype q_dtype, pa_stream_t stream);

/*
 * pa_prefill_fp8 -- pa_prefill over an FP8 E4M3 cache with per-tensor scales.
 *
 * Source: "PagedAttention in mistral.rs", section "KV Cache Quantization"
 * (an FP8 E4M3 paged cache, dequantised in the attention), with the same
 * page's prefill. Same computation, arguments and errors as pa_prefill, with
 *   K_j[d] = e4m3(k_cache[blk][g][row][d]) * k_scale
 * and V_j likewise with v_scale (the caches written by pa_reshape_and_cache
 * with PA_KV_FP8_E4M3). k_cache, v_cache: E4M3 bytes [NB][Hkv][bs][D]. On the
 * tensor cores the codes are widened exactly to f16 and q is carried in f16
 * (exact for a bf16 query inside f16's range); k_scale multiplies the logit
 * scale and v_scale the output; fp32 accumulation. Pages are moved by 1-D
 * bulk copies (no limit on the cache's rows). k_scale or v_scale not finite
 * and positive -> PA_ERR_SCALE.
 */
pa_status pa_prefill_fp8(void* out, const void* query,
                         const uint8_t* k_cache, const uint8_t* v_cache,
                         const int32_t* block_tables, const int32_t* cu_q,
                         const int32_t* context_lens, int num_tokens, int num_seqs,
                         int num_heads, int num_kv_heads, int head_dim, int block_size,
                         int num_blocks, int max_blocks_per_seq, int max_q_len, float scale,
                         float k_scale, float v_scale, pa_dtype q_dtype, pa_stream_t stream);

/*
 * pa_decode_plan -- a split plan for pa_decode_partials at these sizes.
 * Writes the number of context splits per (sequence, kv head) and the pages
 * (blocks) each split covers; split i covers slots
 * [i*pages_per_split*bs, (i+1)*pages_per_split*bs). Sized so the splits of a
 * batch fill a 152-SM GPU several times over. Host-only; never touches the GPU.
 */
pa_status pa_decode_plan(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                         int block_size, int max_blocks_per_seq, int window,
                         int* num_splits, int* pages_per_split);

/*
 * Bytes of workspace for pa_decode's balanced path (and for
 * pa_decode_balanced). It depends only on the query-head group size and
 * head_dim, not on the batch: one arrival counter per persistent CTA, then
 * the partial results of at most two pieces per persistent CTA (about 3.8 MB
 * for G = 4, D = 128). 0 for invalid head counts.
 */
size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads,
                                int head_dim, int block_size,
                                int max_blocks_per_seq, int window);

/*
 * pa_decode_workspace_clear / pa_decode_balanced -- pa_decode's balanced path
 * as its two stream operations, exposed so a caller can time the decode
 * kernel alone or clear the workspace once for several decodes.
 *
 * pa_decode_workspace_clear: enqueues a zero fill of the workspace's arrival
 * counters (its first 3840 bytes). Errors: PA_ERR_NULL, PA_ERR_WORKSPACE
 * (fewer bytes), PA_ERR_ALIGN, PA_ERR_CUDA.
 *
 * pa_decode_balanced: one launch. The pages of every (sequence, kv head)
 * context, taken in (sequence, kv head, page) order, are cut into C equal
 * contiguous ranges, C = the kernel's resident capacity on this device
 * (written to *num_ctas); persistent CTA c streams range c. A context lying
 * wholly inside one range is written to `out` by that CTA. A context cut by
 * range boundaries leaves per-CTA partials (max logit, sum, normalised
 * output) in the workspace; each CTA then adds the pages of its partial to the
 * context's arrival counter, and the CTA whose addition completes the context
 * combines the partials by log-sum-exp weights into `out` and sets the
 * counter back to zero. Sequences with nothing to attend get zero rows.
 * Precondition: the arrival counters are zero when the kernel starts, as
 * pa_decode_workspace_clear leaves them and as every launch that raised no
 * device error leaves them. Arguments and errors otherwise as pa_decode
 * (workspace required: PA_ERR_NULL when missing, PA_ERR_WORKSPACE when smaller
 * than pa_decode_workspace_size()).
 */
pa_status pa_decode_workspace_clear(void* workspace, size_t workspace_bytes, pa_stream_t stream);
pa_status pa_decode_balanced(void* out, const void* query,
                             const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, const int32_t* context_lens,
                             int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                             int block_size, int num_blocks, int max_blocks_per_seq,
                             float scale, int window, pa_dtype q_dtype, pa_kv_dtype kv_dtype,
                             float k_scale, float v_scale,
                             void* workspace, size_t workspace_bytes, int* num_ctas,
                             pa_stream_t stream);

/*
 * pa_decode_cascade -- decode of a batch whose block tables all start with
 * the same prefix blocks ("PagedAttention in mistral.rs", opening section:
 * prefix caching keeps a prefix's KV state in the paged cache and reuses
 * it). Same result as pa_decode with window 0, computed in three launches:
 *   1. the shared prefix (pages 0 .. prefix_pages - 1 of row 0 of
 *      block_tables) for all S * G query heads of each kv head at once, on
 *      the tensor cores in 128-row tiles, cut into up to (prefix tokens /
 *      64) token ranges, into partial slots 1 .. ;
 *   2. each sequence's own pages after the prefix (pages prefix_pages ..),
 *      one CTA per (sequence, kv head), into slot 0; this launch starts
 *      beside the first on the SMs it leaves free and waits for it at its
 *      end;
 *   3. pa_reduce of the slots into `out`.
 * The prefix K/V is read once per kv head for the whole batch instead of
 * once per sequence.
 * Preconditions (checked on the device, error bits as pa_decode): the first
 * prefix_pages entries of every row of block_tables are the same blocks
 * (else PA_DEVERR_BLOCK_ID), and every context_lens[s] >= prefix_pages * bs
 * (else PA_DEVERR_CONTEXT_LEN). Supported: AUTO caches of q_dtype BF16 or F16
 * (else PA_ERR_DTYPE; 8-bit caches: pa_decode_cascade_fp8 / _int8 below),
 * D in {64, 128} (else PA_ERR_HEAD_DIM),
 * 1 <= prefix_pages <= MB and NB * Hkv * bs <= 2^31 - 1 cache rows (else
 * PA_ERR_SHAPE). workspace: at least
 * pa_decode_cascade_workspace_size() bytes (PA_ERR_NULL / PA_ERR_WORKSPACE),
 * 16-byte aligned; contents on entry do not matter. Other arguments and
 * errors as pa_decode. Accuracy: the prefix's softmax weights are rounded to
 * the input type before the P x V product (fp32 accumulation), so the result
 * agrees with pa_decode to within the bf16 / f16 output tolerance, not bit for
 * bit.
 */
size_t pa_decode_cascade_workspace_size(int num_seqs, int num_heads, int num_kv_heads,
                                        int head_dim, int block_size, int prefix_pages);
pa_status pa_decode_cascade(void* out, const void* query,
                            const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, const int32_t* context_lens,
                            int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                            int block_size, int num_blocks, int max_blocks_per_seq,
                            float scale, pa_dtype q_dtype, int prefix_pages,
                            void* workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_decode_cascade_fp8 / pa_decode_cascade_int8 -- pa_decode_cascade over
 * an FP8 E4M3 cache with per-tensor scales (k_scale, v_scale; as pa_decode
 * with PA_KV_FP8_E4M3) or over an INT8 cache with per-row scales (k_scales,
 * v_scales fp32 [NB][Hkv][bs]; as pa_decode_int8). Same launches, result,
 * preconditions, workspace and errors as pa_decode_cascade; the shared
 * prefix's 8-bit pages come by 1-D bulk copies (no limit on the cache's rows)
 * and are widened exactly to f16 in shared memory for the tensor cores, q is
 * carried in f16 (exact for a bf16 query inside f16's range); FP8: k_scale
 * multiplies the logit scale and v_scale the output; INT8: the K row scale
 * multiplies the logit and the V row scale the weight before it is rounded
 * to f16. The sequences' own pages go through the decode of that cache kind.
 * k_scale or v_scale not finite and positive -> PA_ERR_SCALE; NULL row scales
 * -> PA_ERR_NULL, not 16-byte aligned -> PA_ERR_ALIGN.
 */
pa_status pa_decode_cascade_fp8(void* out, const void* query,
                                const uint8_t* k_cache, const uint8_t* v_cache,
                                const int32_t* block_tables, const int32_t* context_lens,
                                int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                int block_size, int num_blocks, int max_blocks_per_seq,
                                float scale, float k_scale, float v_scale, pa_dtype q_dtype,
                                int prefix_pages, void* workspace, size_t workspace_bytes,
                                pa_stream_t stream);
pa_status pa_decode_cascade_int8(void* out, const void* query,
                                 const int8_t* k_cache, const int8_t* v_cache,
                                 const float* k_scales, const float* v_scales,
                                 const int32_t* block_tables, const int32_t* context_lens,
                                 int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                 int block_size, int num_blocks, int max_blocks_per_seq,
                                 float scale, pa_dtype q_dtype, int prefix_pages,
                                 void* workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_copy_blocks -- copy whole cache blocks, for copy-on-write of shared
 * blocks ("libmir-metal trace/kv.rs": fragmented copy-on-write block maps).
 * For each pair i, block block_pairs[2i] of both caches (all kv heads, K and
 * V) is copied over block block_pairs[2i + 1]. block_pairs: device int32
 * [num_pairs][2]. elem_bytes: 1 (FP8), 2 (bf16 / f16) or 4 (fp32); the block's
 * bytes Hkv * bs * D * elem_bytes must be a multiple of 16 (else
 * PA_ERR_HEAD_DIM). A pair naming a block outside [0, num_blocks) is skipped
 * and sets PA_DEVERR_BLOCK_ID. Pairs must not overlap (a destination that is
 * another pair's source gives an unspecified result).
 */
pa_status pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* block_pairs,
                         int num_pairs, int num_kv_heads, int head_dim, int block_size,
                         int num_blocks, int elem_bytes, pa_stream_t stream);

/*
 * pa_decode_partials -- the split phase of pa_decode with an explicit plan.
 *
 * For split i of (s, h) (slots [i*P*bs, (i+1)*P*bs) intersected with
 * [0, L_s), P = pages_per_split), writes
 *   max_logits[s][h][i] = m_i = max logit (natural-log units, includes scale)
 *   exp_sums[s][h][i]   = l_i = sum_j exp(logit_j - m_i)
 *   tmp_out[s][h][i][:] = sum_j exp(logit_j - m_i) V_j / l_i
 * A split holding no slot writes m_i = -inf, l_i = 0 and leaves tmp_out[..][i]
 * untouched. tmp_out fp32 [S][Hq][NS][D]; max_logits, exp_sums fp32 [S][Hq][NS].
 * Requires num_splits * pages_per_split >= the ring (W / bs) or MB blocks.
 * Other arguments as pa_decode.
 */
pa_status pa_decode_partials(float* tmp_out, float* max_logits, float* exp_sums,
                             const void* query, const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, const int32_t* context_lens,
                             int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                             int block_size, int num_blocks, int max_blocks_per_seq,
                             float scale, int window, pa_dtype q_dtype, pa_kv_dtype kv_dtype,
                             float k_scale, float v_scale,
                             int num_splits, int pages_per_split, pa_stream_t stream);

/*
 * pa_reduce -- log-sum-exp combination of split partials.
 *
 * For each (s, h): M = max over splits with l_i > 0 of m_i,
 *   w_i = l_i * exp(m_i - M),  out[s][h][:] = sum_i w_i tmp_out[s][h][i][:] / sum_i w_i,
 * rounded to out_dtype (round to nearest even). Splits with l_i == 0 are
 * skipped entirely (their tmp_out rows are not read); if all are empty the
 * output row is 0. Layouts as pa_decode_partials; out [S][Hq][D] of out_dtype.
 * Partials of disjoint context segments produced by separate calls may be
 * combined this way as long as they share one layout.
 */
pa_status pa_reduce(void* out, const float* tmp_out, const float* max_logits,
                    const float* exp_sums, int num_seqs, int num_heads, int head_dim,
                    int num_splits, pa_dtype out_dtype, pa_stream_t stream);

/*
 * pa_decode_static_scratch -- pa_decode for callers that cannot allocate.
 *
 * The pages have no counterpart of this call; it exists for callers that have
 * no way to hand pa_decode a workspace: code running inside a host program
 * that owns every device allocation and offers no allocator, or code that must
 * never call cudaMalloc (it can synchronise the device and take unbounded
 * time). It computes exactly what pa_decode computes, with the same kernels,
 * but keeps the partial results in an array the library itself holds in
 * device memory: PA_STATIC_SCRATCH_BYTES (8 MiB) on every GPU where the
 * library's device code has been loaded, kept until the process exits. It
 * allocates nothing.
 *
 *  - Limit: when these sizes need more partial storage than
 *    PA_STATIC_SCRATCH_BYTES (pa_decode_workspace_size() larger than it), the
 *    call returns PA_ERR_WORKSPACE at once and enqueues nothing. Every head
 *    dimension and group size pa_decode supports fits. This size check comes
 *    before the argument checks of pa_decode; every other argument rule and
 *    error of pa_decode applies unchanged.
 *  - Set-up: each call looks up the array's address on the current device
 *    (cudaGetSymbolAddress); `stream` must belong to that device. The first
 *    call on a device may be the first use of the library's device code
 *    there, in which case the CUDA runtime loads that code and reserves the
 *    array then (a device allocation and an implicit synchronisation inside
 *    the runtime, not by this library): make the first call on each device
 *    during set-up, before any stream capture begins.
 *  - Sharing: all calls on a device share the one array, which keeps whatever
 *    the last call left in it. Nothing in it needs to start at zero (each call
 *    clears the counters it relies on). Calls
 *    whose kernels may overlap on the GPU (different streams, or different
 *    host threads, without ordering between them) race on it and must be
 *    serialised by the caller.
 */
#define PA_STATIC_SCRATCH_BYTES (8u << 20)
pa_status pa_decode_static_scratch(void* out, const void* query,
                                   const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, const int32_t* context_lens,
                                   int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                   int block_size, int num_blocks, int max_blocks_per_seq,
                                   float scale, int window, pa_dtype q_dtype,
                                   pa_kv_dtype kv_dtype, float k_scale, float v_scale,
                                   pa_stream_t stream);

/*
 * pa_block_budget -- how many cache blocks a KV memory budget buys
 * ("PagedAttention in mistral.rs", "Using the CLI" and the Rust API
 * example: the pool is sized by a GPU memory amount in MB, by a fraction of
 * the GPU's memory, or by a context size in tokens; the block size is the
 * number of tokens per block). Host only; never touches the GPU.
 *
 * One block holds block_size tokens of K and V for every kv head of every
 * layer:  block_bytes = num_layers * 2 * num_kv_heads * block_size * row_bytes,
 *         row_bytes = head_dim * element size (4 for F32, 2 for BF16/F16, 1
 *                     for an FP8 E4M3 or INT8 cache), plus 4 for the fp32
 *                     row scale of an INT8 cache.
 *   PA_BUDGET_MB:       amount = MB (2^20 bytes) for the cache;
 *                       blocks = floor(amount * 2^20 / block_bytes).
 *   PA_BUDGET_FRACTION: amount in (0, 1] of available_bytes (the caller's
 *                       figure, e.g. free device memory);
 *                       blocks = floor(amount * available_bytes / block_bytes).
 *   PA_BUDGET_CONTEXT:  amount = tokens of context to hold;
 *                       blocks = ceil(amount / block_size).
 * Returns the number of blocks (>= 0), or a negative pa_status: PA_ERR_SHAPE
 * for a non-positive layer / head / block count or an amount out of range,
 * PA_ERR_DTYPE for unknown types, PA_ERR_HEAD_DIM for head_dim <= 0.
 */
typedef enum {
    PA_BUDGET_MB = 0,
    PA_BUDGET_FRACTION = 1,
    PA_BUDGET_CONTEXT = 2
} pa_budget_kind;
int64_t pa_block_budget(pa_budget_kind kind, double amount, size_t available_bytes,
                        int num_layers, int num_kv_heads, int head_dim, int block_size,
                        pa_dtype dtype, pa_kv_dtype kv_dtype);

/*
 * pa_get_device_error -- synchronise `stream`, then read and clear the error
 * word of the current device. *error_bits (may be NULL) receives the
 * PA_DEVERR_* bits. Returns PA_OK when no bit was set, PA_ERR_DEVICE when
 * some were, PA_ERR_CUDA when the synchronisation itself failed.
 */
pa_status pa_get_device_error(pa_stream_t stream, uint32_t* error_bits);

/*
 * pa_test_set_unarmed_page -- test hook for the bounded waits (no page of the
 * pages describes it). With page >= 0, every decode launched afterwards by
 * this process (pa_decode, pa_decode_balanced, pa_decode_partials and the
 * calls built on them) stops its producer, in every CTA, before it arms the
 * stage of the CTA's page number `page` (counted from the CTA's first page):
 * no copy is issued for that stage or after it. The consumer warps' wait for
 * that stage then gives up after its limit (200 ms), sets
 * PA_DEVERR_TIMEOUT and the CTA ends in order, having waited for every copy
 * it did issue; the outputs of such a launch are unspecified. A negative page
 * (the initial state) switches the hook off. Not thread-safe with respect to
 * launches in flight on other host threads; for tests only.
 */
void pa_test_set_unarmed_page(int page);

/* Static English text for a pa_status value (never NULL). */
const char* pa_status_string(int status);

/* Library ABI version, (major << 16) | minor. */
int pa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* PA_H */
