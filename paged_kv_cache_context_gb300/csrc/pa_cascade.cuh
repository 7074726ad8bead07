// pa_cascade.cuh -- shared-prefix (cascade) attention: the kernel launcher's
// parameters, shared by pa_cascade.cu (the kernel) and pa_api.cu (the entry
// point that also runs the suffix decode and the combine).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

// Attention of every sequence's query heads to the blocks of a prefix that
// all of a batch's block tables share ("PagedAttention in mistral.rs":
// prefix caching; the shared blocks are read once per kv head for the whole
// batch instead of once per sequence). For kv head g the rows are the S * G
// query heads (s, g * G + j) that share it, so the prefix part is a dense
// contraction Q [S*G, D] x K^T [D, T] and P [S*G, T] x V [T, D].
//
// The prefix tokens [0, prefix_tokens) are cut into num_prefix_splits ranges
// of tokens_per_split tokens; split i writes the partial of every row over
// its range into slot slot0 + i of the pa_reduce layout:
//   tmp_out [S][Hq][num_slots][D], max_logits / exp_sums [S][Hq][num_slots]
// (normalised output, largest logit in natural-log units, sum of
// exp(logit - max); a range with no token gives -inf / 0 and leaves tmp_out).
struct PrefixParams {
  // the K and V caches as 2-D tensors of [NB * Hkv * bs rows][D elements],
  // boxes of 64 elements x bs rows with the 128-byte swizzle
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  float* tmp_out;
  float* max_logits;
  float* exp_sums;
  const void* query;            // [S][Hq][D] (a 16-bit cache holds the same type)
  const uint8_t* k_cache;       // [NB][Hkv][bs][D]
  const uint8_t* v_cache;
  const float* k_scales;        // INT8 caches: row scales [NB][Hkv][bs] (else unused)
  const float* v_scales;
  const int32_t* block_tables;  // [S][MB]; the first prefix_pages entries of every row agree
  const int32_t* context_lens;  // [S]; every context covers the prefix
  unsigned* err;                // device error word
  int num_seqs, num_heads, num_kv_heads, group, head_dim, block_size, num_blocks;
  int max_blocks_per_seq, prefix_pages, prefix_tokens;
  int num_slots, slot0, num_prefix_splits, tokens_per_split;
  float scale_log2;  // scale * log2(e) (* k_scale for an FP8 cache)
  float v_scale;     // FP8 caches: multiplies the output (else unused)
};

// Rows of one tensor-core query tile (the M of one MMA), rows of query heads
// one shared-prefix CTA takes, and tokens per staged K/V tile.
constexpr int kPrefixTcRows = 128;
constexpr int kPrefixCtaRows = 128;
constexpr int kPrefixTile = 64;

// dtype: the query's, 1 = bf16, 2 = f16 (pa_dtype values); kind: the
// cache's, 0 = the query's type, 1 = INT8 codes with row scales, 2 = FP8 E4M3
// codes. Returns cudaErrorInvalidValue for other types, kinds or head
// dimensions (64 and 128 are built).
cudaError_t launch_prefix_attention(const PrefixParams& p, int dtype, int kind,
                                    cudaStream_t stream);

// Causal multi-query (prefill) attention over the paged cache ("PagedAttention
// in mistral.rs": a prefill phase next to the paged decode, and speculative
// decoding, both attend several query tokens of a sequence at once). Sequence
// s owns query tokens [cu_q[s], cu_q[s+1]); they are the last q_len_s
// positions of its context of n_s = context_lens[s] tokens, whose K/V are in
// the cache already: token i sits at position n_s - q_len_s + i and attends
// to positions 0 .. that position. For kv head g the rows of a sequence are
// its q_len_s * G (token, head-in-group) pairs, so Q K^T and P V are dense
// contractions over the sequence's pages.
struct PrefillParams {
  // the K and V caches as 2-D tensors (as in PrefixParams)
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  void* out;                    // [T][Hq][D], same element type as the query
  const void* query;            // [T][Hq][D]
  const uint8_t* k_cache;       // [NB][Hkv][bs][D]
  const uint8_t* v_cache;
  const int32_t* block_tables;  // [S][MB]
  const int32_t* cu_q;          // [S + 1]: query token offsets
  const int32_t* context_lens;  // [S]: context length including the chunk
  const float* k_scales;        // INT8 caches: row scales [NB][Hkv][bs] (else unused)
  const float* v_scales;
  unsigned* err;
  int num_seqs, num_heads, num_kv_heads, group, head_dim, block_size, num_blocks;
  int num_tokens, max_blocks_per_seq, max_q_len;
  float scale_log2;  // scale * log2(e) (* k_scale for an FP8 cache)
  float v_scale;     // FP8 caches: multiplies the output (else unused)
};

// dtype and kind as launch_prefix_attention's.
cudaError_t launch_prefill_attention(const PrefillParams& p, int dtype, int kind,
                                     cudaStream_t stream);

// Copies whole blocks (all kv heads, K and V) src -> dst for each pair of
// block_pairs [n][2]; block ids outside [0, num_blocks) set PA_DEVERR_BLOCK_ID
// and are skipped. block_bytes (a multiple of 16) = Hkv * bs * D * element size.
cudaError_t launch_copy_blocks(uint8_t* k_cache, uint8_t* v_cache, const int32_t* block_pairs,
                               int num_pairs, int num_blocks, size_t block_bytes, unsigned* err,
                               cudaStream_t stream);

}  // namespace pa
