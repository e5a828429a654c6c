/*
 * qsa_indexer.h -- C ABI of libqsa: the weighted paged MQA indexer of a
 * DeepSeek-V3.2-style sparse-attention decode step and its per-row top-k.
 *
 * The operations are the two named by "[XPU] Enable multiple key kernels for
 * sparse attention" (vLLM PR 37888 report, "Implementation" and "Key source
 * snippets"): fp8_paged_mqa_logits and top_k_per_row_decode.  That page
 * prints their signatures only; what they compute is taken in the plainest
 * way the signatures support and is stated below.  Conventions (device
 * pointers, fail-closed validation, no allocation, asynchronous launch on
 * the caller's stream, device-side data errors reported in *error_word) are
 * those of qsa.h.
 */
#ifndef QSA_INDEXER_H
#define QSA_INDEXER_H

#include "qsa.h"

#ifdef __cplusplus
extern "C" {
#endif

#define QSA_IDX_HEAD_DIM   128   /* indexer query / key width (E4M3 values) */
#define QSA_IDX_MAX_TOPK   2048  /* largest topk_tokens */
#define QSA_DERR_IDX_BLOCK 16u   /* a cache block id negative / >= num_blocks,
                                    or past the block table's columns: its
                                    tokens get -inf */

/*
 * qsa_paged_mqa_logits -- for row r = b*next_n + j (query token j of
 * request b) and column t:
 *
 *   L_r = min(context_lens[b] - next_n + j + 1, max_model_len)   (>= 0)
 *   logits[r, t] = scale_t * sum_{h<H} weights[r, h] * ReLU(q[r, h, :] . k_t)
 *                  for t < L_r, and -inf for L_r <= t < max_model_len,
 *
 * where k_t (128 E4M3 values) and scale_t (fp32) are token t of request b:
 * cache block block_tables[b, t / block_size], slot t % block_size.  A cache
 * block is block_size * 132 bytes: the block's 128-byte value rows (token
 * order), then its block_size fp32 scales.  The dot products are formed by
 * FP8 tensor-core MMAs with fp32 accumulation; the head sum is fp32.
 *
 * Arguments
 *   q             E4M3 [num_rows, num_heads, 128], contiguous (q_dtype QSA_DT_F8E4M3)
 *   kv_cache      bytes [num_blocks, block_size * 132] (kv_dtype QSA_DT_F8E4M3),
 *                 16-byte aligned; block_size in {8, 16, 32, 64, 128}
 *   weights       fp32 [num_rows, num_heads], contiguous
 *   context_lens  int32 [batch]; num_rows = batch * next_n
 *   block_tables  int32 [batch, bt_cols], row stride bt_stride0, column stride 1
 *   num_heads     16, 32, 64 or 128; next_n in [1, 4]; num_heads * next_n <= 256
 *   logits        fp32 [num_rows, max_model_len], row stride logits_stride0
 *                 (>= max_model_len), written in full; may not overlap an input
 *   error_word    device uint32 or NULL
 */
QSA_API qsa_status qsa_paged_mqa_logits(
    const void* q, qsa_dtype q_dtype, int64_t num_rows, int64_t num_heads,
    const void* kv_cache, qsa_dtype kv_dtype, int64_t num_blocks, int64_t block_size,
    const void* weights, qsa_dtype weights_dtype,
    const void* context_lens, qsa_dtype ctx_dtype, int64_t batch,
    const void* block_tables, qsa_dtype bt_dtype, int64_t bt_cols, int64_t bt_stride0,
    int64_t next_n,
    void* logits, qsa_dtype logits_dtype, int64_t max_model_len, int64_t logits_stride0,
    uint32_t* error_word, qsa_stream_t stream);

/*
 * qsa_top_k_per_row_decode -- for row r = b*next_n + j:
 *   L_r = min(max(seq_lens[b] - next_n + j + 1, 0), num_cols);
 *   indices[r, 0..k) = the k = min(topk_tokens, L_r) columns t < L_r with the
 *   largest logits[r, t], largest first, equal logits by ascending t;
 *   indices[r, k..topk_tokens) = -1.
 * Exact (a radix select over the logits' ordered bit patterns); NaN logits
 * are outside the contract.
 *
 * Arguments
 *   logits        fp32, element (r, t) at logits + r*stride0 + t*stride1
 *                 (elements; stride1 >= 1), num_rows x num_cols
 *   seq_lens      int32 [batch]; num_rows = batch * next_n; next_n >= 1
 *   topk_tokens   1 .. 2048
 *   indices       int32 [num_rows, topk_tokens], row stride idx_stride0; may
 *                 not overlap an input
 */
QSA_API qsa_status qsa_top_k_per_row_decode(
    const void* logits, qsa_dtype logits_dtype, int64_t num_rows, int64_t num_cols,
    int64_t stride0, int64_t stride1, int64_t next_n,
    const void* seq_lens, qsa_dtype seq_lens_dtype, int64_t batch,
    int64_t topk_tokens, void* indices, qsa_dtype idx_dtype, int64_t idx_stride0,
    qsa_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* QSA_INDEXER_H */
