/*
 * qsa_oracle.h -- plain, slow, single-threaded CPU oracle for the QSA sparse
 * decode path.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg are its only callers; the product path never
 * links, loads or calls it, and it shares no code, header, table or helper
 * with the CUDA library.
 *
 * What it restates (citations name the page and its section):
 *   - "vLLM: integrate FP16 packed QSA extension" (intel/llm-scaler PR 651),
 *     Summary and "Exact contracts" (Selection, Attention): shapes, dtypes,
 *     strides, the fixed token_topk=2048 / compress_ratio=4 contract, the
 *     [R,2051] output padded with -1, descending-score / ascending-index order.
 *   - qsa_cache.py (vLLM fork, Qwen4Exp QSA side caches):
 *     _build_qsa_metadata_kernel (visible-block rule),
 *     compressed_qsa_slot_mapping (a compressed key exists for group g once
 *     token 4g+3 exists), _logical_to_physical_qsa_slots (paging; a negative
 *     physical block is padding).
 *
 * Precision.  The selection score decides integers (which blocks are chosen),
 * so the oracle evaluates it in the kernel's arithmetic: IEEE binary32 with
 * round-to-nearest-even in one fixed summation order (qsa_oracle_score).
 * Attention is evaluated in binary64.
 *
 * Parity pins: every function here is pinned by tests under tests/ against
 * brute force, closed forms and invariants (see the test files' docstrings).
 */
#ifndef QSA_ORACLE_H
#define QSA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* error bits the oracle reports (a row keeps going; bad blocks are skipped) */
#define QSA_ORACLE_ERR_REQUEST  1u  /* token_to_request out of [0, num_reqs) */
#define QSA_ORACLE_ERR_CMP_PAGE 2u  /* compressed page id missing/out of range */
#define QSA_ORACLE_ERR_KV_PAGE  4u  /* K/V page id missing/out of range */

/* fp16 bits -> binary64 (exact). */
double qsa_oracle_half_to_double(uint16_t h);

/* OCP FP8 E4M3 ("fn": no infinities; S.1111.111 is NaN) bits -> binary64
 * (exact). */
double qsa_oracle_e4m3_to_double(uint8_t v);

/* compressed-key element types */
#define QSA_ORACLE_KEY_F16   0
#define QSA_ORACLE_KEY_E4M3  1

/* Canonical binary32 selection score of one compressed key against the four
 * indexer heads: sum over h of ReLU(q_h . k).  q: [4][128] fp16 bits,
 * k: [128] fp16 bits.  The summation order is fixed (see the .c file). */
float qsa_oracle_score(const uint16_t* q, const uint16_t* k);

/* Visible compressed blocks and the inclusive tail end for one row. */
int64_t qsa_oracle_visible_blocks(int64_t seq_len, int64_t pos);
int64_t qsa_oracle_tail_end(int64_t seq_len, int64_t pos);

/*
 * Selection for R rows.
 *   q_sel         [R][4][128] fp16 bits
 *   cmp_pages     num_cmp_pages pointers; page p -> [128 keys][128] fp16 bits
 *                 (a NULL entry is a page the caller did not provide)
 *   cmp_pt        int32, row-major with stride pt_stride0, max_pages columns
 *   t2r           [R] int32, seq_lens [num_reqs] int32, qpos [R] int64
 *   out           [R][out_width] int32 (out_width >= 2051; all written)
 * Returns the OR of the error bits seen.
 */
uint32_t qsa_oracle_select(int64_t R, const uint16_t* q_sel,
                           const uint16_t* const* cmp_pages, int64_t num_cmp_pages,
                           const int32_t* cmp_pt, int64_t num_reqs, int64_t max_pages,
                           int64_t pt_stride0, const int32_t* t2r,
                           const int32_t* seq_lens, const int64_t* qpos,
                           int32_t* out, int64_t out_width);

/* Selection with the compressed keys stored as key_kind elements (page p ->
 * [128 keys][128] elements of that type); QSA_ORACLE_KEY_F16 is
 * qsa_oracle_select. */
uint32_t qsa_oracle_select_keys(int64_t R, const uint16_t* q_sel, int key_kind,
                                const void* const* cmp_pages, int64_t num_cmp_pages,
                                const int32_t* cmp_pt, int64_t num_reqs, int64_t max_pages,
                                int64_t pt_stride0, const int32_t* t2r,
                                const int32_t* seq_lens, const int64_t* qpos,
                                int32_t* out, int64_t out_width);

/* Canonical score of an E4M3 key [128] (same order as qsa_oracle_score). */
float qsa_oracle_score_e4m3(const uint16_t* q, const uint8_t* k);

/* Same, but also returns the binary32 score of every selected block in the
 * order emitted (scores_out [R][512], unused entries -1.0f) -- used by tests
 * that check ordering properties. */
uint32_t qsa_oracle_select_scored(int64_t R, const uint16_t* q_sel,
                                  const uint16_t* const* cmp_pages, int64_t num_cmp_pages,
                                  const int32_t* cmp_pt, int64_t num_reqs, int64_t max_pages,
                                  int64_t pt_stride0, const int32_t* t2r,
                                  const int32_t* seq_lens, const int64_t* qpos,
                                  int32_t* out, int64_t out_width, float* scores_out);

/*
 * Sparse attention for R rows, in binary64.
 *   q        [R][3][256] fp16 bits
 *   kv_pages num_kv_pages pointers; page p -> [512 tokens][512] fp16 bits
 *            (token t: K = halves 0..255, V = halves 256..511); NULL = absent
 *   kv_pt    int32, stride pt_stride0, max_kv_pages columns
 *   t2r      [R] int32
 *   idx      [R][width] int32 logical token indices, -1 = hole
 *   scale    logit scale (1/16 for the contract)
 *   out      [R][3][256] binary64
 * Returns the OR of the error bits seen.
 */
uint32_t qsa_oracle_attention(int64_t R, const uint16_t* q,
                              const uint16_t* const* kv_pages, int64_t num_kv_pages,
                              const int32_t* kv_pt, int64_t num_reqs, int64_t max_kv_pages,
                              int64_t pt_stride0, const int32_t* t2r,
                              const int32_t* idx, int64_t width, double scale,
                              double* out);

#ifdef __cplusplus
}
#endif
#endif
