/*
 * qsa_metadata.h -- C ABI of libqsa: the per-forward metadata of one QSA side
 * cache, the step that runs before selection and produces its
 * token_to_request and query_positions.
 *
 * Operation restated from qsa_cache.py (vLLM fork, Qwen4Exp QSA side caches):
 * _build_qsa_metadata_kernel (and its torch twin _build_qsa_metadata_torch),
 * _logical_positions, circular_qsa_slot_mapping and
 * compressed_qsa_slot_mapping.  Conventions (device pointers, fail-closed
 * validation, no allocation, asynchronous launch) are those of qsa.h.
 */
#ifndef QSA_METADATA_H
#define QSA_METADATA_H

#include "qsa.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Slot value of a token that writes nothing (vLLM's PAD_SLOT_ID). */
#define QSA_PAD_SLOT (-1)

/*
 * qsa_build_metadata -- for every scheduled token t < num_tokens, with
 * mapped = (t < num_mapped_tokens):
 *
 *   token_to_req[t]      the last request i < num_reqs whose query starts at
 *                        or before t (query_start_loc[i] <= t); 0 if unmapped
 *   logical_positions[t] seq_lens[req] - query_len[req] + (t - query_start_loc[req]),
 *                        query_len[i] = query_start_loc[i+1] - query_start_loc[i];
 *                        -1 if unmapped
 *   visible_blocks[t]    max(0, min((pos+1) // cr, L // cr)), L = seq_lens[req]
 *                        (0 if unmapped); cr = compress_ratio
 *   slot_mapping[t]      one of three rules, by mode:
 *     circular_buffer_size = C > 0 (the compressor's raw-key ring; one block
 *       per request, block table column 0): the query's last C tokens write
 *       block*C + pos % C, where block = block_table[req, 0]; every other
 *       token, a negative block or a table without columns gives -1
 *     else compress_ratio != 1 (the compressed-key cache, storage_block_size
 *       = S keys per block): only a token that closes a compression group
 *       ((pos+1) % cr == 0) writes, at group g = pos // cr:
 *       block_table[req, g // S] * S + g % S; -1 when g // S is past the
 *       table's columns, the block is negative, or common_slot_mapping[t] < 0
 *     else: common_slot_mapping[t] (copied)
 *
 * Work list (work_metadata != NULL; the pre-indexer's per-request items):
 * request i gets n_i = max(1, L_i // cr - (L_i - query_len_i) // cr) items
 * when query_len_i > 0 (one per compression group closed inside its query
 * chunk, at least one), else none; items are numbered request by request,
 * and work_metadata[w] = {request, item index within the request} for
 * w < sum n_i, {-1, -1} for the rest of the max_num_work entries.
 *
 * Arguments
 *   query_start_loc     int32 [num_reqs + 1] (dtype tag qsl_dtype), non-decreasing
 *                       from 0 (device data; not checked)
 *   seq_lens            int32 [num_reqs]; seq_lens[i] >= query_len[i] expected
 *   common_slot_mapping int64 [num_tokens]; required unless circular_buffer_size
 *                       > 0 (then ignored, may be NULL)
 *   block_table         int32 [bt_rows, bt_cols], element strides bt_stride0,
 *                       bt_stride1 (>= 1); bt_rows >= num_reqs; bt_cols may be
 *                       0 (NULL allowed then)
 *   num_reqs            >= 1
 *   num_mapped_tokens   the host's copy of query_start_loc[num_reqs] (0 <=
 *                       num_mapped_tokens < 2^31); tokens at or past it are
 *                       padding
 *   num_tokens          tokens to write (0 <= num_tokens < 2^31)
 *   storage_block_size  > 0, compress_ratio > 0, circular_buffer_size >= 0
 *                       (each < 2^31)
 *   token_to_req        int32 [num_tokens]      (outputs: device memory, written
 *   logical_positions   int64 [num_tokens]       in full, may not overlap each
 *   visible_blocks      int32 [num_tokens]       other or any input; NULL
 *   slot_mapping        int64 [num_tokens]       allowed when num_tokens == 0)
 *   work_metadata       int32 [max_num_work][2] or NULL; max_num_work >= 0
 *                       (< 2^31)
 *
 * Returns QSA_OK, or a validation status with nothing launched.  Every
 * device access is bounded by the host-checked sizes (requests are searched
 * inside [0, num_reqs), table columns inside [0, bt_cols)), so malformed
 * device data gives wrong values, never an out-of-range access.
 */
QSA_API qsa_status qsa_build_metadata(
    const void* query_start_loc, qsa_dtype qsl_dtype,
    const void* seq_lens, qsa_dtype seq_lens_dtype,
    const void* common_slot_mapping, qsa_dtype common_dtype,
    const void* block_table, qsa_dtype bt_dtype, int64_t bt_rows, int64_t bt_cols,
    int64_t bt_stride0, int64_t bt_stride1,
    int64_t num_reqs, int64_t num_mapped_tokens, int64_t num_tokens,
    int64_t storage_block_size, int64_t compress_ratio, int64_t circular_buffer_size,
    int32_t* token_to_req, int64_t* logical_positions, int32_t* visible_blocks,
    int64_t* slot_mapping, int32_t* work_metadata, int64_t max_num_work,
    qsa_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* QSA_METADATA_H */
