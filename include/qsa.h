/*
 * qsa.h -- C ABI of libqsa, the GB300 (sm_103a) QSA sparse decode path.
 *
 * Two operations, each one or more CUDA kernels launched asynchronously on
 * the caller's stream:
 *
 *   qsa_select_paged_tokens   "vLLM: integrate FP16 packed QSA extension",
 *                             Summary (fused selection bullet) and
 *                             "Exact contracts" / Selection.
 *   qsa_sparse_attention      same page, Summary (exact-packed attention
 *                             bullet) and "Exact contracts" / Attention.
 *   qsa_select_attend         both in one call and one workspace: the two
 *                             operations' kernels chained on the stream by
 *                             programmatic dependent launch.
 *
 * The visible-block rule used by selection comes from qsa_cache.py
 * (_build_qsa_metadata_kernel: visible = max(0, min((pos+1)//4, seq_len//4))).
 *
 * Conventions for every entry point
 *   - Every tensor pointer is DEVICE memory owned by the caller.  Inputs are
 *     never written; outputs are written in full.
 *   - The call validates all host-visible arguments first (dtype tags, shapes,
 *     strides, alignment, contract constants, workspace size, aliasing).  On
 *     any mismatch it returns a nonzero qsa_status and launches nothing
 *     ("fail closed").
 *   - Nothing is allocated, nothing synchronises with the host, nothing is
 *     read back.  Scratch memory comes from the caller's workspace, whose size
 *     is given by the matching *_workspace_bytes query; its contents on entry
 *     do not matter and are clobbered.
 *   - Values only the device can see (page ids, request ids, indices) are
 *     checked on the device: an out-of-range value makes that block / index
 *     count as absent (a hole) and ORs a QSA_DERR_* bit into *error_word when
 *     error_word is not NULL.  Kernels never trap.
 *   - Concurrent calls that share a workspace race; give each stream its own.
 *   - Any host thread may call.  The work runs on the calling thread's current
 *     device (cudaGetDevice): when no context or that device's primary
 *     context is current, the call binds the thread to the primary context
 *     before it launches (a context the caller made current itself is used
 *     as it is); the stream and every pointer must belong to that context.
 *     The one-time setup of the large-shared-memory kernels (their attribute
 *     and occupancy queries) is kept per device for the life of the
 *     process: after cudaDeviceReset, or from a second context on the same
 *     device, launches fail with QSA_ERR_CUDA (nothing runs) rather than
 *     redo it.
 *   - FP16 tensors must start on a 16-byte boundary; int tensors on their
 *     element size.  num_rows == 0 is a legal no-op.
 */
#ifndef QSA_H
#define QSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define QSA_API __attribute__((visibility("default")))
#else
#define QSA_API
#endif

/* Fixed contract ("Exact contracts" / Selection and Attention). */
#define QSA_TOKEN_TOPK       2048  /* tokens selected from compressed blocks */
#define QSA_COMPRESS_RATIO   4     /* tokens per compressed key */
#define QSA_TOPK_BLOCKS      512   /* QSA_TOKEN_TOPK / QSA_COMPRESS_RATIO */
#define QSA_OUT_WIDTH        2051  /* 2048 + 3-token tail */
#define QSA_SEL_HEADS        4     /* selection query [R,4,128] */
#define QSA_SEL_DIM          128
#define QSA_CMP_PAGE_KEYS    128   /* compressed cache [P,128,1,128] */
#define QSA_ATT_HEADS        3     /* attention query/output [R,3,256] */
#define QSA_ATT_DIM          256
#define QSA_KV_PAGE_TOKENS   512   /* K/V strides [262144,512,256,1] */
#define QSA_KV_PAGE_STRIDE   262144
#define QSA_KV_TOKEN_STRIDE  512
#define QSA_V_OFFSET         256   /* V storage_offset relative to K */

typedef int qsa_status;
#define QSA_OK              0
#define QSA_ERR_NULL        1  /* a required pointer is NULL */
#define QSA_ERR_DTYPE       2  /* a dtype tag is not the contract's */
#define QSA_ERR_SHAPE       3  /* a shape is not the contract's */
#define QSA_ERR_STRIDE      4  /* a stride / storage offset is not the contract's */
#define QSA_ERR_ALIGN       5  /* a pointer is misaligned */
#define QSA_ERR_CONTRACT    6  /* token_topk / compress_ratio / scale / width */
#define QSA_ERR_WORKSPACE   7  /* workspace missing or too small */
#define QSA_ERR_ALIAS       8  /* an output overlaps an input */
#define QSA_ERR_CUDA        9  /* a CUDA runtime call or launch failed */
#define QSA_ERR_SCRATCH_LIMIT 10 /* request exceeds the static scratch array */

typedef int qsa_dtype;
#define QSA_DT_F16   1
#define QSA_DT_BF16  2
#define QSA_DT_F32   3
#define QSA_DT_I32   4
#define QSA_DT_I64   5
#define QSA_DT_F8E4M3 6   /* OCP FP8 E4M3 ("fn"): compressed keys only */

/* Device-detected data errors, ORed into *error_word (never cleared by the
 * library; the caller zeroes it when it wants a fresh reading). */
#define QSA_DERR_REQUEST   1u  /* token_to_request[r] outside [0, num_reqs) */
#define QSA_DERR_CMP_PAGE  2u  /* compressed page id negative / >= P, or the
                                  block lies beyond the page-table columns */
#define QSA_DERR_KV_PAGE   4u  /* K/V page id negative / >= P_kv, or the
                                  index lies beyond the page-table columns */
#define QSA_DERR_TIMEOUT   8u  /* a device-side wait exceeded its 1 s bound;
                                  the call's outputs are not valid */

typedef struct CUstream_st* qsa_stream_t;  /* == cudaStream_t; NULL = legacy */

/* Human-readable name of a status code (static storage). */
QSA_API const char* qsa_status_string(qsa_status status);

/* Library version: major*10000 + minor*100 + patch. */
QSA_API int qsa_version(void);

/*
 * Workspace for qsa_select_paged_tokens: bytes needed for num_rows rows whose
 * compressed page table has cmp_pt_cols columns (each row may hold up to
 * cmp_pt_cols*128 visible blocks).  Alignment 256 bytes.
 */
QSA_API size_t qsa_select_workspace_bytes(int64_t num_rows, int64_t cmp_pt_cols);

/*
 * qsa_select_paged_tokens -- per row r:
 *   req = token_to_request[r], L = seq_lens[req], pos = query_positions[r]
 *   V   = max(0, min((pos+1)//4, L//4))          visible compressed blocks
 *   for b in [0,V): page = cmp_page_table[req, b//128];
 *       key_b = cmp_cache[page, b%128, 0, :]     (128 halves)
 *       s_b   = sum_{h<4} ReLU(q_sel[r,h,:] . key_b)   (binary32, one fixed
 *               summation order; see the design notes)
 *   keep the min(512, #scored) blocks with the largest s_b (exact ties: the
 *   smaller b first), in that order; write out[r, 4j..4j+3] = 4b..4b+3 for
 *   the j-th kept block, then the tail tokens 4V..min(pos, L-1) ascending,
 *   then -1 up to column 2050.
 *
 * Arguments
 *   q_sel            FP16 [num_rows,4,128], strides q_sel_strides (must be
 *                    {512,128,1}: contiguous)
 *   cmp_cache        [P,128,1,128], shape cmp_shape, strides cmp_strides in
 *                    elements (must be {16384,128,*,1}; the size-1 dim's
 *                    stride is ignored).  cmp_dtype QSA_DT_F16, or
 *                    QSA_DT_F8E4M3 for the optional e4m3 compressed indexer
 *                    cache (qsa_cache.py, QSAStateBackend cache dtypes): each
 *                    key element is decoded exactly (E4M3 values are exact in
 *                    fp16) and scored by the same rule and order.
 *   cmp_page_table   int32 [num_reqs, cmp_pt_cols], row stride cmp_pt_stride0
 *                    (elements, >= cmp_pt_cols), column stride 1
 *   token_to_request int32 [num_rows]
 *   seq_lens         int32 [num_reqs]
 *   query_positions  int64 [num_rows]
 *   token_topk       must be 2048; compress_ratio must be 4
 *   out_indices      int32 [num_rows, out_width] with row stride out_stride0;
 *                    out_width must be 2051
 *   workspace        device scratch of >= qsa_select_workspace_bytes(
 *                    num_rows, cmp_pt_cols) bytes, 256-byte aligned
 *   error_word       device uint32 or NULL (QSA_DERR_* bits ORed in)
 *   stream           launch stream
 */
QSA_API qsa_status qsa_select_paged_tokens(
    const void* q_sel, qsa_dtype q_sel_dtype, int64_t num_rows,
    const int64_t q_sel_strides[3],
    const void* cmp_cache, qsa_dtype cmp_dtype, const int64_t cmp_shape[4],
    const int64_t cmp_strides[4],
    const void* cmp_page_table, qsa_dtype cmp_pt_dtype, int64_t num_reqs,
    int64_t cmp_pt_cols, int64_t cmp_pt_stride0,
    const void* token_to_request, qsa_dtype t2r_dtype,
    const void* seq_lens, qsa_dtype seq_lens_dtype,
    const void* query_positions, qsa_dtype qpos_dtype,
    int32_t token_topk, int32_t compress_ratio,
    void* out_indices, qsa_dtype out_dtype, int64_t out_width, int64_t out_stride0,
    void* workspace, size_t workspace_bytes,
    uint32_t* error_word, qsa_stream_t stream);

/*
 * Workspace for qsa_sparse_attention: bytes needed for num_rows rows of
 * index_width logical indices.  Alignment 256 bytes.
 */
QSA_API size_t qsa_attention_workspace_bytes(int64_t num_rows, int64_t index_width);

/*
 * qsa_sparse_attention -- per row r and head h < 3:
 *   req = token_to_request[r]; the valid entries are the j with
 *   indices[r,j] = i >= 0 whose page kv_page_table[req, i//512] is in range;
 *   K_j = k_cache[page, i%512, 0, :], V_j = v_cache[page, i%512, 0, :];
 *   z_j = scale * (q[r,h,:] . K_j)
 *   out[r,h,:] = sum_j e^{z_j} V_j / sum_j e^{z_j}  (FP32 accumulation,
 *                rounded to FP16 nearest-even); every occurrence of a
 *                duplicated index is its own term; no valid entry -> zeros.
 *
 * Arguments
 *   q                FP16 [num_rows,3,256] contiguous (q_strides {768,256,1})
 *   k_cache, v_cache FP16 views [P_kv,512,1,256] of one exact-packed buffer:
 *                    strides {262144,512,*,1} each (size-1 dim ignored) and
 *                    v_cache == k_cache + 256 halves (V storage_offset 256)
 *   kv_page_table    int32 [num_reqs, kv_pt_cols], row stride kv_pt_stride0
 *   token_to_request int32 [num_rows]
 *   indices          int32 [num_rows, index_width], row stride idx_stride0;
 *                    -1 (any negative) = hole; index_width in [0, 2051]
 *   scale            finite and > 0 (the contract uses 1/sqrt(256) = 1/16)
 *   out              FP16 [num_rows,3,256] contiguous; must not overlap any
 *                    input
 *   workspace        >= qsa_attention_workspace_bytes(num_rows, index_width)
 *   error_word       device uint32 or NULL
 */
QSA_API qsa_status qsa_sparse_attention(
    const void* q, qsa_dtype q_dtype, int64_t num_rows, const int64_t q_strides[3],
    const void* k_cache, const void* v_cache, qsa_dtype kv_dtype,
    const int64_t kv_shape[4], const int64_t k_strides[4], const int64_t v_strides[4],
    const void* kv_page_table, qsa_dtype kv_pt_dtype, int64_t num_reqs,
    int64_t kv_pt_cols, int64_t kv_pt_stride0,
    const void* token_to_request, qsa_dtype t2r_dtype,
    const void* indices, qsa_dtype idx_dtype, int64_t index_width, int64_t idx_stride0,
    float scale,
    void* out, qsa_dtype out_dtype, const int64_t out_strides[3],
    void* workspace, size_t workspace_bytes,
    uint32_t* error_word, qsa_stream_t stream);

/*
 * Workspace for qsa_select_attend: bytes needed for num_rows rows whose
 * compressed page table has cmp_pt_cols columns.  Alignment 256 bytes.
 */
QSA_API size_t qsa_select_attend_workspace_bytes(int64_t num_rows, int64_t cmp_pt_cols);

/*
 * qsa_select_attend -- one decode step: qsa_select_paged_tokens followed by
 * qsa_sparse_attention over the indices it selects ("vLLM: integrate FP16
 * packed QSA extension", Summary: the fused selection and the exact-packed
 * attention kernel; "Exact contracts" / Selection and Attention), in one
 * call with one workspace.
 *
 * Results: out_indices bit for bit those of qsa_select_paged_tokens; out as
 * qsa_sparse_attention over out_indices (within its tolerance; bit for bit
 * too for batches above the fused limit).
 *
 * Arguments: the selection's, as qsa_select_paged_tokens (num_reqs rows in
 * both page tables), then the attention's, as qsa_sparse_attention without
 * its own token_to_request and index list (it uses token_to_request and
 * out_indices); one workspace of >= qsa_select_attend_workspace_bytes(
 * num_rows, cmp_pt_cols) bytes, 256-byte aligned.  out_indices and out must
 * not overlap each other, any input or the workspace.
 *
 * How it runs: for a batch of at most qsa_select_attend_fused_rows() rows
 * whose compressed page table is narrow enough (qsa_select_attend_fused_
 * cluster() says; wide tables mean long rows, which the score kernel spread
 * over every SM scores sooner), one kernel with one thread-block cluster
 * per row -- the cluster's 1 to 16 CTAs
 * score the row's pages, each runs the row's top-512 into its own shared
 * memory (the index hand-off) and attends over its share of the entries,
 * and the partials merge through distributed shared memory.  Larger batches
 * run the kernels of the two calls on the stream, chained by programmatic
 * dependent launch (score, top-k, attention, merge).  Nothing waits on the
 * host.  The indices are bit-identical either way; the attention output of
 * the fused kernel sums the softmax terms in another order than the two
 * calls' kernels (same tolerance).  Calls that share a workspace must not
 * overlap on the GPU.
 */
QSA_API qsa_status qsa_select_attend(
    const void* q_sel, qsa_dtype q_sel_dtype, int64_t num_rows,
    const int64_t q_sel_strides[3],
    const void* cmp_cache, qsa_dtype cmp_dtype, const int64_t cmp_shape[4],
    const int64_t cmp_strides[4],
    const void* cmp_page_table, qsa_dtype cmp_pt_dtype, int64_t num_reqs,
    int64_t cmp_pt_cols, int64_t cmp_pt_stride0,
    const void* token_to_request, qsa_dtype t2r_dtype,
    const void* seq_lens, qsa_dtype seq_lens_dtype,
    const void* query_positions, qsa_dtype qpos_dtype,
    int32_t token_topk, int32_t compress_ratio,
    void* out_indices, qsa_dtype out_dtype, int64_t out_width, int64_t out_stride0,
    const void* q_attn, qsa_dtype q_attn_dtype, const int64_t q_attn_strides[3],
    const void* k_cache, const void* v_cache, qsa_dtype kv_dtype,
    const int64_t kv_shape[4], const int64_t k_strides[4], const int64_t v_strides[4],
    const void* kv_page_table, qsa_dtype kv_pt_dtype,
    int64_t kv_pt_cols, int64_t kv_pt_stride0,
    float scale,
    void* out, qsa_dtype out_attn_dtype, const int64_t out_strides[3],
    void* workspace, size_t workspace_bytes,
    uint32_t* error_word, qsa_stream_t stream);

/*
 * The largest batch qsa_select_attend runs as its fused small-batch kernel
 * on the current device: as many rows as the device holds clusters of the
 * kernel at once (1 to 16 CTAs of one SM each), at most 256 (and only for
 * narrow enough page tables, see qsa_select_attend_fused_cluster).
 * cmp_dtype is the compressed cache's tag (QSA_DT_F16 or QSA_DT_F8E4M3;
 * another tag gives 0).  0 also when the device runs no such cluster.  The
 * first call on a device queries its cluster occupancy (host only, nothing
 * launched).
 */
QSA_API int64_t qsa_select_attend_fused_rows(qsa_dtype cmp_dtype);

/*
 * How qsa_select_attend runs a batch of num_rows rows whose compressed page
 * table has cmp_pt_cols columns on the current device: the CTAs of the
 * fused kernel's cluster per row (1 to 16: the most for which the device
 * holds num_rows such clusters at once), or 0 for the chained kernels.  The
 * fused kernel is taken when num_rows <= 256, the device holds num_rows
 * clusters of at least one CTA, cmp_pt_cols <= 128 * num_rows, and its
 * estimated time is at most the chained kernels': 25 us + 0.9 us per page
 * that one of its CTAs scores (ceil(cmp_pt_cols / CTAs) pages) against
 * 50 us + 6.25 ns per page of the batch (num_rows * cmp_pt_cols), fits to
 * decode steps measured on a GB300.  0 for a tag other than QSA_DT_F16 and
 * QSA_DT_F8E4M3 and for num_rows <= 0.
 */
QSA_API int64_t qsa_select_attend_fused_cluster(int64_t num_rows, int64_t cmp_pt_cols,
                                                qsa_dtype cmp_dtype);

/*
 * qsa_select_paged_tokens_static_scratch -- the same selection, for callers
 * that cannot give the library a device workspace.  The pages have no
 * counterpart to this entry point.
 *
 * Who needs it: code that cannot allocate device memory where it calls us,
 * e.g. a plugin that its host framework hands only input and output buffers
 * (no allocator), or a serving loop that bans cudaMalloc after start-up
 * because it synchronises the device and may fail under memory pressure.
 *
 * Scratch: a fixed array of QSA_STATIC_SCRATCH_BYTES inside the library,
 * held on every GPU that loads it until the process exits.  A call needs
 * qsa_select_workspace_bytes(num_rows, cmp_pt_cols) bytes of it; a larger
 * request returns QSA_ERR_SCRATCH_LIMIT without launching.  The call
 * allocates nothing.  All calls share the array: calls whose kernels overlap
 * on the GPU (different streams or host threads) race, so serialise them.
 * Nothing in the array needs clearing between calls: every slot a call
 * reads is written earlier in the same call -- as long as the call's device
 * waits complete.  If *error_word comes back with QSA_DERR_TIMEOUT, the
 * scoring stopped early, the top-k may have read slots left by an earlier
 * call (possibly of another workload), and out_indices is undefined; check
 * the error word before using the indices.
 *
 * Set-up: every call looks up the array's device address in the current
 * context (cudaGetSymbolAddress; no allocation).  The first call on a
 * device may also load the library's GPU code onto it; make that first call
 * before any stream capture.
 *
 * Validation: the arguments are checked exactly as qsa_select_paged_tokens
 * checks them (a malformed call returns that entry point's status); only a
 * well-formed request larger than the array returns QSA_ERR_SCRATCH_LIMIT.
 *
 * Arguments, validation and results are those of qsa_select_paged_tokens
 * without the workspace pair.
 */
#define QSA_STATIC_SCRATCH_BYTES (4u << 20)  /* 4 MiB: keys of 986,895 blocks */

QSA_API size_t qsa_static_scratch_bytes(void);

QSA_API qsa_status qsa_select_paged_tokens_static_scratch(
    const void* q_sel, qsa_dtype q_sel_dtype, int64_t num_rows,
    const int64_t q_sel_strides[3],
    const void* cmp_cache, qsa_dtype cmp_dtype, const int64_t cmp_shape[4],
    const int64_t cmp_strides[4],
    const void* cmp_page_table, qsa_dtype cmp_pt_dtype, int64_t num_reqs,
    int64_t cmp_pt_cols, int64_t cmp_pt_stride0,
    const void* token_to_request, qsa_dtype t2r_dtype,
    const void* seq_lens, qsa_dtype seq_lens_dtype,
    const void* query_positions, qsa_dtype qpos_dtype,
    int32_t token_topk, int32_t compress_ratio,
    void* out_indices, qsa_dtype out_dtype, int64_t out_width, int64_t out_stride0,
    uint32_t* error_word, qsa_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* QSA_H */
