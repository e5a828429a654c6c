// qsa_abi.cu -- the extern "C" boundary declared in include/qsa.h.
//
// Validation follows the fixed contracts of "vLLM: integrate FP16 packed QSA
// extension" ("Exact contracts"; the page's suite includes fail-closed
// dtype/layout/output checks): every host-visible argument is checked before
// anything is launched, and a mismatch returns a status without touching the
// GPU.  Only arguments that passed validation reach qsa::launch_*.
#include "qsa.h"
#include "qsa_internal.h"

#include <cmath>
#include <cstdint>

namespace {

using qsa::kAttDim;
using qsa::kAttHeads;
using qsa::kCmpPageKeys;
using qsa::kSelDim;
using qsa::kSelHeads;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Span {
  uintptr_t lo, hi;  // [lo, hi)
};

Span span(const void* p, int64_t bytes) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return Span{lo, lo + (uintptr_t)(bytes > 0 ? bytes : 0)};
}

bool overlaps(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi && a.hi > a.lo && b.hi > b.lo; }

constexpr int64_t kMaxRows = 65535;   // grid.y limit of the row-parallel kernels

}  // namespace

extern "C" {

const char* qsa_status_string(qsa_status s) {
  switch (s) {
    case QSA_OK: return "ok";
    case QSA_ERR_NULL: return "null pointer";
    case QSA_ERR_DTYPE: return "dtype is not the contract's";
    case QSA_ERR_SHAPE: return "shape is not the contract's";
    case QSA_ERR_STRIDE: return "stride or storage offset is not the contract's";
    case QSA_ERR_ALIGN: return "misaligned pointer";
    case QSA_ERR_CONTRACT: return "contract constant mismatch (token_topk, compress_ratio, scale or width)";
    case QSA_ERR_WORKSPACE: return "workspace missing or too small";
    case QSA_ERR_ALIAS: return "output overlaps an input";
    case QSA_ERR_CUDA: return "CUDA launch failed";
    case QSA_ERR_SCRATCH_LIMIT:
      return "request exceeds the static scratch array (use qsa_select_paged_tokens with a workspace)";
    default: return "unknown status";
  }
}

int qsa_version(void) { return 100; }

size_t qsa_select_workspace_bytes(int64_t num_rows, int64_t cmp_pt_cols) {
  if (num_rows <= 0 || cmp_pt_cols <= 0) return 0;
  return qsa::select_workspace_bytes(num_rows, cmp_pt_cols);
}

size_t qsa_attention_workspace_bytes(int64_t num_rows, int64_t index_width) {
  if (num_rows <= 0) return 0;
  return qsa::attention_workspace_bytes(num_rows, index_width < 0 ? 0 : index_width);
}

qsa_status qsa_select_paged_tokens(
    const void* q_sel, qsa_dtype q_sel_dtype, int64_t num_rows, const int64_t q_sel_strides[3],
    const void* cmp_cache, qsa_dtype cmp_dtype, const int64_t cmp_shape[4],
    const int64_t cmp_strides[4], const void* cmp_page_table, qsa_dtype cmp_pt_dtype,
    int64_t num_reqs, int64_t cmp_pt_cols, int64_t cmp_pt_stride0,
    const void* token_to_request, qsa_dtype t2r_dtype, const void* seq_lens,
    qsa_dtype seq_lens_dtype, const void* query_positions, qsa_dtype qpos_dtype,
    int32_t token_topk, int32_t compress_ratio, void* out_indices, qsa_dtype out_dtype,
    int64_t out_width, int64_t out_stride0, void* workspace, size_t workspace_bytes,
    uint32_t* error_word, qsa_stream_t stream) {
  // contract constants and dtypes ("Exact contracts" / Selection)
  if (token_topk != qsa::kTokenTopk || compress_ratio != qsa::kRatio) return QSA_ERR_CONTRACT;
  if (out_width != qsa::kOutWidth) return QSA_ERR_CONTRACT;
  if (q_sel_dtype != QSA_DT_F16) return QSA_ERR_DTYPE;
  if (cmp_dtype != QSA_DT_F16 && cmp_dtype != QSA_DT_F8E4M3) return QSA_ERR_DTYPE;
  const int64_t cmp_esize = cmp_dtype == QSA_DT_F16 ? 2 : 1;
  if (cmp_pt_dtype != QSA_DT_I32 || t2r_dtype != QSA_DT_I32 || seq_lens_dtype != QSA_DT_I32)
    return QSA_ERR_DTYPE;
  if (qpos_dtype != QSA_DT_I64 || out_dtype != QSA_DT_I32) return QSA_ERR_DTYPE;
  if (!q_sel_strides || !cmp_shape || !cmp_strides) return QSA_ERR_NULL;
  if (num_rows < 0 || num_rows > kMaxRows) return QSA_ERR_SHAPE;
  if (cmp_shape[0] < 0 || cmp_shape[1] != kCmpPageKeys || cmp_shape[2] != 1 ||
      cmp_shape[3] != kSelDim)
    return QSA_ERR_SHAPE;
  if (num_reqs < 0 || cmp_pt_cols < 0) return QSA_ERR_SHAPE;
  // the streaming loads address page p at row 256*p of a 32-bit row space;
  // per-launch page counts are 32-bit (at most 2^20 pages per request)
  if (cmp_shape[0] > (int64_t)(INT32_MAX / (2 * kCmpPageKeys))) return QSA_ERR_SHAPE;
  if (cmp_pt_cols > (int64_t)1 << 20) return QSA_ERR_SHAPE;
  if (num_rows == 0) return QSA_OK;
  if (num_reqs == 0 || cmp_pt_cols == 0) return QSA_ERR_SHAPE;
  // strides: q contiguous [R,4,128]; cache pages [P,128,1,128] contiguous
  if (q_sel_strides[0] != kSelHeads * kSelDim || q_sel_strides[1] != kSelDim ||
      q_sel_strides[2] != 1)
    return QSA_ERR_STRIDE;
  if (cmp_strides[0] != (int64_t)kCmpPageKeys * kSelDim || cmp_strides[1] != kSelDim ||
      cmp_strides[3] != 1)
    return QSA_ERR_STRIDE;
  if (cmp_pt_stride0 < cmp_pt_cols || out_stride0 < out_width) return QSA_ERR_STRIDE;
  if (!q_sel || !cmp_page_table || !token_to_request || !seq_lens || !query_positions ||
      !out_indices)
    return QSA_ERR_NULL;
  if (cmp_shape[0] > 0 && !cmp_cache) return QSA_ERR_NULL;
  if (!aligned(q_sel, 16) || !aligned(cmp_cache, 16) || !aligned(cmp_page_table, 4) ||
      !aligned(token_to_request, 4) || !aligned(seq_lens, 4) || !aligned(query_positions, 8) ||
      !aligned(out_indices, 4) || !aligned(error_word, 4))
    return QSA_ERR_ALIGN;
  const size_t need = qsa::select_workspace_bytes(num_rows, cmp_pt_cols);
  if (!workspace || workspace_bytes < need) return QSA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return QSA_ERR_ALIGN;

  const Span o = span(out_indices, ((num_rows - 1) * out_stride0 + out_width) * 4);
  const Span ins[] = {
      span(q_sel, num_rows * kSelHeads * kSelDim * 2),
      span(cmp_cache, cmp_shape[0] * kCmpPageKeys * kSelDim * cmp_esize),
      span(cmp_page_table, ((num_reqs - 1) * cmp_pt_stride0 + cmp_pt_cols) * 4),
      span(token_to_request, num_rows * 4),
      span(seq_lens, num_reqs * 4),
      span(query_positions, num_rows * 8),
      span(workspace, (int64_t)need),
  };
  for (const Span& s : ins)
    if (overlaps(o, s)) return QSA_ERR_ALIAS;
  if (error_word) {
    const Span e = span(error_word, 4);
    if (overlaps(o, e)) return QSA_ERR_ALIAS;
    for (const Span& s : ins)
      if (overlaps(e, s)) return QSA_ERR_ALIAS;
  }

  qsa::SelectParams p{};
  p.q_sel = static_cast<const __half*>(q_sel);
  p.cmp = cmp_cache;
  p.key_fp8 = cmp_dtype == QSA_DT_F8E4M3 ? 1 : 0;
  p.num_pages = cmp_shape[0];
  p.pt = static_cast<const int32_t*>(cmp_page_table);
  p.num_reqs = num_reqs;
  p.pt_cols = cmp_pt_cols;
  p.pt_stride0 = cmp_pt_stride0;
  p.t2r = static_cast<const int32_t*>(token_to_request);
  p.seq_lens = static_cast<const int32_t*>(seq_lens);
  p.qpos = static_cast<const int64_t*>(query_positions);
  p.out = static_cast<int32_t*>(out_indices);
  p.out_stride0 = out_stride0;
  p.scores = static_cast<uint32_t*>(workspace);
  p.vcap = cmp_pt_cols * kCmpPageKeys;
  p.err = error_word;
  p.R = (int)num_rows;
  const cudaError_t e = qsa::launch_select(p, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QSA_OK : QSA_ERR_CUDA;
}

qsa_status qsa_sparse_attention(
    const void* q, qsa_dtype q_dtype, int64_t num_rows, const int64_t q_strides[3],
    const void* k_cache, const void* v_cache, qsa_dtype kv_dtype, const int64_t kv_shape[4],
    const int64_t k_strides[4], const int64_t v_strides[4], const void* kv_page_table,
    qsa_dtype kv_pt_dtype, int64_t num_reqs, int64_t kv_pt_cols, int64_t kv_pt_stride0,
    const void* token_to_request, qsa_dtype t2r_dtype, const void* indices, qsa_dtype idx_dtype,
    int64_t index_width, int64_t idx_stride0, float scale, void* out, qsa_dtype out_dtype,
    const int64_t out_strides[3], void* workspace, size_t workspace_bytes, uint32_t* error_word,
    qsa_stream_t stream) {
  if (q_dtype != QSA_DT_F16 || kv_dtype != QSA_DT_F16 || out_dtype != QSA_DT_F16)
    return QSA_ERR_DTYPE;
  if (kv_pt_dtype != QSA_DT_I32 || t2r_dtype != QSA_DT_I32 || idx_dtype != QSA_DT_I32)
    return QSA_ERR_DTYPE;
  if (!(std::isfinite(scale) && scale > 0.f)) return QSA_ERR_CONTRACT;
  if (index_width < 0 || index_width > qsa::kOutWidth) return QSA_ERR_CONTRACT;
  if (!q_strides || !kv_shape || !k_strides || !v_strides || !out_strides) return QSA_ERR_NULL;
  if (num_rows < 0 || num_rows > kMaxRows) return QSA_ERR_SHAPE;
  if (kv_shape[0] < 0 || kv_shape[1] != qsa::kKvPageTokens || kv_shape[2] != 1 ||
      kv_shape[3] != kAttDim)
    return QSA_ERR_SHAPE;
  if (num_reqs < 0 || kv_pt_cols < 0) return QSA_ERR_SHAPE;
  // tokens are addressed as 32-bit page*512 + slot
  if (kv_shape[0] > (int64_t)(UINT32_MAX / qsa::kKvPageTokens)) return QSA_ERR_SHAPE;
  if (num_rows == 0) return QSA_OK;
  if (num_reqs == 0 || kv_pt_cols == 0) return QSA_ERR_SHAPE;
  if (q_strides[0] != kAttHeads * kAttDim || q_strides[1] != kAttDim || q_strides[2] != 1)
    return QSA_ERR_STRIDE;
  if (out_strides[0] != kAttHeads * kAttDim || out_strides[1] != kAttDim || out_strides[2] != 1)
    return QSA_ERR_STRIDE;
  // exact-packed K/V: strides [262144,512,*,1] (size-1 head dim ignored)
  for (const int64_t* st : {k_strides, v_strides})
    if (st[0] != qsa::kKvPageHalves || st[1] != qsa::kKvTokenHalves || st[3] != 1)
      return QSA_ERR_STRIDE;
  if (kv_pt_stride0 < kv_pt_cols || idx_stride0 < index_width) return QSA_ERR_STRIDE;
  if (!q || !kv_page_table || !token_to_request || !out) return QSA_ERR_NULL;
  if (index_width > 0 && !indices) return QSA_ERR_NULL;
  if (kv_shape[0] > 0 && (!k_cache || !v_cache)) return QSA_ERR_NULL;
  // V storage_offset 256 relative to K (one buffer, K then V per token)
  if (kv_shape[0] > 0 &&
      reinterpret_cast<uintptr_t>(v_cache) !=
          reinterpret_cast<uintptr_t>(k_cache) + (uintptr_t)kAttDim * 2)
    return QSA_ERR_STRIDE;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(kv_page_table, 4) ||
      !aligned(token_to_request, 4) || !aligned(indices, 4) || !aligned(out, 16) ||
      !aligned(error_word, 4))
    return QSA_ERR_ALIGN;
  const size_t need = qsa::attention_workspace_bytes(num_rows, index_width);
  if (!workspace || workspace_bytes < need) return QSA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return QSA_ERR_ALIGN;

  const Span o = span(out, num_rows * kAttHeads * kAttDim * 2);
  const Span ins[] = {
      span(q, num_rows * kAttHeads * kAttDim * 2),
      span(k_cache, kv_shape[0] * qsa::kKvPageHalves * 2),
      span(kv_page_table, ((num_reqs - 1) * kv_pt_stride0 + kv_pt_cols) * 4),
      span(token_to_request, num_rows * 4),
      span(indices, index_width > 0 ? ((num_rows - 1) * idx_stride0 + index_width) * 4 : 0),
      span(workspace, (int64_t)need),
  };
  for (const Span& s : ins)
    if (overlaps(o, s)) return QSA_ERR_ALIAS;
  if (error_word) {
    const Span e = span(error_word, 4);
    if (overlaps(o, e)) return QSA_ERR_ALIAS;
    for (const Span& s : ins)
      if (overlaps(e, s)) return QSA_ERR_ALIAS;
  }

  qsa::AttentionParams p{};
  p.q = static_cast<const __half*>(q);
  p.kv = static_cast<const __half*>(k_cache);
  p.num_pages = kv_shape[0];
  p.pt = static_cast<const int32_t*>(kv_page_table);
  p.num_reqs = num_reqs;
  p.pt_cols = kv_pt_cols;
  p.pt_stride0 = kv_pt_stride0;
  p.t2r = static_cast<const int32_t*>(token_to_request);
  p.idx = static_cast<const int32_t*>(indices);
  p.width = index_width;
  p.idx_stride0 = idx_stride0;
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.out = static_cast<__half*>(out);
  p.part = static_cast<float*>(workspace);
  p.nsplit = qsa::attention_splits(index_width);
  p.err = error_word;
  p.R = (int)num_rows;
  const cudaError_t e = qsa::launch_attention(p, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QSA_OK : QSA_ERR_CUDA;
}

}  // extern "C"
