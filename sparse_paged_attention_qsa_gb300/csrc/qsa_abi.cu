// qsa_abi.cu -- the extern "C" boundary declared in include/qsa.h.
//
// Validation follows the fixed contracts of "vLLM: integrate FP16 packed QSA
// extension" ("Exact contracts"; the page's suite includes fail-closed
// dtype/layout/output checks): every host-visible argument is checked before
// anything is launched, and a mismatch returns a status without touching the
// GPU.  Only arguments that passed validation reach qsa::launch_*.
#include "qsa.h"
#include "qsa_internal.h"
#include "qsa_fused.h"
#include "qsa_host.h"

#include <algorithm>
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

constexpr int64_t kMaxRows = 65535;   // rows per call (keeps every grid dimension in range)

// Selection arguments (everything but the workspace): contract constants,
// dtypes, shapes, strides, null pointers, alignment.  On success fills *p
// (all but the workspace), the output's span and the inputs' spans.
qsa_status check_select(
    const void* q_sel, qsa_dtype q_sel_dtype, int64_t num_rows, const int64_t q_sel_strides[3],
    const void* cmp_cache, qsa_dtype cmp_dtype, const int64_t cmp_shape[4],
    const int64_t cmp_strides[4], const void* cmp_page_table, qsa_dtype cmp_pt_dtype,
    int64_t num_reqs, int64_t cmp_pt_cols, int64_t cmp_pt_stride0,
    const void* token_to_request, qsa_dtype t2r_dtype, const void* seq_lens,
    qsa_dtype seq_lens_dtype, const void* query_positions, qsa_dtype qpos_dtype,
    int32_t token_topk, int32_t compress_ratio, void* out_indices, qsa_dtype out_dtype,
    int64_t out_width, int64_t out_stride0, uint32_t* error_word, qsa::SelectParams* p,
    Span* out_span, Span (&ins)[6], bool* empty) {
  *empty = false;
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
  if (num_rows == 0) {
    *empty = true;
    return QSA_OK;
  }
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
  *out_span = span(out_indices, ((num_rows - 1) * out_stride0 + out_width) * 4);
  ins[0] = span(q_sel, num_rows * kSelHeads * kSelDim * 2);
  ins[1] = span(cmp_cache, cmp_shape[0] * kCmpPageKeys * kSelDim * cmp_esize);
  ins[2] = span(cmp_page_table, ((num_reqs - 1) * cmp_pt_stride0 + cmp_pt_cols) * 4);
  ins[3] = span(token_to_request, num_rows * 4);
  ins[4] = span(seq_lens, num_reqs * 4);
  ins[5] = span(query_positions, num_rows * 8);
  p->q_sel = static_cast<const __half*>(q_sel);
  p->cmp = cmp_cache;
  p->key_fp8 = cmp_dtype == QSA_DT_F8E4M3 ? 1 : 0;
  p->num_pages = cmp_shape[0];
  p->pt = static_cast<const int32_t*>(cmp_page_table);
  p->num_reqs = num_reqs;
  p->pt_cols = cmp_pt_cols;
  p->pt_stride0 = cmp_pt_stride0;
  p->t2r = static_cast<const int32_t*>(token_to_request);
  p->seq_lens = static_cast<const int32_t*>(seq_lens);
  p->qpos = static_cast<const int64_t*>(query_positions);
  p->out = static_cast<int32_t*>(out_indices);
  p->out_stride0 = out_stride0;
  p->vcap = cmp_pt_cols * kCmpPageKeys;
  p->err = error_word;
  p->R = (int)num_rows;
  return QSA_OK;
}

// Attention arguments (everything but the workspace), as check_select.
qsa_status check_attention(
    const void* q, qsa_dtype q_dtype, int64_t num_rows, const int64_t q_strides[3],
    const void* k_cache, const void* v_cache, qsa_dtype kv_dtype, const int64_t kv_shape[4],
    const int64_t k_strides[4], const int64_t v_strides[4], const void* kv_page_table,
    qsa_dtype kv_pt_dtype, int64_t num_reqs, int64_t kv_pt_cols, int64_t kv_pt_stride0,
    const void* token_to_request, qsa_dtype t2r_dtype, const void* indices, qsa_dtype idx_dtype,
    int64_t index_width, int64_t idx_stride0, float scale, void* out, qsa_dtype out_dtype,
    const int64_t out_strides[3], uint32_t* error_word, qsa::AttentionParams* p, Span* out_span,
    Span (&ins)[5], bool* empty) {
  *empty = false;
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
  if (num_rows == 0) {
    *empty = true;
    return QSA_OK;
  }
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
  *out_span = span(out, num_rows * kAttHeads * kAttDim * 2);
  ins[0] = span(q, num_rows * kAttHeads * kAttDim * 2);
  ins[1] = span(k_cache, kv_shape[0] * qsa::kKvPageHalves * 2);
  ins[2] = span(kv_page_table, ((num_reqs - 1) * kv_pt_stride0 + kv_pt_cols) * 4);
  ins[3] = span(token_to_request, num_rows * 4);
  ins[4] = span(indices, index_width > 0 ? ((num_rows - 1) * idx_stride0 + index_width) * 4 : 0);
  p->q = static_cast<const __half*>(q);
  p->kv = static_cast<const __half*>(k_cache);
  p->num_pages = kv_shape[0];
  p->pt = static_cast<const int32_t*>(kv_page_table);
  p->num_reqs = num_reqs;
  p->pt_cols = kv_pt_cols;
  p->pt_stride0 = kv_pt_stride0;
  p->t2r = static_cast<const int32_t*>(token_to_request);
  p->idx = static_cast<const int32_t*>(indices);
  p->width = index_width;
  p->idx_stride0 = idx_stride0;
  p->scale_log2 = (float)((double)scale * 1.4426950408889634);
  p->out = static_cast<__half*>(out);
  p->err = error_word;
  p->R = (int)num_rows;
  return QSA_OK;
}

// Workspace of the one-call step: the selection's score keys and unit
// maxima, then the attention's partials.
struct OneCallLayout {
  size_t part, total;
};

OneCallLayout one_call_layout(int64_t num_rows, int64_t cmp_pt_cols) {
  const auto up = [](size_t n) { return (n + 255) & ~(size_t)255; };
  OneCallLayout l;
  l.part = up(qsa::select_workspace_bytes(num_rows, cmp_pt_cols));
  l.total = l.part + up(qsa::attention_workspace_bytes(num_rows, qsa::kOutWidth));
  return l;
}

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

size_t qsa_select_attend_workspace_bytes(int64_t num_rows, int64_t cmp_pt_cols) {
  if (num_rows <= 0 || cmp_pt_cols <= 0) return 0;
  return one_call_layout(num_rows, cmp_pt_cols).total;
}

int64_t qsa_select_attend_fused_rows(qsa_dtype cmp_dtype) {
  if (cmp_dtype != QSA_DT_F16 && cmp_dtype != QSA_DT_F8E4M3) return 0;
  qsa::bind_calling_thread();
  return qsa::fused_decode_max_rows(cmp_dtype == QSA_DT_F8E4M3);
}

int64_t qsa_select_attend_fused_cluster(int64_t num_rows, int64_t cmp_pt_cols,
                                        qsa_dtype cmp_dtype) {
  if (cmp_dtype != QSA_DT_F16 && cmp_dtype != QSA_DT_F8E4M3) return 0;
  if (num_rows <= 0 || num_rows > INT32_MAX) return 0;
  qsa::bind_calling_thread();
  return qsa::fused_decode_cluster((int)num_rows, cmp_pt_cols, cmp_dtype == QSA_DT_F8E4M3);
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
  qsa::SelectParams p{};
  Span o, ins[6];
  bool empty = false;
  const qsa_status st = check_select(
      q_sel, q_sel_dtype, num_rows, q_sel_strides, cmp_cache, cmp_dtype, cmp_shape, cmp_strides,
      cmp_page_table, cmp_pt_dtype, num_reqs, cmp_pt_cols, cmp_pt_stride0, token_to_request,
      t2r_dtype, seq_lens, seq_lens_dtype, query_positions, qpos_dtype, token_topk,
      compress_ratio, out_indices, out_dtype, out_width, out_stride0, error_word, &p, &o, ins,
      &empty);
  if (st != QSA_OK || empty) return st;
  // aliasing among the caller's tensors first, then the workspace (so a call
  // without a workspace still learns of every other argument error)
  for (const Span& s : ins)
    if (overlaps(o, s)) return QSA_ERR_ALIAS;
  if (error_word) {
    const Span e = span(error_word, 4);
    if (overlaps(o, e)) return QSA_ERR_ALIAS;
    for (const Span& s : ins)
      if (overlaps(e, s)) return QSA_ERR_ALIAS;
  }
  const size_t need = qsa::select_workspace_bytes(num_rows, cmp_pt_cols);
  if (!workspace || workspace_bytes < need) return QSA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return QSA_ERR_ALIGN;
  const Span ws = span(workspace, (int64_t)need);
  if (overlaps(o, ws)) return QSA_ERR_ALIAS;
  if (error_word && overlaps(span(error_word, 4), ws)) return QSA_ERR_ALIAS;
  p.scores = static_cast<uint32_t*>(workspace);
  p.umax = p.scores + num_rows * p.vcap;
  qsa::bind_calling_thread();
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
  qsa::AttentionParams p{};
  Span o, ins[5];
  bool empty = false;
  const qsa_status st = check_attention(
      q, q_dtype, num_rows, q_strides, k_cache, v_cache, kv_dtype, kv_shape, k_strides, v_strides,
      kv_page_table, kv_pt_dtype, num_reqs, kv_pt_cols, kv_pt_stride0, token_to_request, t2r_dtype,
      indices, idx_dtype, index_width, idx_stride0, scale, out, out_dtype, out_strides, error_word,
      &p, &o, ins, &empty);
  if (st != QSA_OK || empty) return st;
  const size_t need = qsa::attention_workspace_bytes(num_rows, index_width);
  if (!workspace || workspace_bytes < need) return QSA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return QSA_ERR_ALIGN;
  const Span ws = span(workspace, (int64_t)need);
  if (overlaps(o, ws)) return QSA_ERR_ALIAS;
  for (const Span& s : ins)
    if (overlaps(o, s)) return QSA_ERR_ALIAS;
  if (error_word) {
    const Span e = span(error_word, 4);
    if (overlaps(o, e) || overlaps(e, ws)) return QSA_ERR_ALIAS;
    for (const Span& s : ins)
      if (overlaps(e, s)) return QSA_ERR_ALIAS;
  }
  p.part = static_cast<float*>(workspace);
  p.nsplit = qsa::attention_splits(num_rows, index_width);
  qsa::bind_calling_thread();
  const cudaError_t e = qsa::launch_attention(p, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QSA_OK : QSA_ERR_CUDA;
}

qsa_status qsa_select_attend(
    const void* q_sel, qsa_dtype q_sel_dtype, int64_t num_rows, const int64_t q_sel_strides[3],
    const void* cmp_cache, qsa_dtype cmp_dtype, const int64_t cmp_shape[4],
    const int64_t cmp_strides[4], const void* cmp_page_table, qsa_dtype cmp_pt_dtype,
    int64_t num_reqs, int64_t cmp_pt_cols, int64_t cmp_pt_stride0,
    const void* token_to_request, qsa_dtype t2r_dtype, const void* seq_lens,
    qsa_dtype seq_lens_dtype, const void* query_positions, qsa_dtype qpos_dtype,
    int32_t token_topk, int32_t compress_ratio, void* out_indices, qsa_dtype out_dtype,
    int64_t out_width, int64_t out_stride0, const void* q_attn, qsa_dtype q_attn_dtype,
    const int64_t q_attn_strides[3], const void* k_cache, const void* v_cache,
    qsa_dtype kv_dtype, const int64_t kv_shape[4], const int64_t k_strides[4],
    const int64_t v_strides[4], const void* kv_page_table, qsa_dtype kv_pt_dtype,
    int64_t kv_pt_cols, int64_t kv_pt_stride0, float scale, void* out, qsa_dtype out_attn_dtype,
    const int64_t out_strides[3], void* workspace, size_t workspace_bytes, uint32_t* error_word,
    qsa_stream_t stream) {
  qsa::SelectParams p{};
  Span o_sel, ins_sel[6];
  bool empty = false;
  qsa_status st = check_select(
      q_sel, q_sel_dtype, num_rows, q_sel_strides, cmp_cache, cmp_dtype, cmp_shape, cmp_strides,
      cmp_page_table, cmp_pt_dtype, num_reqs, cmp_pt_cols, cmp_pt_stride0, token_to_request,
      t2r_dtype, seq_lens, seq_lens_dtype, query_positions, qpos_dtype, token_topk,
      compress_ratio, out_indices, out_dtype, out_width, out_stride0, error_word, &p, &o_sel,
      ins_sel, &empty);
  if (st != QSA_OK) return st;
  // the attention reads the selection's output as its index list
  qsa::AttentionParams a{};
  Span o_att, ins_att[5];
  bool empty_att = false;
  st = check_attention(q_attn, q_attn_dtype, num_rows, q_attn_strides, k_cache, v_cache, kv_dtype,
                       kv_shape, k_strides, v_strides, kv_page_table, kv_pt_dtype, num_reqs,
                       kv_pt_cols, kv_pt_stride0, token_to_request, t2r_dtype, out_indices,
                       out_dtype, out_width, out_stride0, scale, out, out_attn_dtype, out_strides,
                       error_word, &a, &o_att, ins_att, &empty_att);
  if (st != QSA_OK || empty) return st;
  const OneCallLayout l = one_call_layout(num_rows, cmp_pt_cols);
  if (!workspace || workspace_bytes < l.total) return QSA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return QSA_ERR_ALIGN;
  const Span ws = span(workspace, (int64_t)l.total);
  // outputs: the indices and the attention output; inputs: both operations'
  // inputs (not the index list, which is the selection's own output)
  const Span outs[] = {o_sel, o_att};
  const Span ins[] = {ins_sel[0], ins_sel[1], ins_sel[2], ins_sel[3], ins_sel[4], ins_sel[5],
                      ins_att[0], ins_att[1], ins_att[2], ws};
  if (overlaps(o_sel, o_att)) return QSA_ERR_ALIAS;
  for (const Span& o : outs)
    for (const Span& s : ins)
      if (overlaps(o, s)) return QSA_ERR_ALIAS;
  if (error_word) {
    const Span e = span(error_word, 4);
    for (const Span& o : outs)
      if (overlaps(e, o)) return QSA_ERR_ALIAS;
    for (const Span& s : ins)
      if (overlaps(e, s)) return QSA_ERR_ALIAS;
  }
  unsigned char* w = static_cast<unsigned char*>(workspace);
  p.scores = reinterpret_cast<uint32_t*>(w);
  p.umax = p.scores + num_rows * p.vcap;
  a.part = reinterpret_cast<float*>(w + l.part);
  qsa::bind_calling_thread();
  const cudaError_t e = qsa::launch_select_attend(p, a, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QSA_OK : QSA_ERR_CUDA;
}

}  // extern "C"
