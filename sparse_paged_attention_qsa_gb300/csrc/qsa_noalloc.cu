// qsa_noalloc.cu -- qsa_select_paged_tokens_static_scratch: selection for
// callers that cannot hand the library a device workspace.
//
// Some callers cannot allocate device memory at the point where they call
// us: a plugin that a host framework gives only its input and output buffers
// (no allocator handle), or a serving loop that forbids cudaMalloc after
// start-up because it synchronises the device and can fail under memory
// pressure.  For them this entry point takes its scratch from a fixed array
// compiled into the library instead of from a caller workspace.
//
// The array lives in device global memory on every GPU that loads the
// library, for as long as the process runs.  Its size is the hard limit on
// what one call may ask for; larger requests are refused with
// QSA_ERR_SCRATCH_LIMIT and must use qsa_select_paged_tokens with a
// workspace.  All calls share the one array, so calls whose kernels overlap
// on the GPU (other streams, other host threads) race and must be serialised
// by the caller.  Every scratch slot a call reads is written earlier in the
// same call when its device waits complete, so nothing needs clearing
// between calls (the timeout case is below).
//
// The host cannot use the array's name as a device address.  Every call
// looks the address up with cudaGetSymbolAddress in the context current at
// the call (cheap, and it allocates nothing), so a reset device or another
// context on the same ordinal never receives an address from an earlier
// context.  The first call on a device may also load the library's GPU code
// onto it, so make that first call before any stream capture.
//
// Validation comes first: the call is checked exactly as the workspace entry
// point checks it (with no workspace, which makes a well-formed call stop at
// the workspace check without launching), so a malformed call returns the
// status that entry point gives; only a well-formed request larger than the
// array returns QSA_ERR_SCRATCH_LIMIT.
//
// After a device wait gives up (QSA_DERR_TIMEOUT in the error word) the
// scoring stopped early and the top-k may have read slots of the array that
// an earlier call wrote; the indices of that call are undefined.
#include "qsa.h"
#include "qsa_internal.h"
#include "qsa_host.h"

namespace {

constexpr size_t kStaticScratchBytes = QSA_STATIC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_select_scratch[kStaticScratchBytes];

}  // namespace

extern "C" {

size_t qsa_static_scratch_bytes(void) { return kStaticScratchBytes; }

qsa_status qsa_select_paged_tokens_static_scratch(
    const void* q_sel, qsa_dtype q_sel_dtype, int64_t num_rows, const int64_t q_sel_strides[3],
    const void* cmp_cache, qsa_dtype cmp_dtype, const int64_t cmp_shape[4],
    const int64_t cmp_strides[4], const void* cmp_page_table, qsa_dtype cmp_pt_dtype,
    int64_t num_reqs, int64_t cmp_pt_cols, int64_t cmp_pt_stride0,
    const void* token_to_request, qsa_dtype t2r_dtype, const void* seq_lens,
    qsa_dtype seq_lens_dtype, const void* query_positions, qsa_dtype qpos_dtype,
    int32_t token_topk, int32_t compress_ratio, void* out_indices, qsa_dtype out_dtype,
    int64_t out_width, int64_t out_stride0, uint32_t* error_word, qsa_stream_t stream) {
  // argument checks of the workspace entry point; with no workspace a
  // well-formed, non-empty call stops at QSA_ERR_WORKSPACE, launching nothing
  const qsa_status st = qsa_select_paged_tokens(
      q_sel, q_sel_dtype, num_rows, q_sel_strides, cmp_cache, cmp_dtype, cmp_shape, cmp_strides,
      cmp_page_table, cmp_pt_dtype, num_reqs, cmp_pt_cols, cmp_pt_stride0, token_to_request,
      t2r_dtype, seq_lens, seq_lens_dtype, query_positions, qpos_dtype, token_topk,
      compress_ratio, out_indices, out_dtype, out_width, out_stride0, nullptr, 0, error_word,
      stream);
  if (st != QSA_ERR_WORKSPACE) return st;    // an argument error, or an empty batch (QSA_OK)
  if (qsa::select_workspace_bytes(num_rows, cmp_pt_cols) > kStaticScratchBytes)
    return QSA_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  qsa::bind_calling_thread();
  if (cudaGetSymbolAddress(&scratch, g_select_scratch) != cudaSuccess || scratch == nullptr)
    return QSA_ERR_CUDA;
  return qsa_select_paged_tokens(
      q_sel, q_sel_dtype, num_rows, q_sel_strides, cmp_cache, cmp_dtype, cmp_shape, cmp_strides,
      cmp_page_table, cmp_pt_dtype, num_reqs, cmp_pt_cols, cmp_pt_stride0, token_to_request,
      t2r_dtype, seq_lens, seq_lens_dtype, query_positions, qpos_dtype, token_topk,
      compress_ratio, out_indices, out_dtype, out_width, out_stride0, scratch,
      kStaticScratchBytes, error_word, stream);
}

}  // extern "C"
