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
// same call, so nothing needs clearing between calls.
//
// The host cannot use the array's name as a device address; the device
// address is looked up with cudaGetSymbolAddress once per device, the first
// time this entry point runs with that device current.  That first call may
// also load the library's GPU code onto the device, so make it before any
// stream capture.
#include "qsa.h"
#include "qsa_internal.h"

#include <mutex>

namespace {

constexpr size_t kStaticScratchBytes = QSA_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_select_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_select_scratch on the current device (set up once).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_select_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

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
  if (num_rows > 0 && cmp_pt_cols > 0 &&
      qsa::select_workspace_bytes(num_rows, cmp_pt_cols) > kStaticScratchBytes)
    return QSA_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  if (num_rows > 0) {
    if (scratch_address(&scratch) != cudaSuccess) return QSA_ERR_CUDA;
  }
  return qsa_select_paged_tokens(
      q_sel, q_sel_dtype, num_rows, q_sel_strides, cmp_cache, cmp_dtype, cmp_shape, cmp_strides,
      cmp_page_table, cmp_pt_dtype, num_reqs, cmp_pt_cols, cmp_pt_stride0, token_to_request,
      t2r_dtype, seq_lens, seq_lens_dtype, query_positions, qpos_dtype, token_topk,
      compress_ratio, out_indices, out_dtype, out_width, out_stride0, scratch,
      scratch ? kStaticScratchBytes : 0, error_word, stream);
}

}  // extern "C"
