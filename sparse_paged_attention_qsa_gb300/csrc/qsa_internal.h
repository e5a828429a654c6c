// qsa_internal.h -- launch interface between the C-ABI layer (qsa_abi.cu) and
// the kernels (qsa_select.cu, qsa_attention.cu).  Arguments arrive here
// already validated; pointers are device pointers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

namespace qsa {

// Fixed contract ("vLLM: integrate FP16 packed QSA extension", Exact contracts)
constexpr int kTokenTopk = 2048;
constexpr int kRatio = 4;
constexpr int kTopkBlocks = kTokenTopk / kRatio;      // 512
constexpr int kOutWidth = kTokenTopk + kRatio - 1;    // 2051
constexpr int kSelHeads = 4;
constexpr int kSelDim = 128;
constexpr int kCmpPageKeys = 128;
constexpr int kCmpPageHalves = kCmpPageKeys * kSelDim;  // 16384
constexpr int kAttHeads = 3;
constexpr int kAttDim = 256;
constexpr int kKvPageTokens = 512;
constexpr int64_t kKvPageHalves = 262144;
constexpr int kKvTokenHalves = 512;

// device-side data error bits (same values as QSA_DERR_* in include/qsa.h)
constexpr uint32_t kErrRequest = 1u;
constexpr uint32_t kErrCmpPage = 2u;
constexpr uint32_t kErrKvPage = 4u;
constexpr uint32_t kErrTimeout = 8u;

struct SelectParams {
  const __half* q_sel;        // [R,4,128]
  const void* cmp;            // [P,128,1,128] fp16 or E4M3, page stride 16384 elements
  int key_fp8;                // 1: E4M3 keys, 0: fp16 keys
  int64_t num_pages;
  const int32_t* pt;          // [num_reqs, pt_cols], row stride pt_stride0
  int64_t num_reqs, pt_cols, pt_stride0;
  const int32_t* t2r;         // [R]
  const int32_t* seq_lens;    // [num_reqs]
  const int64_t* qpos;        // [R]
  int32_t* out;               // [R, 2051], row stride out_stride0
  int64_t out_stride0;
  uint32_t* scores;           // workspace: [R, vcap] ordered score keys
  uint32_t* umax;             // workspace: [R, vcap/16] largest key of each run of 16 blocks
  int64_t vcap;               // pt_cols * 128
  uint32_t* err;              // nullable
  int R;
#ifdef QSA_WAIT_TEST
  int64_t test_withhold;      // test build: CTA 0 issues no copy for this stage fill (-1: none)
#endif
};


struct AttentionParams {
  const __half* q;            // [R,3,256]
  const __half* kv;           // exact-packed base: token t of page p at
                              // kv + p*262144 + t*512; K = +0..255, V = +256..511
  int64_t num_pages;
  const int32_t* pt;          // [num_reqs, pt_cols], row stride pt_stride0
  int64_t num_reqs, pt_cols, pt_stride0;
  const int32_t* t2r;         // [R]
  const int32_t* idx;         // [R, width], row stride idx_stride0
  int64_t width, idx_stride0;
  float scale_log2;           // scale * log2(e)
  __half* out;                // [R,3,256]
  float* part;                // workspace partials
  int nsplit;
  uint32_t* err;              // nullable
  int R;
  int inputs_early;           // 1: the kernel before it on the stream writes none of q,
                              // t2r, pt (only idx), so they may be read before its end
};

// Launch `kernel` so that it may start while the previous kernel in the
// stream is finishing (programmatic dependent launch); the kernel must call
// pdl_wait() before reading what that kernel wrote.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_after(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

size_t select_workspace_bytes(int64_t R, int64_t pt_cols);
size_t attention_workspace_bytes(int64_t R, int64_t width);
cudaError_t launch_select(const SelectParams& p, cudaStream_t stream);
cudaError_t launch_attention(const AttentionParams& p, cudaStream_t stream);
// Select, then attend over the selection's output (a.idx, a.width and
// a.nsplit are set here); a.part holds attention_workspace_bytes(R, 2051).
cudaError_t launch_select_attend(const SelectParams& p, const AttentionParams& a,
                                 cudaStream_t stream);
int attention_splits(int64_t R, int64_t width);

}  // namespace qsa
