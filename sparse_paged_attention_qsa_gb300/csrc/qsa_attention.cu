// qsa_attention.cu -- qsa_sparse_attention on sm_103a.
//
// "vLLM: integrate FP16 packed QSA extension", Summary (exact-packed
// attention kernel) and "Exact contracts"/Attention: FP16 Q/out [R,3,256];
// FP16 K/V exact-packed with strides [262144,512,256,1] and V at storage
// offset 256 (one KV head shared by the three query heads); logical indices
// [R,2051] int32 with holes and duplicates; caller-owned output.
//
// Split-width flash decoding (device code in qsa_attn_impl.cuh):
//   attn_partial_kernel  grid (splits, R); each CTA takes 256 consecutive
//                        entries of one row's index list (64 when the batch
//                        has at most 16 rows); each warp compacts its
//                        entries to the valid tokens and walks them 8 at a
//                        time (8 KiB of K/V in flight per warp).  Logits
//                        (mixed-precision FMA, fp16 operands, binary32
//                        accumulation) are reduced with one warp
//                        reduce-scatter per batch; the online softmax runs in
//                        base 2.  The four warps merge in shared memory and
//                        the CTA writes one partial (m, l, acc[256]) per head
//                        to the workspace.
//   attn_combine_kernel  one CTA per row merges the splits by log-sum-exp and
//                        rounds to FP16 (nearest even).  No valid entry -> 0.
#include "qsa_internal.h"
#include "qsa_device.cuh"
#include "qsa_attn_impl.cuh"

namespace qsa {
namespace {

using attn::kPartFloats;

constexpr int kAttWarps = 4;
constexpr int kAttThreads = kAttWarps * 32;
// Entries of a row's index list per CTA: 256 for batches of many rows (each
// warp walks 64 entries, 8 batches: the CTA's fixed costs -- the dependent
// index -> page-table -> K/V loads before streaming and the merge after it
// -- are amortised; 128 entries: 0.106 ms on 256 x 2048 rows, 256: 0.101,
// 512: 0.116 with too few CTAs to fill the GPU evenly), 64 for small batches
// (each warp walks 16 entries, 2 batches: a single row's 2051 entries go to
// 33 CTAs, so the row's latency is a couple of memory round trips).
constexpr int kSplitLarge = 256;
constexpr int kSplitSmall = 64;
constexpr int kSmallRows = 16;     // batches of at most this many rows take the small split
constexpr int kMaxSplitsLarge = (kOutWidth + kSplitLarge - 1) / kSplitLarge;   // 9
constexpr int kMaxSplitsSmall = (kOutWidth + kSplitSmall - 1) / kSplitSmall;   // 33

int split_entries(int64_t R) { return R <= kSmallRows ? kSplitSmall : kSplitLarge; }

// One CTA = kSplit consecutive entries of one row's index list, kSplit / 4
// per warp.
template <int kSplit>
__global__ void __launch_bounds__(kAttThreads)
attn_partial_kernel(const AttentionParams p) {
  constexpr int kWarpEntries = kSplit / kAttWarps;
  const int split = blockIdx.x;
  const int r = blockIdx.y;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;

  __shared__ attn::MergeSmem<kAttWarps> sm;
  __shared__ uint32_t sm_tok[kAttWarps][kWarpEntries];

  pdl_trigger();   // the combine kernel may be scheduled early (it waits)
  pdl_wait();      // launched as a dependent of the previous kernel (the selection's
                   // top-k when called after it): its output is complete and visible
  const int req = p.t2r[r];
  const bool rok = req >= 0 && req < p.num_reqs;
  if (!rok && split == 0 && tid == 0) report(p.err, kErrRequest);

  uint32_t qh[kAttHeads][4];
  attn::load_query(p, r, lane, qh);
  const int nvalid = attn::resolve_entries<kWarpEntries>(
      p, r, req, rok, (int64_t)split * kSplit + warp * kWarpEntries, sm_tok[warp], lane);
  attn::WarpState st;
  attn::init_state(st);
  attn::attend_tokens(p, sm_tok[warp], nvalid, qh, st, lane);
  attn::merge_warps<kAttWarps>(st, sm, p.part + ((int64_t)r * p.nsplit + split) * kPartFloats,
                               tid, warp, lane);
}

// One CTA per row: log-sum-exp merge of the row's split partials; thread d
// handles dim d of every head.
template <int kMaxSplits>
__global__ void __launch_bounds__(kAttDim)
attn_combine_kernel(const AttentionParams p) {
  __shared__ attn::CombineSmem<kMaxSplits> sm;
  const int r = blockIdx.x;
  pdl_wait();      // every split partial is written and visible
  attn::combine_row<kMaxSplits>(p, r, p.part + (int64_t)r * p.nsplit * kPartFloats, p.nsplit, sm,
                                threadIdx.x);
}

}  // namespace

int attention_splits(int64_t R, int64_t width) {
  const int e = split_entries(R);
  const int64_t s = (width + e - 1) / e;
  return s > 0 ? (int)s : 1;
}

size_t attention_workspace_bytes(int64_t R, int64_t width) {
  const size_t n = (size_t)R * (size_t)attention_splits(R, width) * kPartFloats * sizeof(float);
  return (n + 255) & ~(size_t)255;
}

cudaError_t launch_attention(const AttentionParams& p, cudaStream_t stream) {
  if (p.R == 0) return cudaSuccess;
  dim3 grid((unsigned)p.nsplit, (unsigned)p.R);
  // a programmatic dependent of whatever ran before on the stream: after the
  // selection's top-k (which triggers at its start) the launch and CTA
  // scheduling overlap the top-k's tail; the kernel waits before any read
  const bool small = p.R <= kSmallRows;
  cudaError_t e = small ? launch_after(attn_partial_kernel<kSplitSmall>, grid,
                                       dim3(kAttThreads), 0, stream, p)
                        : launch_after(attn_partial_kernel<kSplitLarge>, grid,
                                       dim3(kAttThreads), 0, stream, p);
  if (e != cudaSuccess) return e;
  return small ? launch_after(attn_combine_kernel<kMaxSplitsSmall>, dim3(p.R), dim3(kAttDim), 0,
                              stream, p)
               : launch_after(attn_combine_kernel<kMaxSplitsLarge>, dim3(p.R), dim3(kAttDim), 0,
                              stream, p);
}

}  // namespace qsa
