// qsa_attention.cu -- qsa_sparse_attention on sm_103a.
//
// "vLLM: integrate FP16 packed QSA extension", Summary (exact-packed
// attention kernel) and "Exact contracts"/Attention: FP16 Q/out [R,3,256];
// FP16 K/V exact-packed with strides [262144,512,256,1] and V at storage
// offset 256 (one KV head shared by the three query heads); logical indices
// [R,2051] int32 with holes and duplicates; caller-owned output.
//
// Flash decoding over pieces of each row's index list (device code in
// qsa_attn_impl.cuh): a warp compacts its entries to valid tokens and walks
// them 8 at a time -- the 3 x 8 logits as one chain of 16 mma.m16n8k16
// (fp16 operands, binary32 accumulation), base-2 online softmax, P.V with
// packed binary32 FMAs; the warps of a CTA merge in shared memory into one
// partial (m, l, acc[256]) per head, and one CTA per row merges a row's
// partials by log-sum-exp and rounds to FP16 (nearest even; no valid entry
// gives 0).  Two ways of cutting the lists:
//   attn_stream_kernel   batches of more than 32 rows: one wave of CTAs, each
//                        streaming an equal run of 32-entry chunks of the
//                        lists laid end to end (runs cross row boundaries);
//                        every warp keeps the next batch's K/V in flight
//                        while it computes the current one;
//   attn_partial_kernel  batches of up to 32 rows: grid (33, R), 64 entries
//                        per CTA, so a single row's 2051 entries are spread
//                        over 33 CTAs and its latency is a few memory round
//                        trips.
#include "qsa_internal.h"
#include "qsa_device.cuh"
#include "qsa_attn_impl.cuh"

#include <mutex>

namespace qsa {
namespace {

using attn::kPartFloats;

constexpr int kAttWarps = 4;
constexpr int kAttThreads = kAttWarps * 32;
// batches of at most this many rows take the split kernel: more CTAs per row
// than the stream split gives them (17 rows: attention 0.021 vs 0.029 ms;
// 32 rows: 0.029 vs 0.031 ms; from 64 rows the stream split is as fast or faster)
constexpr int kSmallRows = 32;
constexpr int kSplit = 64;         // entries of a row's list per CTA of the split kernel
constexpr int kMaxSplits = (kOutWidth + kSplit - 1) / kSplit;   // 33

// One CTA = kSplit consecutive entries of one row's index list, kSplit / 4
// per warp.
__global__ void __launch_bounds__(kAttThreads)
attn_partial_kernel(const AttentionParams p) {
  constexpr int kWarpEntries = kSplit / kAttWarps;
  const int split = blockIdx.x;
  const int r = blockIdx.y;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;

  __shared__ attn::MergeSmem<kAttWarps> sm;
  __shared__ attn::QFrag qf;
  __shared__ uint32_t sm_tok[kAttWarps][kWarpEntries];

  pdl_trigger();   // the combine kernel may be scheduled early (it waits)
  // Launched as a dependent of the previous kernel on the stream (the
  // selection's top-k when called after it), whose output -- the index
  // list -- is complete and visible only after pdl_wait().  When that
  // kernel is known to write nothing else the attention reads, the request
  // id, the query and the request's page-table row are fetched first.
  int req = 0;
  if (p.inputs_early) {
    req = p.t2r[r];
    attn::stage_query(p, r, qf, tid, kAttThreads);
    if (tid == 0 && req >= 0 && req < p.num_reqs)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(p.pt + (int64_t)req * p.pt_stride0));
  }
  pdl_wait();
  if (!p.inputs_early) {
    req = p.t2r[r];
    attn::stage_query(p, r, qf, tid, kAttThreads);
  }
  const bool rok = req >= 0 && req < p.num_reqs;
  if (!rok && split == 0 && tid == 0) report(p.err, kErrRequest);
  const int nvalid = attn::resolve_entries<kWarpEntries>(
      p, r, req, rok, (int64_t)split * kSplit + warp * kWarpEntries, sm_tok[warp], lane);
  __syncthreads();   // the query fragments are staged
  attn::WarpState st;
  attn::init_state(st);
  attn::attend_tokens_mma(p, sm_tok[warp], nvalid, qf, st, lane);
  attn::finish_mma_state(st, lane);
  attn::merge_warps<kAttWarps>(st, sm, p.part + ((int64_t)r * p.nsplit + split) * kPartFloats,
                               tid, warp, lane);
}

// --- stream-K split (batches of more than kSmallRows rows) -------------------
//
// The rows' index lists, cut into 32-entry chunks (C per row), are laid end
// to end (T = R*C chunks) and cut into G equal runs, one per CTA, with G the
// number of CTAs the GPU holds at once: one wave, every CTA streams the same
// number of entries, and a CTA's dependent index -> page-table -> K/V chain
// is paid once per row it touches instead of once per fixed-width split.  A run
// crosses row boundaries; per row it touches, the CTA merges its four warps
// and writes one partial into the row's slot b - b_lo(row), b_lo(row) being
// the first CTA whose run reaches the row.  Every run holds at least Lmin
// chunks, so a row meets at most kStreamSlots runs.

constexpr int kChunk = 32;                // entries per chunk (one warp load of indices)
constexpr int kPieceChunks = 4;           // chunks a warp resolves at once
constexpr int kStreamSlots = 9;           // partials per row
constexpr int kMinRunChunks = 8;

struct StreamPlan {
  int64_t T;        // chunks in all
  int64_t G;        // CTAs
  int64_t C;        // chunks per row
};

// the CTA whose run holds chunk x
__device__ __forceinline__ int64_t run_of(int64_t x, const StreamPlan& s) {
  return ((x + 1) * s.G - 1) / s.T;
}

// Resolve the warp's chunks j0, j0 + 4, ... (j0 + 4k < je, k < kPieceChunks)
// of row r's index list to tokens, compacted in order into tok[]; returns
// how many.  All index loads are issued before the page-table loads.
__device__ __forceinline__ int resolve_piece(const AttentionParams& p, int64_t r, int req, bool rok,
                                             int64_t j0, int64_t je, uint32_t* tok, int lane) {
  int32_t iv[kPieceChunks];
#pragma unroll
  for (int k = 0; k < kPieceChunks; ++k) {
    const int64_t j = j0 + 4 * k;
    const int64_t e = j * kChunk + lane;
    iv[k] = j < je && e < p.width ? p.idx[r * p.idx_stride0 + e] : -1;
  }
#pragma unroll
  for (int k = 0; k < kPieceChunks; ++k) iv[k] = rok ? iv[k] : -1;
  int32_t pg[kPieceChunks];
#pragma unroll
  for (int k = 0; k < kPieceChunks; ++k) {
    const int64_t col = iv[k] >> 9;
    pg[k] = iv[k] >= 0 && col < p.pt_cols ? p.pt[(int64_t)req * p.pt_stride0 + col] : -1;
  }
  int nvalid = 0;
#pragma unroll
  for (int k = 0; k < kPieceChunks; ++k) {
    const bool valid = iv[k] >= 0 && pg[k] >= 0 && pg[k] < p.num_pages;
    if (iv[k] >= 0 && !valid) report(p.err, kErrKvPage);
    const unsigned vmask = __ballot_sync(0xffffffffu, valid);
    if (valid)
      tok[nvalid + __popc(vmask & ((1u << lane) - 1u))] =
          (uint32_t)pg[k] * kKvPageTokens + (uint32_t)(iv[k] & 511);
    nvalid += __popc(vmask);
  }
  __syncwarp();
  return nvalid;
}

__global__ void __launch_bounds__(kAttThreads)
attn_stream_kernel(const AttentionParams p, const StreamPlan sp) {
  __shared__ attn::MergeSmem<kAttWarps> sm;
  __shared__ attn::QFrag qf;
  __shared__ uint32_t sm_tok[kAttWarps][kPieceChunks * kChunk];
  const int64_t b = blockIdx.x;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int64_t x1 = sp.T * (b + 1) / sp.G;

  pdl_trigger();   // the combine kernel may be scheduled early (it waits)
  for (int64_t x = sp.T * b / sp.G; x < x1;) {
    // one row segment: row r, chunks [c0, c1) of its list
    const int64_t r = x / sp.C;
    const int64_t c0 = x - r * sp.C;
    const int64_t c1 = (x1 < (r + 1) * sp.C ? x1 : (r + 1) * sp.C) - r * sp.C;
    const int req = p.t2r[r];
    const bool rok = req >= 0 && req < p.num_reqs;
    if (!rok && c0 == 0 && tid == 0) report(p.err, kErrRequest);
    attn::stage_query(p, (int)r, qf, tid, kAttThreads);
    int64_t j0 = c0 + warp;                    // the warp's chunks: j0, j0 + 4, ...
    int n = j0 < c1 ? resolve_piece(p, r, req, rok, j0, c1, sm_tok[warp], lane) : 0;
    __syncthreads();                           // the query fragments are staged
    attn::WarpState st;
    attn::init_state(st);
    while (j0 < c1) {
      attn::attend_tokens_mma_pipe(p, sm_tok[warp], n, qf, st, lane);
      j0 += 4 * kPieceChunks;
      __syncwarp();                            // the piece's tokens are read
      if (j0 < c1) n = resolve_piece(p, r, req, rok, j0, c1, sm_tok[warp], lane);
    }
    attn::finish_mma_state(st, lane);
    // the row's slot; < p.nsplit by the plan's run length (checked on the
    // host), guarded here so a plan error can never write past the row
    const int64_t slot = b - run_of(r * sp.C, sp);
    attn::merge_warps<kAttWarps>(st, sm, p.part + (r * p.nsplit + (slot < p.nsplit ? slot : 0)) *
                                                      kPartFloats,
                                 tid, warp, lane);
    __syncthreads();   // shared memory is reused by the next segment
    x = r * sp.C + c1;
  }
}

// One CTA per row: merge the row's stream partials (slots 0 .. n-1).
__global__ void __launch_bounds__(kAttDim)
attn_stream_combine_kernel(const AttentionParams p, const StreamPlan sp) {
  __shared__ attn::CombineSmem<kStreamSlots> sm;
  const int64_t r = blockIdx.x;
  pdl_wait();      // every partial is written and visible
  const int n = (int)(run_of(r * sp.C + sp.C - 1, sp) - run_of(r * sp.C, sp) + 1);
  attn::combine_row<kStreamSlots>(p, (int)r, p.part + r * p.nsplit * kPartFloats, n, sm,
                                  threadIdx.x);
}

// One CTA per row: log-sum-exp merge of the row's split partials; thread d
// handles dim d of every head.
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
  if (R > kSmallRows) return kStreamSlots;
  const int64_t s = (width + kSplit - 1) / kSplit;
  return s > 0 ? (int)s : 1;
}

size_t attention_workspace_bytes(int64_t R, int64_t width) {
  const size_t n = (size_t)R * (size_t)attention_splits(R, width) * kPartFloats * sizeof(float);
  return (n + 255) & ~(size_t)255;
}

namespace {

// CTAs of the stream kernel the device holds at once (cached per device)
cudaError_t stream_ctas(int64_t* out) {
  static std::mutex mu;
  static int64_t ctas[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (ctas[dev] == 0) {
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_stream_kernel, kAttThreads, 0);
    if (e != cudaSuccess) return e;
    ctas[dev] = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
  }
  *out = ctas[dev];
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_attention(const AttentionParams& p, cudaStream_t stream) {
  if (p.R == 0) return cudaSuccess;
  if (p.R > kSmallRows) {
    int64_t slots = 0;
    cudaError_t e = stream_ctas(&slots);
    if (e != cudaSuccess) return e;
    StreamPlan sp;
    sp.C = p.width > 0 ? (p.width + kChunk - 1) / kChunk : 1;   // width 0: one empty chunk
    sp.T = (int64_t)p.R * sp.C;
    // every run >= lmin chunks: a row of C chunks meets <= kStreamSlots runs
    const int64_t need = (sp.C - 1 + kStreamSlots - 2) / (kStreamSlots - 1);
    const int64_t lmin = need > kMinRunChunks ? need : kMinRunChunks;
    const int64_t g = sp.T / lmin;
    sp.G = g < 1 ? 1 : (g < slots ? g : slots);
    // the shortest run, floor(T/G), must keep a row within kStreamSlots runs
    const int64_t shortest = sp.T / sp.G;
    if (sp.G > 1 && (sp.C - 1 + shortest - 1) / shortest + 1 > kStreamSlots)
      return cudaErrorInvalidValue;
    if (p.nsplit < kStreamSlots) return cudaErrorInvalidValue;
    // a plain launch, not a programmatic dependent of the selection's top-k:
    // the runs are sized for a GPU-wide single wave, and CTAs placed early
    // beside the top-k's made the end-to-end step 0.483 ms instead of 0.444
    // (256 x 131072, pipelined host copies)
    attn_stream_kernel<<<dim3((unsigned)sp.G), dim3(kAttThreads), 0, stream>>>(p, sp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_after(attn_stream_combine_kernel, dim3((unsigned)p.R), dim3(kAttDim), 0, stream,
                        p, sp);
  }
  // a programmatic dependent of whatever ran before on the stream: after the
  // selection's top-k (which triggers at its start) the launch and CTA
  // scheduling overlap the top-k's tail; the kernels wait before any read
  cudaError_t e = launch_after(attn_partial_kernel, dim3((unsigned)p.nsplit, (unsigned)p.R),
                               dim3(kAttThreads), 0, stream, p);
  if (e != cudaSuccess) return e;
  return launch_after(attn_combine_kernel, dim3(p.R), dim3(kAttDim), 0, stream, p);
}

}  // namespace qsa
