// qsa_fused.h -- the fused small-batch decode step (qsa_fused.cu): one
// thread-block cluster per row scores, selects and attends in one kernel.
// Which batches take it, and its launcher.
#pragma once
#include <cuda.h>
#include "qsa_internal.h"

namespace qsa {

// The step takes batches of at most kFusedMaxRows rows (and as many as the
// device holds clusters of the kernel at once, 1 to 16 CTAs each) ...
constexpr int kFusedMaxRows = 256;
// ... whose compressed page table is at most this many columns wide per
// row of the batch: one cluster scores a row on 1-16 SMs, so a lone row of
// more pages is scored sooner by the score kernel on every SM (one row of
// 131072 tokens, 256 columns: 41.6 us fused against 38.6 us chained; two
// such rows: 40.7 against 42.7) ...
constexpr int kFusedColsPerRow = 128;
// ... and whose estimated time is at most the chained kernels'.  Both are
// linear in the pages scored: the fused step takes about 25 us + 0.9 us per
// page its busiest CTA scores (ceil(pt_cols / CS); a CTA scores about 40 GB/s
// of keys), the chained kernels about 50 us + 6.25 ns per page of the batch
// (R * pt_cols; the score kernel on every SM).  Fits to steps of 1-64 rows
// of 131072 tokens on a GB300 (fused 39.6-142 us, chained 44-156 us, each
// within 5 %; they also pick the faster path at 72-152 rows); in units of
// 1/1600 us:
constexpr int64_t kFusedBaseCost = 40000, kFusedPageCost = 1440;
constexpr int64_t kChainBaseCost = 80000, kChainPageCost = 10;
cudaError_t launch_fused_decode(const SelectParams& p, const AttentionParams& a,
                                const CUtensorMap& map, int cs, cudaStream_t stream);

// The largest batch the fused step takes on the current device.
int fused_decode_max_rows(bool key_fp8);
// CTAs per row's cluster of the fused kernel for R rows and a compressed
// page table of pt_cols columns, 0 = the chained kernels.
int fused_decode_cluster(int R, int64_t pt_cols, bool key_fp8);

}  // namespace qsa
