// qsa_select.cu -- qsa_select_paged_tokens on sm_103a.
//
// "vLLM: integrate FP16 packed QSA extension", Summary (fused selection:
// paged compressed keys, four-head ReLU(Q*K) scores, streaming top-512,
// expansion to 2,048 tokens, three-token tail, [R,2051] int32 padded with -1)
// and "Exact contracts"/Selection (descending score, ascending logical index
// on exact ties).  Visible blocks follow qsa_cache.py,
// _build_qsa_metadata_kernel: max(0, min((pos+1)//4, seq_len//4)).
//
// Two kernels on the caller's stream:
//   score_kernel  persistent (one CTA per SM): streams every visible
//                 compressed page of every row once through a TMA ring in
//                 shared memory (the dominant HBM stream: 256 B per key) and
//                 writes a 32-bit ordered score key per block, and the
//                 largest key of each run of 16 blocks, to the workspace;
//   topk_kernel   one CTA per row: the candidates (every key of a short
//                 row; for a long row the keys of the runs whose maximum
//                 reaches a lower bound of the 512-th largest), exact radix
//                 select of the top 512 over them, ordering of the winners,
//                 expansion, tail and -1 padding.
//
// Score arithmetic (must match the oracle bit for bit): per head, four
// 32-dim slices; in each slice an even-dim and an odd-dim binary32 chain
// (fp16 x fp16 products are exact in binary32), P = E + O; a quad of lanes
// holds the four slices of one key and reduces d = (P0 + P2) + (P1 + P3);
// ReLU; s = (r0 + r1) + (r2 + r3).  The ordered key is bits(s) + 1 (s >= +0,
// so float order equals unsigned order); 0 marks a block without a key.
#include "qsa_internal.h"
#include "qsa_device.cuh"
#include "qsa_select_impl.cuh"
#include "qsa_fused.h"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

namespace qsa {
namespace {

constexpr int kMaxRows = 1024;                          // rows per launch (row tables in smem)
constexpr int kGroupRows = 8;    // rows of one request scored from one page pass (aligned windows)
// row tables: req, visible blocks; group tables: first row (+ sentinel), pages,
// weighted page prefix (64-bit, + total)
constexpr size_t kTableBytes = (size_t)(4 * kMaxRows + 1) * sizeof(int) +
                               (size_t)(kMaxRows + 1) * sizeof(int64_t);
constexpr size_t kScoreSmem = (size_t)kRingBytes + 1024 + 2 * kMaxStages * 8 +
                              kMaxStages * 16 + kTableBytes;
static_assert(kScoreSmem <= 227 * 1024 - 256, "score kernel shared memory");


struct StageDesc {
  int row;        // first row of the group; -1: no more work
  int b0;         // first block of the page
  int nrows;      // rows of the group (each scores its own visible keys)
  int pad;
};

// Work weight of one page for a group of n rows: a page costs at least its
// stream time (about three rows' worth of fp16 scoring; one row for E4M3
// pages, where scoring alone sets the pace), else the scoring of n rows.
template <bool kFp8>
__device__ __forceinline__ int page_cost(int n) {
  constexpr int kFloor = kFp8 ? 1 : 3;
  return n > kFloor ? n : kFloor;
}

// Persistent streaming score kernel over rows [0, p.R) (p.R <= kMaxRows).
//
// Row groups: consecutive rows of one request inside an aligned window of
// kGroupRows rows (a request's speculative / multi-token query rows) read
// the same compressed pages, so each page is streamed once per group and
// scored for every row of the group (each row up to its own visible block
// count).  A plain decode batch has one row per group.
//
// Prologue: every CTA computes the row and group tables in shared memory --
// each row's request and visible blocks, each group's first row and page
// count (the most any of its rows sees), and the prefix sum of the groups'
// weighted page counts (page_cost) -- so the total work can be cut into
// equal contiguous ranges, one per CTA (a CTA changes groups rarely and
// reads consecutive page-table entries).
//
// Main loop, warp-specialised: lane 0 of the producer warp walks the CTA's
// range and streams each page (32 KiB = 128 keys x two 128-byte rows) into a
// ring of shared-memory stages with one 2-D TMA load (128-byte swizzle, L2
// evict-first), writing a small stage descriptor (group's first row, first
// block, rows) before arming the stage; it refills a stage as soon as every
// consumer warp has released it.  The page's n rows x 16 groups of 8 keys
// are split evenly over the 8 consumer warps (2n consecutive units each,
// row-major, taken in pairs of one row), so for n = 1, 2, 4 or 8 a warp keeps
// one row -- and its query slice in registers -- for all of a group's pages.  With the swizzle, lane (key k, slice t) reads row
// 2k + t/2, 16-byte chunks (4(t&1)+j) XOR (row & 7): the 8 lanes of each
// shared-memory phase hit 8 distinct bank groups, and each lane reads its
// slice in ascending order.
template <bool kFp8>
__global__ void __launch_bounds__(kScoreThreads, 1)
score_kernel(const SelectParams p, const __grid_constant__ CUtensorMap tmap) {
  constexpr int kPageBytes = KeyCfg<kFp8>::kPageBytes;
  constexpr int kStages = KeyCfg<kFp8>::kStages;
  extern __shared__ unsigned char smem_raw[];
  __shared__ int s_abort;
  __shared__ int64_t s_total;
  __shared__ int s_ngroups;
  __shared__ int64_t warp_sum[kScoreWarps];
  const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  const uint32_t base = raw + pad;
  const uint32_t bar_full = base + kRingBytes;
  const uint32_t bar_empty = bar_full + kMaxStages * 8;
  unsigned char* gbase = smem_raw + pad;
  StageDesc* desc = reinterpret_cast<StageDesc*>(gbase + kRingBytes + 2 * kMaxStages * 8);
  int64_t* grp_pre = reinterpret_cast<int64_t*>(desc + kMaxStages);  // weighted prefix [NG+1]
  int* row_req = reinterpret_cast<int*>(grp_pre + kMaxRows + 1);
  int* row_vs = row_req + kMaxRows;
  int* grp_first = row_vs + kMaxRows;        // [NG+1], sentinel p.R
  int* grp_pages = grp_first + kMaxRows + 1;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const bool is_producer_warp = warp == kScoreWarps;
  pdl_trigger();   // the top-k kernel may be scheduled wherever a CTA has exited

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kScoreWarps);
    }
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }

  // ---- prologue (consumer threads): row and group tables ----
  constexpr int kConsumerThreads = kScoreWarps * 32;
  constexpr int kRowsPerThread = kMaxRows / kConsumerThreads;
  static_assert(kMaxRows % kConsumerThreads == 0, "rows per consumer thread");
  if (!is_producer_warp) {
    const auto consumers_sync = [] {
      asm volatile("bar.sync 1, %0;" ::"r"(kConsumerThreads) : "memory");
    };
    // block-wide exclusive scan over the consumer threads (int64)
    const auto scan = [&](int64_t mine, int64_t& total) -> int64_t {
      int64_t incl = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (lane == 31) warp_sum[warp] = incl;
      consumers_sync();
      int64_t before = 0;
      total = 0;
      for (int w = 0; w < kScoreWarps; ++w) {
        before += (w < warp) ? warp_sum[w] : 0;
        total += warp_sum[w];
      }
      consumers_sync();                     // warp_sum is reused by the next scan
      return before + incl - mine;
    };
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) {
      const int r = tid * kRowsPerThread + i;
      if (r < p.R) {
        const RowSetup rs = row_setup(p, r);
        const int64_t Vs = rs.ok ? (rs.V < p.vcap ? rs.V : p.vcap) : 0;
        row_req[r] = rs.ok ? rs.req : -1;
        row_vs[r] = (int)Vs;
      }
    }
    consumers_sync();
    // group starts: window boundary, request change, or a row without a request
    int starts = 0, nstart = 0;
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) {
      const int r = tid * kRowsPerThread + i;
      if (r < p.R) {
        const bool st = (r % kGroupRows) == 0 || row_req[r] < 0 || row_req[r] != row_req[r - 1];
        starts |= (int)st << i;
        nstart += st;
      }
    }
    int64_t ngroups = 0;
    int g = (int)scan(nstart, ngroups);
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i)
      if (starts >> i & 1) grp_first[g++] = tid * kRowsPerThread + i;
    if (tid == 0) grp_first[ngroups] = p.R;
    consumers_sync();
    // per group: pages (the most any of its rows sees) and weighted pages
    int64_t wsum = 0;
    int64_t wg[kRowsPerThread];
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) {
      const int gi = tid * kRowsPerThread + i;
      wg[i] = 0;
      if (gi < ngroups) {
        const int f = grp_first[gi], l = grp_first[gi + 1];
        int vmax = 0;
        for (int r = f; r < l; ++r) vmax = row_vs[r] > vmax ? row_vs[r] : vmax;
        const int pages = (vmax + kCmpPageKeys - 1) / kCmpPageKeys;
        grp_pages[gi] = pages;
        wg[i] = (int64_t)pages * page_cost<kFp8>(l - f);
      }
      wsum += wg[i];
    }
    int64_t total = 0;
    int64_t run = scan(wsum, total);
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) {
      const int gi = tid * kRowsPerThread + i;
      if (gi < ngroups) grp_pre[gi] = run;
      run += wg[i];
    }
    if (tid == 0) {
      grp_pre[ngroups] = total;
      s_total = total;
      s_ngroups = (int)ngroups;
    }
  }
  __syncthreads();

  const int64_t W = s_total;
  const int64_t w_begin = W * blockIdx.x / gridDim.x;
  const int64_t w_end = W * (blockIdx.x + 1) / gridDim.x;
  volatile int* abort_flag = &s_abort;
  int64_t issued = 0;
  int64_t withheld = -1;   // test build: the fill that got no copy (never drained)

  if (is_producer_warp) {
    // ---------------- producer (one lane) ----------------
    if (lane == 0) {
      const uint64_t policy = evict_first_policy();
      const int NG = s_ngroups;
      // first owned page: the first (group, page) whose weighted start is >= w_begin
      int pgrp = NG, pcol = 0;
      if (w_begin < w_end && NG > 0) {
        int lo = 0, hi = NG - 1;             // last group with grp_pre <= w_begin
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (grp_pre[mid] <= w_begin) lo = mid; else hi = mid - 1;
        }
        pgrp = lo;
        const int64_t c = page_cost<kFp8>(grp_first[lo + 1] - grp_first[lo]);
        pcol = (int)((w_begin - grp_pre[lo] + c - 1) / c);
        while (pgrp < NG && pcol >= grp_pages[pgrp]) {
          ++pgrp;
          pcol = 0;
        }
      }
      for (;;) {
        const int s = (int)(issued % kStages);
        const uint32_t ph = (uint32_t)((issued / kStages) & 1);
        if (issued >= kStages && !mbar_wait(bar_empty + 8 * s, ph ^ 1u)) {
          *abort_flag = 1;
          report(p.err, kErrTimeout);
          break;
        }
        if (*abort_flag) break;
        // next owned page with a loadable physical page (the others get no key)
        int32_t pg = -1;
        while (pgrp < NG) {
          const int row0 = grp_first[pgrp];
          const int n = grp_first[pgrp + 1] - row0;
          if (grp_pre[pgrp] + (int64_t)pcol * page_cost<kFp8>(n) >= w_end) break;
          const int b0 = pcol * kCmpPageKeys;
          pg = __ldg(p.pt + (int64_t)row_req[row0] * p.pt_stride0 + pcol);
          if (++pcol >= grp_pages[pgrp]) {
            pcol = 0;
            ++pgrp;
            while (pgrp < NG && grp_pages[pgrp] == 0) ++pgrp;
          }
          if (pg >= 0 && pg < p.num_pages) {
            desc[s].row = row0;
            desc[s].b0 = b0;
            desc[s].nrows = n;
            break;
          }
          for (int j = 0; j < n; ++j) {          // no key for these blocks
            const int nk = min(row_vs[row0 + j] - b0, kCmpPageKeys);
            uint32_t* zr = p.scores + (int64_t)(row0 + j) * p.vcap + b0;
            for (int k = 0; k < nk; ++k) zr[k] = 0u;
            uint32_t* zu = p.umax + (int64_t)(row0 + j) * (p.vcap / kUnitKeys) + b0 / kUnitKeys;
            for (int k = 0; kUnitKeys * k < nk; ++k) zu[k] = 0u;
          }
          report(p.err, kErrCmpPage);
          pg = -1;
        }
        ++issued;
        if (pg >= 0) {
#ifdef QSA_WAIT_TEST
          // test build: leave this fill without a copy, so the consumers'
          // wait on it runs out (the failure-detection test)
          if (blockIdx.x == 0 && issued - 1 == p.test_withhold) {
            withheld = issued - 1;
            continue;
          }
#endif
          mbar_expect_tx(bar_full + 8 * s, kPageBytes);
          tma_load_2d(base + s * kPageBytes, &tmap, 0, pg * KeyCfg<kFp8>::kRowsPerKey * kCmpPageKeys,
                      bar_full + 8 * s, policy);
        } else {                    // range done: mark the stage as the end
          desc[s].row = -1;
          mbar_arrive(bar_full + 8 * s);
          break;
        }
      }
    }
  } else {
    // ---------------- consumers ----------------
    const int t = lane & 3;          // 32-dim slice of the key
    const int kslot = lane >> 2;     // key within a group of 8
    uint32_t q[kSelHeads][16];
    int loaded_row = -1;
    uint32_t* srow = nullptr;
    uint32_t* urow = nullptr;
    for (int64_t used = 0;; ++used) {
      const int s = (int)(used % kStages);
      const uint32_t ph = (uint32_t)((used / kStages) & 1);
      if (!mbar_wait(bar_full + 8 * s, ph)) {
        *abort_flag = 1;
        report(p.err, kErrTimeout);
        break;
      }
      const StageDesc d = desc[s];
      if (d.row < 0) break;
      const uint32_t stage = base + s * kPageBytes;
      // the page's n rows x 16 key groups, row-major, split evenly: this warp
      // takes 2n consecutive units, in pairs of key groups of one row
      const int units = 2 * d.nrows;
      for (int u = warp * units; u < (warp + 1) * units; u += 2) {
        const int row = d.row + u / kKeyGroups;
        const int g0 = u % kKeyGroups;
        uint4 kv[2][4];
        load_key_groups<kFp8, 2>(stage, g0, t, kslot, kv);   // in flight while the row is checked
        const int nk = row_vs[row] - d.b0;   // this row's visible keys in the page
        if (nk <= 8 * g0) continue;          // both groups past the row's visible keys
        if (row != loaded_row) {
          loaded_row = row;
          srow = p.scores + (int64_t)row * p.vcap;
          urow = p.umax + (int64_t)row * (p.vcap / kUnitKeys);
          load_query_slice(p.q_sel + (int64_t)row * kSelHeads * kSelDim, t, q);
        }
        uint32_t um = 0;                     // the unit's (these 16 keys') largest key
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          const uint32_t key = quad_score(q, kv[g], t);
          const int k = (g0 + g) * 8 + kslot;
          if (k < nk) {
            if (t == 0) srow[d.b0 + k] = key;
            um = key > um ? key : um;
          }
        }
        um = __reduce_max_sync(0xffffffffu, um);
        if (lane == 0) urow[(d.b0 + 8 * g0) / kUnitKeys] = um;   // 8 * g0 < nk here
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);   // this warp is done with the stage
      if (*abort_flag) break;
    }
  }
  __syncthreads();
  // After a timeout, let every copy this CTA issued land before it exits
  // (bounded by the full drain limit, whatever the stage waits' limit).
  if (*abort_flag && is_producer_warp && lane == 0) {
    const int64_t first = issued > kStages ? issued - kStages : 0;
    for (int64_t n = first; n < issued; ++n)
      if (n != withheld)
        mbar_wait(bar_full + 8 * (int)(n % kStages), (uint32_t)((n / kStages) & 1),
                  kDrainLimitNs);
  }
}

template <bool kDense>
__global__ void __launch_bounds__(kTopkThreads, 2)
topk_kernel(const SelectParams p) {
  extern __shared__ __align__(16) unsigned char topk_smem[];
  TopkShared& sh = *reinterpret_cast<TopkShared*>(topk_smem);
  pdl_trigger();   // a dependent (the attention kernel) may be scheduled early (it waits)
  topk_row<kDense>(p, blockIdx.x, sh, RowOut{p.out + (int64_t)blockIdx.x * p.out_stride0});
}

}  // namespace

// [R, cols*128] score keys, then [R, cols*8] unit maxima
size_t select_workspace_bytes(int64_t R, int64_t pt_cols) {
  const size_t n = (size_t)R * (size_t)pt_cols * (kCmpPageKeys + kCmpPageKeys / kUnitKeys) *
                   sizeof(uint32_t);
  return (n + 255) & ~(size_t)255;
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 2-D view of the compressed cache in 128-byte rows: fp16 keys are two rows
// of 64 halves (256 rows per page), E4M3 keys one row of 128 bytes (128 rows
// per page); one box = one page; 128-byte swizzle.
cudaError_t encode_cmp_map(const SelectParams& p, CUtensorMap* map) {
  memset(map, 0, sizeof(*map));
  if (p.num_pages <= 0) return cudaSuccess;   // no page can be loaded
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const bool fp8 = p.key_fp8 != 0;
  const cuuint32_t rows_per_page = (fp8 ? 1 : 2) * kCmpPageKeys;
  cuuint64_t dims[2] = {fp8 ? 128u : 64u, (cuuint64_t)p.num_pages * rows_per_page};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {fp8 ? 128u : 64u, rows_per_page};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
                  const_cast<void*>(p.cmp), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

struct DeviceInfo {
  int sms = 0;
  bool smem_set = false;
};

cudaError_t device_info(DeviceInfo** out) {
  static std::mutex mu;
  static DeviceInfo info[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  DeviceInfo& d = info[dev];
  if (!d.smem_set) {
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    for (auto k : {score_kernel<false>, score_kernel<true>}) {
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kScoreSmem);
      if (e != cudaSuccess) return e;
    }
    for (auto k : {topk_kernel<false>, topk_kernel<true>}) {
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTopkSmem);
      if (e != cudaSuccess) return e;
    }
    d.smem_set = true;
  }
  *out = &d;
  return cudaSuccess;
}

}  // namespace

#ifdef QSA_WAIT_TEST
namespace {
int64_t g_test_withhold = -1;
}  // namespace
#endif

cudaError_t launch_select(const SelectParams& p, cudaStream_t stream) {
  if (p.R == 0) return cudaSuccess;
  DeviceInfo* di = nullptr;
  cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return e;
  CUtensorMap map;
  e = encode_cmp_map(p, &map);
  if (e != cudaSuccess) return e;
  // rows in chunks of kMaxRows (the score kernel keeps per-row tables in smem)
  for (int r0 = 0; r0 < p.R; r0 += kMaxRows) {
    SelectParams c = p;
    c.R = p.R - r0 < kMaxRows ? p.R - r0 : kMaxRows;
    c.q_sel = p.q_sel + (int64_t)r0 * kSelHeads * kSelDim;
    c.t2r = p.t2r + r0;
    c.qpos = p.qpos + r0;
    c.out = p.out + (int64_t)r0 * p.out_stride0;
    c.scores = p.scores + (int64_t)r0 * p.vcap;
    c.umax = p.umax + (int64_t)r0 * (p.vcap / kUnitKeys);
#ifdef QSA_WAIT_TEST
    c.test_withhold = r0 == 0 ? g_test_withhold : -1;
#endif
    const int64_t items = (int64_t)c.R * c.pt_cols;
    const int grid = (int)(items < di->sms ? items : di->sms);
    if (c.key_fp8)
      score_kernel<true><<<grid, kScoreThreads, kScoreSmem, stream>>>(c, map);
    else
      score_kernel<false><<<grid, kScoreThreads, kScoreSmem, stream>>>(c, map);
    // rows of at most kCandCap blocks (every row, when the page table is
    // that narrow) take all their keys as candidates
    e = c.vcap <= kCandCap
            ? launch_after(topk_kernel<true>, dim3(c.R), dim3(kTopkThreads), kTopkSmem, stream, c)
            : launch_after(topk_kernel<false>, dim3(c.R), dim3(kTopkThreads), kTopkSmem, stream, c);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

cudaError_t launch_select_attend(const SelectParams& p, const AttentionParams& a,
                                 cudaStream_t stream) {
  // the selection's kernels, then the attention's over its output, all on
  // the caller's stream; the top-k is a programmatic dependent of the score
  // kernel, and the attention of batches of up to 32 rows of the top-k
  if (p.R == 0) return cudaSuccess;
  cudaError_t e;
  const int cs = fused_decode_cluster(p.R, p.pt_cols, p.key_fp8 != 0);
  if (cs > 0) {   // a few rows: one kernel, one cluster per row
    CUtensorMap map;
    e = encode_cmp_map(p, &map);
    if (e != cudaSuccess) return e;
#ifdef QSA_WAIT_TEST
    SelectParams pt = p;
    pt.test_withhold = g_test_withhold;
    return launch_fused_decode(pt, a, map, cs, stream);
#else
    return launch_fused_decode(p, a, map, cs, stream);
#endif
  }
  e = launch_select(p, stream);
  if (e != cudaSuccess) return e;
  AttentionParams ac = a;
  ac.idx = p.out;
  ac.idx_stride0 = p.out_stride0;
  ac.width = kOutWidth;
  ac.nsplit = attention_splits(p.R, kOutWidth);
  ac.inputs_early = 1;   // the kernel before it is the top-k, which writes only the indices
  return launch_attention(ac, stream);
}

}  // namespace qsa

#ifdef QSA_WAIT_TEST
// Test build only, declared in no public header: the next selection launches
// leave fill `issue` of the score kernel's CTA 0 without a copy (-1: none).
extern "C" __attribute__((visibility("default"))) void qsa_test_withhold_score_fill(
    int64_t issue) {
  qsa::g_test_withhold = issue;
}
#endif
