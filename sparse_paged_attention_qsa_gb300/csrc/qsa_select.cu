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

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

namespace qsa {
namespace {

// score kernel: persistent, one CTA per SM, warp-specialised
// The ring holds kRingBytes of pages: 6 fp16 pages (32 KiB) or 12 E4M3 pages
// (16 KiB).  KeyCfg gives the per-key-type sizes.
constexpr int kRingBytes = 6 * kCmpPageKeys * kSelDim * 2;   // 192 KiB in flight per SM
constexpr int kMaxStages = 12;
template <bool kFp8>
struct KeyCfg {
  static constexpr int kPageBytes = kCmpPageKeys * kSelDim * (kFp8 ? 1 : 2);
  static constexpr int kStages = kRingBytes / kPageBytes;
  static constexpr int kRowsPerKey = kFp8 ? 1 : 2;            // 128-byte TMA rows per key
};
constexpr int kScoreWarps = 8;                          // consumer warps
constexpr int kScoreThreads = (kScoreWarps + 1) * 32;   // + one producer warp
constexpr int kKeyGroups = kCmpPageKeys / 8;            // groups of 8 keys per page
static_assert(2 * kScoreWarps == kKeyGroups, "each consumer warp takes whole key-group pairs");
constexpr int kMaxRows = 1024;                          // rows per launch (row tables in smem)
// The score kernel also keeps the largest key of each run of 16 blocks (one
// warp step: two groups of 8 keys), so the top-k reads 1/16 of a row first.
constexpr int kUnitKeys = 16;
constexpr int kGroupRows = 8;    // rows of one request scored from one page pass (aligned windows)
// row tables: req, visible blocks; group tables: first row (+ sentinel), pages,
// weighted page prefix (64-bit, + total)
constexpr size_t kTableBytes = (size_t)(4 * kMaxRows + 1) * sizeof(int) +
                               (size_t)(kMaxRows + 1) * sizeof(int64_t);
constexpr size_t kScoreSmem = (size_t)kRingBytes + 1024 + 2 * kMaxStages * 8 +
                              kMaxStages * 16 + kTableBytes;
static_assert(kScoreSmem <= 227 * 1024 - 256, "score kernel shared memory");

constexpr int kTopkThreads = 512;                       // one key per thread in the sort

struct RowSetup {
  int req;
  int64_t V;        // visible blocks (qsa_cache.py rule)
  int64_t tail_end; // inclusive
  bool ok;
};

__device__ __forceinline__ RowSetup row_setup(const SelectParams& p, int r) {
  RowSetup s;
  s.req = p.t2r[r];
  s.ok = s.req >= 0 && s.req < p.num_reqs;
  s.V = 0;
  s.tail_end = -1;
  if (!s.ok) return s;
  const int64_t L = p.seq_lens[s.req];
  const int64_t pos = p.qpos[r];
  int64_t v = min(floor_div(pos + 1, kRatio), floor_div(L, kRatio));
  s.V = v > 0 ? v : 0;
  s.tail_end = pos < L - 1 ? pos : L - 1;
  return s;
}

// acc + a*b with fp16 operands and a binary32 accumulator (one rounding; the
// fp16 x fp16 product is exact in binary32, so this equals the fp32 chain step)
__device__ __forceinline__ float fma_h(uint32_t a2, uint32_t b2, bool hi, float c) {
  float d;
  if (hi)
    asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.f16 %0, a1, b1, %3;\n\t}"
        : "=f"(d) : "r"(a2), "r"(b2), "f"(c));
  else
    asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.f16 %0, a0, b0, %3;\n\t}"
        : "=f"(d) : "r"(a2), "r"(b2), "f"(c));
  return d;
}

// Four E4M3 values (one 32-bit word, byte 0 = lowest dim) -> two fp16 pairs,
// exact: each 16-bit half of the word is one cvt (no masks or shifts).
__device__ __forceinline__ void e4m3x4_to_h(uint32_t v, uint32_t& a, uint32_t& b) {
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, lo;\n\tcvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
      : "=r"(a), "=r"(b)
      : "r"(v));
}

// 16 E4M3 values (one 16-byte chunk) -> 16 fp16 values as two 16-byte words.
__device__ __forceinline__ void e4m3x16_to_h(uint4 c, uint4& lo, uint4& hi) {
  e4m3x4_to_h(c.x, lo.x, lo.y);
  e4m3x4_to_h(c.y, lo.z, lo.w);
  e4m3x4_to_h(c.z, hi.x, hi.y);
  e4m3x4_to_h(c.w, hi.z, hi.w);
}

// Score of one key held as four 32-dim slices by a quad of lanes, reduced in
// the canonical order; returns the ordered key bits(s)+1 on every lane.
// q: this lane's slice of the 4 heads as fp16 pairs (dims 32t+2j, 32t+2j+1);
// kv: the key's slice as 4 x 16 bytes.
__device__ __forceinline__ uint32_t quad_score(const uint32_t (&q)[kSelHeads][16],
                                               const uint4 (&kv)[4], int t) {
  float E[kSelHeads], O[kSelHeads];
#pragma unroll
  for (int h = 0; h < kSelHeads; ++h) E[h] = O[h] = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w[4] = {kv[i].x, kv[i].y, kv[i].z, kv[i].w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
#pragma unroll
      for (int h = 0; h < kSelHeads; ++h) {
        E[h] = fma_h(q[h][4 * i + m], w[m], false, E[h]);   // even dims
        O[h] = fma_h(q[h][4 * i + m], w[m], true, O[h]);    // odd dims
      }
    }
  }
  float P[kSelHeads];
#pragma unroll
  for (int h = 0; h < kSelHeads; ++h) P[h] = __fadd_rn(E[h], O[h]);   // P_t = E_t + O_t
  // reduce-scatter over the quad: lanes t, t^2 (slices 0+2, 1+3), then t^1;
  // lane t ends with head t's d = (P0 + P2) + (P1 + P3)
  const bool hi2 = (t & 2) != 0;
  const float send0 = hi2 ? P[0] : P[2];
  const float send1 = hi2 ? P[1] : P[3];
  const float keep0 = hi2 ? P[2] : P[0];
  const float keep1 = hi2 ? P[3] : P[1];
  const float A0 = __fadd_rn(keep0, __shfl_xor_sync(0xffffffffu, send0, 2));
  const float A1 = __fadd_rn(keep1, __shfl_xor_sync(0xffffffffu, send1, 2));
  const bool hi1 = (t & 1) != 0;
  const float d = __fadd_rn(hi1 ? A1 : A0, __shfl_xor_sync(0xffffffffu, hi1 ? A0 : A1, 1));
  const float rho = d > 0.f ? d : 0.f;
  const float u = __fadd_rn(rho, __shfl_xor_sync(0xffffffffu, rho, 1));
  const float s = __fadd_rn(u, __shfl_xor_sync(0xffffffffu, u, 2));  // (r0+r1)+(r2+r3)
  return __float_as_uint(s) + 1u;
}

// This lane's query slice [32t, 32t+32) of each of the 4 heads, fp16 pairs.
__device__ __forceinline__ void load_query_slice(const __half* qrow, int t,
                                                 uint32_t (&q)[kSelHeads][16]) {
  const uint4* qp = reinterpret_cast<const uint4*>(qrow);
#pragma unroll
  for (int h = 0; h < kSelHeads; ++h) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = __ldg(qp + h * 16 + t * 4 + i);
      q[h][4 * i + 0] = v.x;
      q[h][4 * i + 1] = v.y;
      q[h][4 * i + 2] = v.z;
      q[h][4 * i + 3] = v.w;
    }
  }
}

// Load NG consecutive groups of 8 keys (from group g0) of the staged page:
// this lane's 32-dim slice of key (g0+g)*8 + kslot, as fp16 pairs.  With the
// 128-byte swizzle, lane (key k, slice t) of an fp16 page reads row 2k + t/2,
// 16-byte chunks (4(t&1)+j) XOR (row & 7); of an E4M3 page, row k, chunks
// (2t+j) XOR (k & 7): the 8 lanes of each shared-memory phase hit 8 distinct
// bank groups.
template <bool kFp8, int NG>
__device__ __forceinline__ void load_key_groups(uint32_t stage, int g0, int t, int kslot,
                                                uint4 (&kv)[NG][4]) {
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    const int k = (g0 + g) * 8 + kslot;
    if (kFp8) {
      const uint32_t r = (uint32_t)k;
      const uint32_t rbase = stage + r * 128;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t chunk = (uint32_t)(2 * t + j) ^ (r & 7u);
        const uint4 c = lds128(rbase + chunk * 16);
        e4m3x16_to_h(c, kv[g][2 * j], kv[g][2 * j + 1]);
      }
    } else {
      const uint32_t r = 2 * k + (t >> 1);
      const uint32_t rbase = stage + r * 128;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t chunk = (uint32_t)(4 * (t & 1) + j) ^ (r & 7u);
        kv[g][j] = lds128(rbase + chunk * 16);
      }
    }
  }
}

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

// ---------------------------------------------------------------------------
// top-k: exact selection of the row's 512 largest 32-bit ordered score keys
// ---------------------------------------------------------------------------
//
// One CTA per row.  Keys are bits(score)+1 (bit 31 clear, 0 = no key).
//  1. Candidates.  A row of at most kCandCap blocks takes every key, with
//     its block index, into the candidate list (one load round up to 4096
//     keys); K = min(512, #keys).  A longer row first reads its unit maxima
//     (the largest key of each run of 16 blocks, written by the score
//     kernel; staged in shared memory up to kUnitCap runs): with at least
//     512 nonzero maxima, one 12-bit radix digit over [min, max] gives a
//     lower bound lo of their 512-th largest, which bounds the 512-th
//     largest key from below (512 distinct keys, the maxima, reach it);
//     else lo = 1.  The runs whose maximum reaches lo (about 520 of 2048
//     on a 32768-key row) are read (64 B each) and their keys >= lo are
//     the candidates (about 590).
//  2. Radix select over the candidates' offsets from lo finds T, the K-th
//     largest key, and `need`, how many keys equal to T belong to the top
//     K.  If more than `need` keys equal T, a second select over (2^31-1 -
//     block index) of those ties keeps the `need` smallest block indices
//     (the tie rule).
//  3. The K (key, ~index) pairs are ordered (a bitonic sort of 512 slots),
//     expanded, tail appended.
// Every select takes 12-bit digits of (x - lo) from the top bit of hi - lo
// down, so its first digit already spreads the members over the range they
// span, and stops at the first digit whose bin holds exactly the members
// still needed.  A row whose hit runs or candidates overflow their lists
// falls back to the same select over all of its keys, re-read from the
// workspace.

constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kCandCap = 8192;                          // candidate (key, block) pairs
constexpr int kUnitCap = 4096;                          // unit maxima staged in smem
constexpr int kDigitBits = 12;
constexpr int kBins = 1 << kDigitBits;                  // 4096 histogram bins
constexpr int kBinsPerThread = kBins / kTopkThreads;    // 8

struct TopkShared {
  uint32_t hist[kBins];            // radix histogram; between selects, the hit-unit list
  uint32_t umax[kUnitCap];         // the row's unit maxima (rows of <= 65536 blocks)
  unsigned long long keys[kTopkBlocks];
  uint32_t cand_x[kCandCap];
  uint32_t cand_i[kCandCap];
  uint32_t wsum[kTopkWarps];
  uint32_t wmin[kTopkWarps];
  uint32_t wmax[kTopkWarps];
  uint32_t found_digit, found_above;
  int count;                       // kept pairs in keys[]
  int nhit, ncand;
};
constexpr size_t kTopkSmem = sizeof(TopkShared);

// Score keys are written by another kernel; read them from L2 (not through
// the non-coherent path), 16 bytes at a time.
__device__ __forceinline__ uint4 ld_cg16(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

__device__ __forceinline__ uint32_t u4_at(const uint4& v, int j) {
  return j == 0 ? v.x : (j == 1 ? v.y : (j == 2 ? v.z : v.w));
}

// Suffix scan of the histogram: find the digit d with
// above(d) < need <= above(d) + hist[d]; returns d and above(d).
__device__ __forceinline__ void find_digit(TopkShared& sh, uint32_t need, int tid, int lane,
                                           int warp) {
  // Keys from one score pass always hold such a digit.  If the workspace is
  // not from one pass (a score kernel whose wait gave up), none may: the
  // result is then digit 0 with nothing above, so every index stays in range.
  if (tid == 0) {
    sh.found_digit = 0;
    sh.found_above = 0;
  }
  uint32_t h[kBinsPerThread];
  uint32_t local = 0;
#pragma unroll
  for (int b = 0; b < kBinsPerThread; ++b) {
    h[b] = sh.hist[tid * kBinsPerThread + b];
    local += h[b];
  }
  uint32_t suf = local;                           // inclusive suffix within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_down_sync(0xffffffffu, suf, o);
    if (lane + o < 32) suf += v;
  }
  if (lane == 0) sh.wsum[warp] = suf;
  __syncthreads();
  uint32_t higher = 0;
  for (int w = warp + 1; w < kTopkWarps; ++w) higher += sh.wsum[w];
  uint32_t above = higher + suf - local;          // keys in bins above this thread's
  if (above < need && above + local >= need) {
#pragma unroll
    for (int b = kBinsPerThread - 1; b >= 0; --b) {
      if (above < need && above + h[b] >= need) {
        sh.found_digit = (uint32_t)(tid * kBinsPerThread + b);
        sh.found_above = above;
      }
      above += h[b];
    }
  }
  __syncthreads();
}

// Radix select result.  Exactly `need` of the members equal to T are among
// the k largest and every member above T is; `clean` means that the k
// largest are exactly the members >= T (T may then lie below the k-th
// largest member, at the low end of its digit).
struct Selected {
  uint32_t T, need;
  bool clean;
};

// Members of a select are the nonzero src[c], c in [0, n) -- a row's keys
// or the candidate keys -- or, for a tie select, the items
// equal to T mapped to (2^31-1 - block index), the block index being c, or
// cand_i[c] for candidates.
template <bool kTie, bool kCandIdx>
__device__ __forceinline__ uint32_t item_key(const TopkShared& sh, const uint32_t* src, int64_t c,
                                             uint32_t T) {
  const uint32_t x = src[c];
  if (!kTie) return x;
  return x == T ? 0x7fffffffu - (kCandIdx ? sh.cand_i[c] : (uint32_t)c) : 0u;
}

// Every member lies in [lo, hi].  Digits of (x - lo) are taken kDigitBits at
// a time from the top set bit of hi - lo down.  The select stops as soon as
// the bin of the k-th largest member holds exactly the members still needed
// (then every member >= lo + prefix is in the top k: `clean`), after
// `max_passes` passes (T is then a lower bound of the k-th largest member:
// at least k members are >= T), or at the last digit, where T is exact.
template <bool kTie, bool kCandIdx>
__device__ Selected radix_select(TopkShared& sh, const uint32_t* src, int64_t n, uint32_t k,
                                 uint32_t lo, uint32_t hi, uint32_t T = 0, int max_passes = 3) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int shift = 32 - __clz((hi - lo) | 1u);          // bits still to resolve (>= 1)
  uint32_t prefix = 0, need = k;
  bool clean = false;
#pragma unroll 1
  for (int pass = 0; shift > 0 && pass < max_passes && !clean; ++pass) {
    const int w = shift < kDigitBits ? shift : kDigitBits;
    shift -= w;
    const uint32_t himask = shift + w >= 32 ? 0u : (0xffffffffu << (shift + w));
    const uint32_t dmask = (1u << w) - 1u;
    for (int i = tid; i < kBins; i += kTopkThreads) sh.hist[i] = 0;
    __syncthreads();
    for (int64_t c = tid; c < n; c += kTopkThreads) {
      const uint32_t x = item_key<kTie, kCandIdx>(sh, src, c, T);
      const uint32_t rel = x - lo;
      if (x != 0u && (rel & himask) == prefix) atomicAdd(&sh.hist[(rel >> shift) & dmask], 1u);
    }
    __syncthreads();
    find_digit(sh, need, tid, lane, warp);
    prefix |= sh.found_digit << shift;
    need -= sh.found_above;
    clean = sh.hist[sh.found_digit] == need;
    __syncthreads();
  }
  return Selected{lo + prefix, need, clean};
}

// Warp-wide: the lanes with `take` get consecutive slots from *counter (one
// shared atomic per warp); returns this lane's slot (meaningful where take).
__device__ __forceinline__ int warp_slot(int* counter, bool take, int lane) {
  const unsigned bal = __ballot_sync(0xffffffffu, take);
  int base = 0;
  if (lane == 0 && bal) base = atomicAdd(counter, __popc(bal));
  base = __shfl_sync(0xffffffffu, base, 0);
  return base + __popc(bal & ((1u << lane) - 1u));
}

// Warp-wide: reserve `cnt` consecutive slots of *counter for each lane (one
// shared atomic per warp); returns this lane's first slot.
__device__ __forceinline__ int warp_reserve(int* counter, int cnt, int lane) {
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  int base = 0;
  if (lane == 31 && incl > 0) base = atomicAdd(counter, incl);
  base = __shfl_sync(0xffffffffu, base, 31);
  return base + incl - cnt;
}

// Append (key, ~index) for the lanes with `take`.  Every lane of the warp
// must call this together.
__device__ __forceinline__ void emit_warp(TopkShared& sh, bool take, uint32_t x, int64_t idx,
                                          int lane) {
  const int slot = warp_slot(&sh.count, take, lane);
  // at most 512 keys are taken when the keys come from one score pass; the
  // bound keeps a workspace that does not (after a timeout) inside keys[]
  if (take && slot < kTopkBlocks)
    sh.keys[slot] = ((unsigned long long)x << 32) | (0xffffffffu - (uint32_t)idx);
}

__device__ __forceinline__ unsigned long long shfl_xor_u64(unsigned long long v, int m) {
  const uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)v, m);
  const uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(v >> 32), m);
  return ((unsigned long long)hi << 32) | lo;
}

// Top-k of row r by the CTA's kTopkThreads threads into `sh`.  The CTA
// runs in the top-k kernel, a programmatic dependent of the score kernel,
// and waits for it after the row's setup.  kDense: every row of the launch
// has at most kCandCap blocks (the page table is at most kCandCap / 128
// columns wide), and all of a row's keys are its candidates.  Ends after its
// last write of p.out (no final barrier).
template <bool kDense>
__device__ __forceinline__ void topk_row(const SelectParams& p, int r, TopkShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31;
  const RowSetup rs = row_setup(p, r);
  int32_t* out = p.out + (int64_t)r * p.out_stride0;
  if (!rs.ok) {
    pdl_wait();
    for (int j = tid; j < kOutWidth; j += kTopkThreads) out[j] = -1;
    if (tid == 0) report(p.err, kErrRequest);
    return;
  }
  const int warp = tid >> 5;
  if (tid == 0 && rs.V > p.vcap) report(p.err, kErrCmpPage);
  const int64_t Vs = rs.V < p.vcap ? rs.V : p.vcap;
  const uint32_t* sc = p.scores + (int64_t)r * p.vcap;   // 512-byte aligned (vcap % 128 == 0)
  const int64_t nu = (Vs + kUnitKeys - 1) / kUnitKeys;   // units of 16 blocks
  const uint32_t* ur = p.umax + (int64_t)r * (p.vcap / kUnitKeys);   // 32-byte aligned rows
  const bool u_in_smem = nu <= kUnitCap;
  const uint32_t* usrc = u_in_smem ? sh.umax : ur;
  if (tid == 0) {
    sh.count = 0;
    sh.nhit = 0;
    sh.ncand = 0;
  }
  __syncthreads();
  pdl_wait();      // the score kernel's keys are complete and visible

  // The candidates: a row of at most kCandCap keys takes all of them (one
  // load round); a longer row the keys that reach a lower bound of its
  // 512-th largest, found from the unit maxima.
  uint32_t lo = 1u, M = 0, K = 0;
  int ncand = 0;
  bool fits = true;
  if (kDense) {
    // 1'. every key a candidate (block index = position); the largest key M
    // and the count of keys (nonzero) give K = min(512, keys)
    uint32_t nz = 0;
    {
      const uint4* s4 = reinterpret_cast<const uint4*>(sc);
      const int64_t n4 = (Vs + 3) >> 2;                  // the last vector may pass Vs
      constexpr int kPer = 2;                            // vectors per thread and round
      for (int64_t b = tid; b < n4; b += kPer * kTopkThreads) {   // one round up to 4096 keys
        uint4 v[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int64_t i = b + (int64_t)u * kTopkThreads;
          v[u] = i < n4 ? ld_cg16(s4 + i) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int64_t g0 = 4 * (b + (int64_t)u * kTopkThreads);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (g0 + j < Vs) {
              const uint32_t x = u4_at(v[u], j);
              sh.cand_x[g0 + j] = x;
              sh.cand_i[g0 + j] = (uint32_t)(g0 + j);
              nz += x != 0u;
              M = x > M ? x : M;
            }
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        nz += __shfl_xor_sync(0xffffffffu, nz, o);
        M = max(M, __shfl_xor_sync(0xffffffffu, M, o));
      }
      if (lane == 0) {
        sh.wsum[warp] = nz;
        sh.wmax[warp] = M;
      }
      __syncthreads();
      nz = 0;
      for (int w = 0; w < kTopkWarps; ++w) {
        nz += sh.wsum[w];
        M = max(M, sh.wmax[w]);
      }
    }
    ncand = (int)Vs;
    K = nz < (uint32_t)kTopkBlocks ? nz : (uint32_t)kTopkBlocks;
  } else {
    // 1. unit maxima: how many are nonzero, the smallest nonzero, the largest
    // (M, the row's largest key); staged in shared memory
    uint32_t nz = 0, umin = 0xffffffffu;
    {
      const uint4* u4 = reinterpret_cast<const uint4*>(ur);
      const int64_t nu4 = (nu + 3) >> 2;                   // the last vector may pass nu
      for (int64_t b = tid; b < nu4; b += 2 * kTopkThreads) {
        uint4 v[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int64_t i = b + (int64_t)u * kTopkThreads;
          v[u] = i < nu4 ? ld_cg16(u4 + i) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int64_t g0 = 4 * (b + (int64_t)u * kTopkThreads);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t x = g0 + j < nu ? u4_at(v[u], j) : 0u;
            if (u_in_smem && g0 + j < nu) sh.umax[g0 + j] = x;
            nz += x != 0u;
            umin = x != 0u && x < umin ? x : umin;
            M = x > M ? x : M;
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        nz += __shfl_xor_sync(0xffffffffu, nz, o);
        umin = min(umin, __shfl_xor_sync(0xffffffffu, umin, o));
        M = max(M, __shfl_xor_sync(0xffffffffu, M, o));
      }
      if (lane == 0) {
        sh.wsum[warp] = nz;
        sh.wmin[warp] = umin;
        sh.wmax[warp] = M;
      }
      __syncthreads();
      nz = 0;
      for (int w = 0; w < kTopkWarps; ++w) {
        nz += sh.wsum[w];
        umin = min(umin, sh.wmin[w]);
        M = max(M, sh.wmax[w]);
      }
    }
    // With >= 512 nonzero maxima (>= 512 keys), a lower bound of their 512-th
    // largest -- one digit pass -- bounds the 512-th largest key from below
    const bool many = nz >= (uint32_t)kTopkBlocks;
    lo = many ? radix_select<false, false>(sh, usrc, nu, kTopkBlocks, umin, M, 0u, 1).T : 1u;

    // 2. units whose maximum reaches lo (listed in the histogram space), then
    // their keys >= lo into the candidate list; one shared atomic per warp and
    // step
    uint32_t* hit = sh.hist;
    for (int64_t base = 0; base < nu; base += 8 * kTopkThreads) {
      uint32_t mask = 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t c = base + (int64_t)u * kTopkThreads + tid;
        mask |= (uint32_t)(c < nu && usrc[c] >= lo) << u;   // lo >= 1: nonzero maxima only
      }
      int slot = warp_reserve(&sh.nhit, __popc(mask), lane);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (mask >> u & 1u) {
          if (slot < kBins) hit[slot] = (uint32_t)(base + (int64_t)u * kTopkThreads + tid);
          ++slot;
        }
      }
    }
    __syncthreads();
    const int nhit = sh.nhit;
    if (nhit <= kBins) {
      for (int base = 0; base < nhit; base += kTopkThreads) {
        const int h = base + tid;
        const int64_t g = h < nhit ? (int64_t)hit[h] : -1;
        uint4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          v[j] = g >= 0 ? ld_cg16(sc + kUnitKeys * g + 4 * j) : make_uint4(0, 0, 0, 0);
        uint32_t mask = 0;                                   // bit j: key j of the unit
#pragma unroll
        for (int j = 0; j < kUnitKeys; ++j) {
          const uint32_t x = g >= 0 && kUnitKeys * g + j < Vs ? u4_at(v[j >> 2], j & 3) : 0u;
          mask |= (uint32_t)(x >= lo) << j;
        }
        int slot = warp_reserve(&sh.ncand, __popc(mask), lane);
#pragma unroll
        for (int j = 0; j < kUnitKeys; ++j) {
          if (mask >> j & 1u) {
            if (slot < kCandCap) {
              sh.cand_x[slot] = u4_at(v[j >> 2], j & 3);
              sh.cand_i[slot] = (uint32_t)(kUnitKeys * g + j);
            }
            ++slot;
          }
        }
      }
    }
    __syncthreads();
    ncand = sh.ncand;
    fits = nhit <= kBins && ncand <= kCandCap;
    // K = min(512, #keys): with >= 512 nonzero maxima there are >= 512 keys;
    // otherwise every key is a candidate (fewer than 512 units hold keys)
    K = many ? (uint32_t)kTopkBlocks
             : (ncand < kTopkBlocks ? (uint32_t)ncand : (uint32_t)kTopkBlocks);
  }
  const uint32_t tie_lo = 0x80000000u - (uint32_t)Vs;      // 2^31-1 - (Vs-1)

  if (K > 0) {
    if (fits) {
      // 3. radix select over the candidates
      const Selected sel = radix_select<false, true>(sh, sh.cand_x, ncand, K, lo, M);
      const uint32_t T = sel.T;
      for (int base = 0; base < ncand; base += kTopkThreads) {
        const int c = base + tid;
        const uint32_t x = c < ncand ? sh.cand_x[c] : 0u;
        emit_warp(sh, x != 0u && (sel.clean ? x >= T : x > T), x,
                  c < ncand ? sh.cand_i[c] : 0u, lane);
      }
      if (!sel.clean) {   // T exact, surplus ties: keep the smallest block indices
        const Selected si =
            radix_select<true, true>(sh, sh.cand_x, ncand, sel.need, tie_lo, 0x7fffffffu, T);
        for (int base = 0; base < ncand; base += kTopkThreads) {
          const int c = base + tid;
          const bool take =
              c < ncand && sh.cand_x[c] == T && 0x7fffffffu - sh.cand_i[c] >= si.T;
          emit_warp(sh, take, T, c < ncand ? sh.cand_i[c] : 0u, lane);
        }
      }
    } else {
      // fallback (many holds here, so K = 512): select over all keys of the row
      const Selected sel = radix_select<false, false>(sh, sc, Vs, K, 1u, M);
      const uint32_t T = sel.T;
      for (int64_t b0 = 0; b0 < Vs; b0 += kTopkThreads) {
        const int64_t i = b0 + tid;
        const uint32_t x = i < Vs ? sc[i] : 0u;
        emit_warp(sh, x != 0u && (sel.clean ? x >= T : x > T), x, i, lane);
      }
      if (!sel.clean) {
        const Selected si =
            radix_select<true, false>(sh, sc, Vs, sel.need, tie_lo, 0x7fffffffu, T);
        for (int64_t b0 = 0; b0 < Vs; b0 += kTopkThreads) {
          const int64_t i = b0 + tid;
          const bool take = i < Vs && sc[i] == T && 0x7fffffffu - (uint32_t)i >= si.T;
          emit_warp(sh, take, T, i, lane);
        }
      }
    }
    __syncthreads();
  }

  // 4. order: a bitonic sort of the 512 slots (kept pairs, then zeros),
  // descending; partners closer than a warp exchange by shuffles, the others
  // through shared memory (two buffers, one barrier per step).  Kept keys
  // are distinct and nonzero, so slot i ends with the i-th largest.
  unsigned long long a = tid < (int)K ? sh.keys[tid] : 0ull;
  {
    unsigned long long* const buf0 = sh.keys;
    unsigned long long* const buf1 = reinterpret_cast<unsigned long long*>(sh.cand_x);
    int nb = 0;
    __syncthreads();                     // every read of keys[] above is done
#pragma unroll
    for (int k = 2; k <= kTopkThreads; k <<= 1) {
#pragma unroll
      for (int j = k >> 1; j > 0; j >>= 1) {
        unsigned long long b;
        if (j >= 32) {
          unsigned long long* const bf = nb ? buf1 : buf0;
          bf[tid] = a;
          __syncthreads();
          b = bf[tid ^ j];
          nb ^= 1;
        } else {
          b = shfl_xor_u64(a, j);
        }
        const bool desc = (tid & k) == 0;
        const bool lower = (tid & j) == 0;
        const unsigned long long hi = a > b ? a : b, lo = a > b ? b : a;
        a = (desc == lower) ? hi : lo;
      }
    }
  }
  if (tid < (int)K) {   // expand the kept block at its position
    const int32_t b = (int32_t)(0xffffffffu - (uint32_t)(a & 0xffffffffull));
    const int32_t tok = b * kRatio;
    out[4 * tid + 0] = tok;
    out[4 * tid + 1] = tok + 1;
    out[4 * tid + 2] = tok + 2;
    out[4 * tid + 3] = tok + 3;
  }
  // then the tail, then -1
  const int64_t tail0 = rs.V * kRatio;
  const int64_t tail_len = rs.tail_end >= tail0 ? rs.tail_end - tail0 + 1 : 0;
  for (int j = 4 * (int)K + tid; j < kOutWidth; j += kTopkThreads) {
    const int64_t tt = j - 4 * (int64_t)K;
    out[j] = tt < tail_len ? (int32_t)(tail0 + tt) : -1;
  }
}

template <bool kDense>
__global__ void __launch_bounds__(kTopkThreads, 2)
topk_kernel(const SelectParams p) {
  extern __shared__ __align__(16) unsigned char topk_smem[];
  TopkShared& sh = *reinterpret_cast<TopkShared*>(topk_smem);
  pdl_trigger();   // a dependent (the attention kernel) may be scheduled early (it waits)
  topk_row<kDense>(p, blockIdx.x, sh);
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
  cudaError_t e = launch_select(p, stream);
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
