// qsa_indexer.cu -- the weighted paged MQA indexer and its per-row top-k,
// declared in include/qsa_indexer.h.
//
// "[XPU] Enable multiple key kernels for sparse attention" (vLLM PR 37888
// report) names the DeepSeek-V3.2 indexer's decode kernels,
// fp8_paged_mqa_logits and top_k_per_row_decode, and prints their
// signatures; the arithmetic restated here is the plainest reading of them
// (see the header): logit = key scale * sum_h w_h * ReLU(q_h . k).
//
// logits_kernel  persistent, one CTA per SM, warp-specialised:
//   warp 0  producer: per 128-token tile of one request, each lane loads one
//           of the tile's cache blocks -- a TMA of its 128-byte value rows
//           (128-byte swizzle) and a bulk copy of its scales -- into a ring
//           of shared-memory stages; the warp arms up to four tiles per
//           iteration from a warp-wide chunk of block-table entries; the
//           request's query rows (all heads of its next_n tokens, same
//           swizzle) and head weights go to one of two query slots once per
//           request the CTA works on;
//   warps 1, 18  MMA issuers, alternate tiles each: one lane issues four
//           tcgen05.mma kind::f8f6f4 (M = 128 tokens, N = next_n x heads,
//           K = 32 each) per tile into a TMEM accumulator of its own
//           (tile n uses accumulator n % 4, or n % 2 when N = 256) once that
//           accumulator's previous tile is consumed, and commits to the
//           accumulator's barrier and to the stage's: a stage is refilled
//           as soon as its MMAs have read the values and the epilogue warps
//           have read the scales and descriptor; warp 1 owns the TMEM
//           allocation;
//   warps 2-17  epilogue in four groups of four warps (one warp per TMEM
//           lane quarter); group g takes the tiles of accumulator g, so no
//           warp waits on a barrier phase ahead of its predecessor: each
//           thread owns one token (its TMEM lane), reads its accumulator row
//           with one tcgen05.ld per 64 columns, forms sum_h w_h * ReLU(d_h)
//           for every query row in fp32 (packed pairs), scales, and writes
//           the logits (consecutive threads, consecutive columns).
// fill_kernel    writes -inf to each row's columns [L_r, max_model_len).
// topk_rows_kernel  one CTA of 512 threads per row: a threshold from 8192
//           sampled logits, one float4 pass keeping the logits at or above
//           it (about 4096 of a long row) in shared memory, an exact radix
//           select of the k-th largest there (digits spread over the
//           candidates' range), emission of the larger ones and of the
//           first ties in column order, bitonic sort of the k (logit,
//           column) pairs.  A row whose candidates do not fit (or are too
//           few) is selected with radix passes over the row itself.
// Every mbarrier wait gives up after 1 s (QSA_DERR_TIMEOUT), drains what the
// CTA has in flight, frees its TMEM and returns.
#include "qsa.h"
#include "qsa_indexer.h"
#include "qsa_device.cuh"
#include "qsa_host.h"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

namespace qsa {
namespace {

constexpr int kDim = QSA_IDX_HEAD_DIM;      // 128 E4M3 values per query head / key
constexpr int kTile = 128;                  // tokens per tile (MMA M)
constexpr int kMaxN = 256;                  // next_n x heads (MMA N)
#ifndef QSA_IDX_EPI_GROUPS
#define QSA_IDX_EPI_GROUPS 4
#endif
// Epilogue groups taking tiles in turn.  A group always owns the same
// accumulators (tile n uses accumulator n % NA and group n % G with G
// dividing NA), so no warp can wait on an accumulator's barrier phase before
// the previous phase has completed.
constexpr int kEpiGroups = QSA_IDX_EPI_GROUPS;
constexpr int kEpiWarps = 4 * kEpiGroups;       // one warp per TMEM lane quarter per group
#ifndef QSA_IDX_ISSUERS
#define QSA_IDX_ISSUERS 2
#endif
constexpr int kIssuers = QSA_IDX_ISSUERS;       // MMA issuer warps: 1 and 2+kEpiWarps.. (lane 0 each)
constexpr int kLogitThreads = (1 + kIssuers + kEpiWarps) * 32;
constexpr int kLogitRegs = kEpiGroups > 3 ? (kIssuers > 2 ? 80 : 96) : (kEpiGroups > 2 ? 128 : 168);
constexpr int kHeadChunk = kLogitRegs < 96 ? 32 : 64;   // TMEM columns per load
constexpr int kMaxBatch = 1024;             // requests per launch (tables in smem)
constexpr int kMaxStages = 12;
constexpr int kMaxAcc = 4;                  // TMEM accumulators (512 columns / N, at most 4)
constexpr int kProdTiles = 4;               // tiles the producer arms per iteration
constexpr size_t kLogitSmem = 220 * 1024;
constexpr size_t kTablesBytes = (size_t)(kMaxBatch + 1) * 8 + (size_t)kMaxBatch * 4;
constexpr size_t kMiscBytes = 1024;         // barriers + stage descriptors

constexpr uint32_t kErrTimeoutBit = 8u;
constexpr uint32_t kErrBlockBit = QSA_DERR_IDX_BLOCK;

struct LogitParams {
  const uint8_t* kv;          // cache base [num_blocks, bs*132]
  const float* w;             // this launch's first row's weights [rows, H]
  const int32_t* ctx;         // this launch's requests' context lengths
  const int32_t* bt;          // this launch's requests' block-table rows
  int64_t num_blocks, bt_cols, bt_s0;
  float* logits;              // this launch's first row
  int64_t ld, max_len;
  uint32_t* err;
  int bs, H, next_n, N;
  int batch;                  // requests in this launch
  int qrow0;                  // query-map row of this launch's first request (b0 * N)
  int stage_bytes, stages;    // stage: tile values (16 KiB) + scales (512 B)
  int qslot_bytes;            // query slot: N*128 query bytes + N*4 weights
  int nacc;                   // TMEM accumulators of N columns
  int bs_log2;                // log2(bs)
  uint32_t tmem_cols;
};

struct TileDesc {
  int b;             // request within the launch; -1: no more work
  int tile;          // tile index within the request
  uint32_t missing;  // bit c: block c of the tile had no valid cache block
  uint32_t qinfo;    // bit 0: query slot, bit 1: its phase, bit 2: the
                     // request's last tile in this CTA (frees the slot)
};

// --- PTX helpers (the mbarrier, TMA and bulk-copy ones are in qsa_device.cuh) ---

// K-major operand, rows of 128 bytes, 128-byte swizzle, 8-row atoms 1024 B apart
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       int accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// NC accumulator columns of this thread's TMEM lane in one load; the wait is
// in the same asm statement, so no use of the outputs can precede it.
template <int NC>
__device__ __forceinline__ void tc_ld(uint32_t taddr, uint32_t (&r)[NC]);
template <>
__device__ __forceinline__ void tc_ld<16>(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
template <>
__device__ __forceinline__ void tc_ld<32>(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
template <>
__device__ __forceinline__ void tc_ld<64>(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
}

// sum over the NC columns from c0 of w[c] * ReLU(d[c]) for this thread's TMEM
// lane (taddr addresses column 0 of its accumulator): one TMEM load, then
// four fp32 chains (packed in pairs)
template <int NC>
__device__ __forceinline__ float head_sum_n(uint32_t taddr, const float* w, int c0) {
  uint32_t r[NC];
  tc_ld<NC>(taddr + (uint32_t)c0, r);
  const float4* w4 = reinterpret_cast<const float4*>(w + c0);
  float2 lo = make_float2(0.f, 0.f), hi = make_float2(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < NC; k += 4) {
    const float4 ww = w4[k / 4];
    lo = ffma2(make_float2(ww.x, ww.y),
               make_float2(fmaxf(__uint_as_float(r[k + 0]), 0.f),
                           fmaxf(__uint_as_float(r[k + 1]), 0.f)), lo);
    hi = ffma2(make_float2(ww.z, ww.w),
               make_float2(fmaxf(__uint_as_float(r[k + 2]), 0.f),
                           fmaxf(__uint_as_float(r[k + 3]), 0.f)), hi);
  }
  return (lo.x + lo.y) + (hi.x + hi.y);
}

// columns [c0, c0 + nc), nc in {16, 32, kHeadChunk}
__device__ __forceinline__ float head_sum(uint32_t taddr, const float* w, int c0, int nc) {
  switch (nc) {
    case 16: return head_sum_n<16>(taddr, w, c0);
    case 32: return head_sum_n<32>(taddr, w, c0);
    default: return head_sum_n<kHeadChunk>(taddr, w, c0);
  }
}

__device__ __forceinline__ int64_t row_len(int64_t ctx, int next_n, int j, int64_t max_len) {
  int64_t L = ctx - next_n + j + 1;
  L = L < max_len ? L : max_len;
  return L > 0 ? L : 0;
}

// --- logits ------------------------------------------------------------------

// up to 5 warps share an SM sub-partition's 16K registers: cap the registers
// so they fit
__global__ void __maxnreg__(kLogitRegs)
logits_kernel(const LogitParams p, const __grid_constant__ CUtensorMap kmap,
              const __grid_constant__ CUtensorMap qmap) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int64_t s_end_tile;                          // first tile index past the range
  __shared__ int64_t s_part[kLogitThreads];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  const uint32_t base = raw + pad;
  unsigned char* gbase = smem_raw + pad;
  const int S = p.stages;
  const int N = p.N;
  // layout: S stages [values 16 KiB | scales 512 B], two query slots
  // [query rows N*128 | weights N*4], barriers + descriptors, tables
  const uint32_t qslots = (uint32_t)(S * p.stage_bytes);
  const uint32_t misc_off = qslots + 2u * (uint32_t)p.qslot_bytes;
  const uint32_t misc = base + misc_off;
  const uint32_t bar_full = misc, bar_empty = misc + 8 * kMaxStages;
  const uint32_t bar_accf = misc + 16 * kMaxStages, bar_acce = bar_accf + 8 * kMaxAcc;
  const uint32_t bar_qfull = bar_acce + 8 * kMaxAcc, bar_qempty = bar_qfull + 16;
  const int NA = p.nacc;                                  // TMEM accumulators
  TileDesc* desc = reinterpret_cast<TileDesc*>(gbase + misc_off + 16 * kMaxStages + 16 * kMaxAcc + 32);
  int64_t* pre = reinterpret_cast<int64_t*>(gbase + misc_off + kMiscBytes);
  int32_t* ctxc = reinterpret_cast<int32_t*>(pre + kMaxBatch + 1);
  const uint32_t scOff = kTile * kDim;                    // scales within a stage
  const uint32_t wOff = (uint32_t)N * kDim;               // weights within a query slot

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      // the tile's MMAs done reading the values (tcgen05.commit) + the four
      // epilogue warps done reading the scales and the descriptor
      mbar_init(bar_empty + 8 * s, 1 + 4);
    }
    for (int a = 0; a < kMaxAcc; ++a) {
      mbar_init(bar_accf + 8 * a, 1);
      mbar_init(bar_acce + 8 * a, 4);     // the four warps of the group that had the tile
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar_qfull + 8 * k, 1);
      mbar_init(bar_qempty + 8 * k, 1 + 4);
    }
    s_abort = 0;
    s_end_tile = INT64_MAX;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    const uint32_t slot = (uint32_t)__cvta_generic_to_shared(&s_tmem);
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                 "r"(p.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // prologue: tiles per request and their prefix sum
  for (int b = tid; b < p.batch; b += kLogitThreads) {
    int64_t c = p.ctx[b];
    c = c < p.max_len ? c : p.max_len;
    ctxc[b] = (int32_t)(c > 0 ? c : 0);
  }
  __syncthreads();
  {
    const int per = (p.batch + kLogitThreads - 1) / kLogitThreads;
    const int lo = tid * per, hi = min(p.batch, lo + per);
    int64_t sum = 0;
    for (int b = lo; b < hi; ++b) sum += (ctxc[b] + kTile - 1) / kTile;
    s_part[tid] = sum;
    __syncthreads();
    if (tid == 0) {
      int64_t run = 0;
      for (int i = 0; i < kLogitThreads; ++i) {
        const int64_t v = s_part[i];
        s_part[i] = run;
        run += v;
      }
      pre[p.batch] = run;
    }
    __syncthreads();
    int64_t run = s_part[tid];
    for (int b = lo; b < hi; ++b) {
      pre[b] = run;
      run += (ctxc[b] + kTile - 1) / kTile;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int64_t W = pre[p.batch];
  const int64_t w_begin = W * blockIdx.x / gridDim.x;
  const int64_t w_end = W * (blockIdx.x + 1) / gridDim.x;
  volatile int* abort_flag = &s_abort;
  volatile int64_t* end_tile = &s_end_tile;
  int64_t issued = 0;    // producer: stages armed
  int64_t last_issued = -1;  // MMA issuer: its last tile
  int segs = 0;          // producer: query slots loaded

  if (warp == 0) {
    // ---------------- producer (whole warp) ----------------
    const int bpt = kTile / p.bs;                     // blocks per tile
    const auto tiles_of = [&](int bb) { return (int64_t)(ctxc[bb] + kTile - 1) / kTile; };
    int b = 0;
    int64_t i = 0, w = w_begin;
    if (w_begin < w_end) {
      int lo = 0, hi = p.batch - 1;                   // last request with pre <= w_begin
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= w_begin) lo = mid; else hi = mid - 1;
      }
      b = lo;
      i = w_begin - pre[b];
      while (i >= tiles_of(b)) {
        ++b;
        i = 0;
      }
    }
    // up to kProdTiles tiles of one request per iteration; lane = t*bpt + c
    // handles block c of tile t: it waits for that tile's stage, and the
    // lanes issue their TMA and scale copies side by side
    const int bpt_log2 = 7 - p.bs_log2;
    const int max_t = min(kProdTiles, 32 >> bpt_log2);
    const int t_lane = lane >> bpt_log2, c_lane = lane & (bpt - 1);
    // 32 consecutive block-table entries of one request, one per lane, read
    // in one coalesced load and handed to the tiles by shuffles
    int chunk_b = -1;
    int64_t chunk_col0 = 0;
    int32_t chunk_id = -1;
    int cur_b = -1, slot = 0;
    int s = 0, round = 0;                             // ring position of the next stage
    for (;;) {
      const int stop = __shfl_sync(0xffffffffu, *abort_flag, 0);
      if (stop) break;
      if (w >= w_end) {                 // range done: an end marker in the next stage
        bool ok = round == 0 || mbar_wait_sleep(bar_empty + 8 * s, (uint32_t)((round - 1) & 1));
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          if (lane == 0) {
            *abort_flag = 1;
            report(p.err, kErrTimeoutBit);
          }
          break;
        }
        if (lane == 0) {
          *end_tile = issued;           // the first tile index past the range
          desc[s].b = -1;
          mbar_arrive(bar_full + 8 * s);
        }
        ++issued;
        break;
      }
      if (b != cur_b) {                 // a new request: its query rows into the next slot
        slot = segs & 1;
        bool ok = segs < 2 || mbar_wait_sleep(bar_qempty + 8 * slot, (uint32_t)(((segs >> 1) - 1) & 1));
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          if (lane == 0) {
            *abort_flag = 1;
            report(p.err, kErrTimeoutBit);
          }
          break;
        }
        if (lane == 0) {
          const uint32_t qf = bar_qfull + 8 * slot;
          const uint32_t qs = base + qslots + (uint32_t)(slot * p.qslot_bytes);
          mbar_expect_tx(qf, (uint32_t)N * kDim + (uint32_t)N * 4);
          tma_load_2d(qs, &qmap, 0, p.qrow0 + b * N, qf);
          bulk_load(qs + wOff, p.w + (int64_t)b * N, (uint32_t)N * 4, qf);
        }
        cur_b = b;
        ++segs;
      }
      const int64_t tiles_b = tiles_of(b);
      const int64_t left = min(tiles_b - i, w_end - w);
      const int T = (int)(left < max_t ? left : max_t);
      const bool active = t_lane < T;
      int st = s + t_lane, rd = round;
      if (st >= S) {
        st -= S;
        ++rd;
      }
      bool ok = !active || rd == 0 || mbar_wait_sleep(bar_empty + 8 * st, (uint32_t)((rd - 1) & 1));
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) {
          *abort_flag = 1;
          report(p.err, kErrTimeoutBit);
        }
        break;
      }
      const int64_t col0 = i * bpt;     // block-table columns [col0, col0 + T*bpt)
      if (b != chunk_b || col0 < chunk_col0 || col0 + T * bpt > chunk_col0 + 32) {
        chunk_b = b;
        chunk_col0 = col0;
        const int64_t col = col0 + lane;
        chunk_id = col < p.bt_cols ? __ldg(p.bt + (int64_t)b * p.bt_s0 + col) : -1;
      }
      const int32_t id = __shfl_sync(0xffffffffu, chunk_id, (int)(col0 - chunk_col0) + lane);
      const int64_t tv = ctxc[b] - (i + t_lane) * kTile;     // tokens left from tile t_lane
      const int nblk = active ? (int)(((tv < kTile ? tv : kTile) + p.bs - 1) >> p.bs_log2) : 0;
      const bool inblk = c_lane < nblk;
      const bool valid = inblk && id >= 0 && id < p.num_blocks;
      const bool miss = inblk && !valid;
      const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
      const uint32_t mmask = __ballot_sync(0xffffffffu, miss);
      const uint32_t full = bar_full + 8 * st;
      if (active && c_lane == 0) {      // the tile's lead lane: descriptor and byte count
        const uint32_t tmask = bpt == 32 ? 0xffffffffu : (1u << bpt) - 1u;
        const uint32_t vt = (vmask >> (t_lane * bpt)) & tmask;
        const uint32_t mt = (mmask >> (t_lane * bpt)) & tmask;
        const bool last = i + t_lane + 1 >= tiles_b || w + t_lane + 1 >= w_end;
        desc[st].b = b;
        desc[st].tile = (int)(i + t_lane);
        desc[st].missing = mt;
        desc[st].qinfo = (uint32_t)slot | ((uint32_t)(((segs - 1) >> 1) & 1) << 1) |
                         ((uint32_t)last << 2);
        mbar_expect_tx(full, (uint32_t)__popc(vt) * (uint32_t)p.bs * (kDim + 4));
        if (mt) report(p.err, kErrBlockBit);
      }
      __syncwarp();
      if (valid) {
        const uint32_t sb = base + (uint32_t)(st * p.stage_bytes);
        tma_load_3d(sb + (uint32_t)(c_lane * p.bs * kDim), &kmap, 0, 0, id, full);
        bulk_load(sb + scOff + (uint32_t)(c_lane * p.bs * 4),
                  p.kv + (int64_t)id * p.bs * (kDim + 4) + (int64_t)p.bs * kDim,
                  (uint32_t)p.bs * 4, full);
      }
      issued += T;
      w += T;
      i += T;
      s += T;
      if (s >= S) {
        s -= S;
        ++round;
      }
      while (w < w_end && i >= tiles_of(b)) {
        ++b;
        i = 0;
      }
    }
  } else if (warp == 1 || warp >= 2 + kEpiWarps) {
    // ---------------- MMA issuers ----------------
    // two issuers take alternate tiles (issuer g: tiles g, g + 2, ...), each
    // into its own accumulators (n % NA has the parity of n) for epilogue
    // group g: two independent MMA -> epilogue pipelines behind one producer
    const int g = warp == 1 ? 0 : warp - (1 + kEpiWarps);   // issuer index
    const int I = kIssuers < NA ? kIssuers : NA;            // active issuers (divides NA)
    if (lane == 0 && g < I) {
      const uint32_t idesc = (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(kTile >> 4) << 24);
      int s = g, round = 0, a = g, around = 0;          // ring / accumulator position of tile n
      uint32_t seen_q = 0xffffffffu;                    // query slot and phase last waited for
      for (int64_t n = g;; n += I) {
        // accumulator a free again: the epilogue is done with the tile that
        // used it
        if (around > 0) {
          if (!mbar_wait_sleep(bar_acce + 8 * a, (uint32_t)((around - 1) & 1))) {
            *abort_flag = 1;
            report(p.err, kErrTimeoutBit);
            break;
          }
        }
        // tile n's data, or the producer's end marker covering tile n
        int state = mbar_test_wait(bar_full + 8 * s, (uint32_t)(round & 1)) ? 1 : 0;
        const uint64_t t0 = global_ns();
        while (state == 0) {
          if (mbar_try_wait_sleep(bar_full + 8 * s, (uint32_t)(round & 1), 1000u)) state = 1;
          else if (n >= *end_tile || *abort_flag) state = 2;
          else if (global_ns() - t0 > kWaitLimitNs) state = 3;
        }
        if (state == 3) {
          *abort_flag = 1;
          report(p.err, kErrTimeoutBit);
          break;
        }
        if (state == 2 || *abort_flag) break;
        const TileDesc d = desc[s];
        if (d.b < 0) break;                             // the end marker's stage
        const int qs = (int)(d.qinfo & 1u);
        if ((d.qinfo & 3u) != seen_q) {         // a new query slot: wait for its rows
          if (!mbar_wait_sleep(bar_qfull + 8 * qs, (d.qinfo >> 1) & 1u)) {
            *abort_flag = 1;
            report(p.err, kErrTimeoutBit);
            break;
          }
          seen_q = d.qinfo & 3u;
        }
        tc_fence_after();
        const uint32_t st = base + (uint32_t)(s * p.stage_bytes);
        const uint64_t da = smem_desc(st);
        const uint64_t db = smem_desc(base + qslots + (uint32_t)(qs * p.qslot_bytes));
        const uint32_t dt = tmem + (uint32_t)(a * N);
#pragma unroll
        for (int k = 0; k < kDim / 32; ++k) tc_mma(dt, da + 2 * k, db + 2 * k, idesc, k);
        tc_commit(bar_accf + 8 * a);
        tc_commit(bar_empty + 8 * s);           // the values may be refilled once read
        if (d.qinfo & 4u) tc_commit(bar_qempty + 8 * qs);
        last_issued = n;
        s += I;
        if (s >= S) {
          s -= S;
          ++round;
        }
        a += I;
        if (a >= NA) {
          a -= NA;
          ++around;
        }
      }
    }
  } else {
    // ---------------- epilogue (warps 2..9) ----------------
    // two groups of four warps (one per TMEM lane quarter) take alternate
    // tiles, so two tiles' waits, TMEM loads and stores overlap; each warp
    // forms every query row of its tile for its 32 tokens
    const int quarter = warp & 3;              // TMEM lanes this warp may read
    const int group = (warp - 2) >> 2;         // tiles group, group + G, ...
    const int row = quarter * 32 + lane;       // token within the tile
    const int H = p.H;
    const int G = kEpiGroups < NA ? kEpiGroups : NA;   // active groups (divides NA)
    int s = group, round = 0, a = group, around = 0;   // position of tile n
    uint32_t seen_q = 0xffffffffu;                     // query slot and phase last waited for
    for (int64_t n = group; group < G; n += G) {
      // wait for tile n's accumulator, or for the end marker to cover tile n
      // (only the group holding the end tile is woken through the barrier)
      int state = 0;
      const uint64_t t0 = global_ns();
      if (mbar_test_wait(bar_accf + 8 * a, (uint32_t)(around & 1))) state = 1;
      while (state == 0) {
        if (mbar_try_wait_sleep(bar_accf + 8 * a, (uint32_t)(around & 1), 1000u)) state = 1;
        else if (n >= *end_tile || *abort_flag) state = 2;
        else if (global_ns() - t0 > kWaitLimitNs) state = 3;
      }
      if (state == 3) {
        *abort_flag = 1;
        report(p.err, kErrTimeoutBit);
        break;
      }
      if (n >= *end_tile || *abort_flag) break;
      // the stage's full barrier has completed for this tile (its refill
      // waits for this group's four warps, below): waiting on it again makes
      // the producer's descriptor and the copied scales visible here
      if (!mbar_wait_sleep(bar_full + 8 * s, (uint32_t)(round & 1))) {
        *abort_flag = 1;
        report(p.err, kErrTimeoutBit);
        break;
      }
      const TileDesc d = desc[s];
      const int qs = (int)(d.qinfo & 1u);
      if ((d.qinfo & 3u) != seen_q) {            // a new query slot: its weights visible
        if (!mbar_wait_sleep(bar_qfull + 8 * qs, (d.qinfo >> 1) & 1u)) {
          *abort_flag = 1;
          report(p.err, kErrTimeoutBit);
          break;
        }
        seen_q = d.qinfo & 3u;
      }
      tc_fence_after();
      const unsigned char* st = gbase + (size_t)s * p.stage_bytes;
      const float scale = reinterpret_cast<const float*>(st + scOff)[row];
      const float* wts =
          reinterpret_cast<const float*>(gbase + qslots + (size_t)qs * p.qslot_bytes + wOff);
      const bool missing = (d.missing >> (row >> p.bs_log2)) & 1u;
      const int64_t t = (int64_t)d.tile * kTile + row;
      __syncwarp();                              // every lane has its scale and the descriptor
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);   // the stage may be refilled
      const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(a * N);
      float out[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (j < p.next_n) {
          float acc = 0.f;
          for (int c = 0; c < H; c += kHeadChunk)
            acc += head_sum(taddr, wts, j * H + c, H < kHeadChunk ? H : kHeadChunk);
          out[j] = scale * acc;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar_acce + 8 * a);
        if (d.qinfo & 4u) mbar_arrive(bar_qempty + 8 * qs);
      }
      const int64_t cb = ctxc[d.b];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (j < p.next_n && t < row_len(cb, p.next_n, j, p.max_len))
          p.logits[((int64_t)d.b * p.next_n + j) * p.ld + t] = missing ? -INFINITY : out[j];
      }
      s += G;
      if (s >= S) {
        s -= S;
        ++round;
      }
      a += G;
      if (a >= NA) {
        a -= NA;
        ++around;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // let this CTA's copies and MMAs finish before the memory and TMEM go away
    if (warp == 0 && lane == 0) {
      const int64_t first = issued > S ? issued - S : 0;
      for (int64_t m = first; m < issued; ++m)
        mbar_wait_sleep(bar_full + 8 * (int)(m % S), (uint32_t)((m / S) & 1));
      for (int g = segs > 2 ? segs - 2 : 0; g < segs; ++g)
        mbar_wait_sleep(bar_qfull + 8 * (g & 1), (uint32_t)((g >> 1) & 1));
    }
    if ((warp == 1 || warp >= 2 + kEpiWarps) && lane == 0 && last_issued >= 0) {
      const int64_t m = last_issued;
      mbar_wait_sleep(bar_accf + 8 * (int)(m % NA), (uint32_t)((m / NA) & 1));
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(p.tmem_cols)
                 : "memory");
  }
}

// -inf for each row's columns [L_r, max_len)
__global__ void fill_kernel(float* logits, int64_t ld, const int32_t* ctx, int next_n,
                            int64_t max_len) {
  const int r = blockIdx.x;
  const int64_t L = row_len(ctx[r / next_n], next_n, r % next_n, max_len);
  float* row = logits + (int64_t)r * ld;
  for (int64_t t = L + threadIdx.x; t < max_len; t += blockDim.x) row[t] = -INFINITY;
}

// --- top-k per row -----------------------------------------------------------

constexpr int kTkThreads = 512;            // 16 warps; two CTAs per SM
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kTkMax = QSA_IDX_MAX_TOPK;   // 2048
constexpr int kTkUnroll = 8;               // scalar logits loaded per lane before use
constexpr int kTkVec = 4;                  // float4 loads per lane before use
constexpr int kTkCand = 10240;             // candidate (key, column) pairs kept in smem
constexpr int kTkChunks = 256;             // sampled 32-column chunks of a long row
constexpr int kTkSample = kTkChunks * 32;  // 8192 sampled keys
constexpr int kTkTarget = 4096;            // candidates the sampled threshold aims at

struct TkParams {
  const float* logits;
  int64_t s0, s1, num_cols;
  const int32_t* seq_lens;
  int next_n;
  int topk;
  int32_t* out;
  int64_t out_s0;
};

struct TkShared {
  unsigned long long sel[kTkMax];
  uint32_t hist[2048];
  uint32_t cand_k[kTkCand];
  uint32_t cand_i[kTkCand];
  uint32_t wsum[kTkWarps];
  uint32_t wmax[kTkWarps];
  uint32_t wties[kTkWarps];
  uint32_t digit, above, dcount;
  int cnt_above;
  int ncand;
};

// Unsigned key with the order of the float (-0 taken as +0: they are equal).
__device__ __forceinline__ uint32_t ordered(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The float whose key is k (k the key of some float; never -0).
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Warp-wide: the lanes with c set take consecutive slots from *counter (one
// shared atomic per warp); returns this lane's slot (meaningful where c).
__device__ __forceinline__ int tk_warp_slot(int* counter, bool c) {
  const int lane = threadIdx.x & 31;
  const uint32_t bal = __ballot_sync(0xffffffffu, c);
  int base = 0;
  if (lane == 0 && bal) base = atomicAdd(counter, __popc(bal));
  base = __shfl_sync(0xffffffffu, base, 0);
  return base + __popc(bal & ((1u << lane) - 1u));
}

// hist[0..nb): the digit d with above(d) < need <= above(d) + hist[d], where
// above(d) counts the keys in digits above d; also its count hist[d].
__device__ void tk_find_digit(TkShared& sh, int nb, uint32_t need) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = nb / kTkThreads;            // 4 or 2 bins per thread
  uint32_t local = 0;
  for (int k = 0; k < per; ++k) local += sh.hist[tid * per + k];
  uint32_t suf = local;                       // inclusive suffix within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_down_sync(0xffffffffu, suf, o);
    if (lane + o < 32) suf += v;
  }
  if (lane == 0) sh.wsum[warp] = suf;
  __syncthreads();
  uint32_t above = suf - local;               // keys in this warp's higher threads
  for (int w2 = warp + 1; w2 < kTkWarps; ++w2) above += sh.wsum[w2];
  for (int k = per - 1; k >= 0; --k) {
    const uint32_t h = sh.hist[tid * per + k];
    if (above < need && need <= above + h) {
      sh.digit = (uint32_t)(tid * per + k);
      sh.above = above;
      sh.dcount = h;
    }
    above += h;
  }
  __syncthreads();
}

// The K-th largest of the smem keys x[0..n) (1 <= K <= n): a radix select
// over x - min(x), 11-bit digits from the top set bit of max(x) - min(x)
// down, so the first digit spreads the keys over the range they really
// span.  *need = how many keys equal to it are among the K largest,
// *tcount = how many keys equal it.  Ends on a block barrier after its last
// read of x.
__device__ uint32_t tk_select(TkShared& sh, const uint32_t* x, int n, uint32_t K,
                              uint32_t* need_out, uint32_t* tcount_out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
  for (int i = tid; i < n; i += kTkThreads) {
    const uint32_t k = x[i];
    lo = min(lo, k);
    hi = max(hi, k);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  if (lane == 0) {
    sh.wsum[warp] = lo;
    sh.wmax[warp] = hi;
  }
  __syncthreads();
  lo = sh.wsum[0];
  hi = sh.wmax[0];
  for (int w2 = 1; w2 < kTkWarps; ++w2) {
    lo = min(lo, sh.wsum[w2]);
    hi = max(hi, sh.wmax[w2]);
  }
  __syncthreads();
  const uint32_t range = hi - lo;
  int shift = range ? 32 - __clz(range) : 0;
  uint32_t prefix = 0, need = K, tcount = (uint32_t)n;
  while (shift > 0) {
    const int w = shift < 11 ? shift : 11;
    shift -= w;
    const uint32_t himask = shift + w >= 32 ? 0u : (0xFFFFFFFFu << (shift + w));
    const uint32_t dmask = (1u << w) - 1u;
    for (int i = tid; i < 2048; i += kTkThreads) sh.hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kTkThreads) {
      const uint32_t rel = x[i] - lo;
      if ((rel & himask) == prefix) atomicAdd(&sh.hist[(rel >> shift) & dmask], 1u);
    }
    __syncthreads();
    tk_find_digit(sh, w <= 10 ? 1024 : 2048, need);
    prefix |= sh.digit << shift;
    need -= sh.above;
    tcount = sh.dcount;
    __syncthreads();
  }
  *need_out = need;
  *tcount_out = tcount;
  return lo + prefix;
}

// One CTA per row.
//  * L <= 10240: the whole row's (key, column) pairs go to shared memory.
//  * longer rows: 256 chunks of 32 columns spread over the row are sampled;
//    their ceil(4096 * 8192 / L)-th largest key T0 is a threshold about 4096
//    of the row's keys reach.  One pass (float4 loads where the row allows)
//    keeps the keys >= T0.  When between K and 10240 keys qualify, the K
//    largest of the row are among them; otherwise (a skewed sample, or
//    heavy ties) the row takes three radix passes over global memory
//    instead (11/11/10 bits) and an emission pass in warp segments ranked
//    by one scan.
// The exact K-th largest key T is selected in shared memory; the keys above
// it and the `need` ties with the smallest columns (a second select, over
// the ties' columns, only when not every tie is kept) are emitted, and a
// bitonic sort orders the K (key, column) pairs.
__global__ void __launch_bounds__(kTkThreads, 2) topk_rows_kernel(const TkParams p) {
  extern __shared__ unsigned char tk_raw[];
  TkShared& sh = *reinterpret_cast<TkShared*>(tk_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = blockIdx.x;
  int64_t L = (int64_t)p.seq_lens[r / p.next_n] - p.next_n + (r % p.next_n) + 1;
  L = L < p.num_cols ? L : p.num_cols;
  L = L > 0 ? L : 0;
  const int K = (int)(L < p.topk ? L : p.topk);
  int32_t* out = p.out + (int64_t)r * p.out_s0;
  const float* row = p.logits + (int64_t)r * p.s0;
  if (K == 0) {
    for (int i = tid; i < p.topk; i += kTkThreads) out[i] = -1;
    return;
  }
  const auto pair = [](uint32_t key, int64_t t) {
    return ((unsigned long long)key << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)t);
  };
  int n;
  if (L <= kTkCand) {
    for (int t = tid; t < (int)L; t += kTkThreads) {
      sh.cand_k[t] = ordered(row[(int64_t)t * p.s1]);
      sh.cand_i[t] = (uint32_t)t;
    }
    n = (int)L;
    __syncthreads();
  } else {
    const int64_t stride = L / kTkChunks;               // >= 40 columns
#pragma unroll 4
    for (int c = warp; c < kTkChunks; c += kTkWarps)
      sh.cand_k[c * 32 + lane] = ordered(row[((int64_t)c * stride + lane) * p.s1]);
    __syncthreads();
    const uint32_t q = (uint32_t)(((int64_t)kTkTarget * kTkSample + L - 1) / L);   // 1..4096
    uint32_t dn, dc;
    const float f0 = key_float(tk_select(sh, sh.cand_k, kTkSample, q, &dn, &dc));
    if (tid == 0) sh.ncand = 0;
    __syncthreads();
    if (p.s1 == 1 && (reinterpret_cast<uintptr_t>(row) & 15u) == 0 && L < (1ll << 31)) {
      const float4* r4 = reinterpret_cast<const float4*>(row);
      const int n4 = (int)(L >> 2);
      for (int b = warp * 32; b < n4; b += kTkThreads * kTkVec) {
        float4 v[kTkVec];
#pragma unroll
        for (int u = 0; u < kTkVec; ++u) {
          const int i = b + u * kTkThreads + lane;
          v[u] = i < n4 ? __ldg(r4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        uint32_t bal[kTkVec][4];
        int tot = 0;
#pragma unroll
        for (int u = 0; u < kTkVec; ++u) {
          const bool in = b + u * kTkThreads + lane < n4;
          bal[u][0] = __ballot_sync(0xffffffffu, in && v[u].x >= f0);
          bal[u][1] = __ballot_sync(0xffffffffu, in && v[u].y >= f0);
          bal[u][2] = __ballot_sync(0xffffffffu, in && v[u].z >= f0);
          bal[u][3] = __ballot_sync(0xffffffffu, in && v[u].w >= f0);
          tot += __popc(bal[u][0]) + __popc(bal[u][1]) + __popc(bal[u][2]) + __popc(bal[u][3]);
        }
        if (tot == 0) continue;                          // warp-uniform
        int base = 0;
        if (lane == 0) base = atomicAdd(&sh.ncand, tot);
        base = __shfl_sync(0xffffffffu, base, 0);
        const uint32_t below = (1u << lane) - 1u;
#pragma unroll
        for (int u = 0; u < kTkVec; ++u) {
          const uint32_t col = 4u * (uint32_t)(b + u * kTkThreads + lane);
          const float f[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int slot = base + __popc(bal[u][j] & below);
            if (((bal[u][j] >> lane) & 1u) && slot < kTkCand) {
              sh.cand_k[slot] = ordered(f[j]);
              sh.cand_i[slot] = col + (uint32_t)j;
            }
            base += __popc(bal[u][j]);
          }
        }
      }
      const int t = 4 * n4 + tid;                        // the last L % 4 columns
      if (t < L && row[t] >= f0) {
        const int slot = atomicAdd(&sh.ncand, 1);
        if (slot < kTkCand) {
          sh.cand_k[slot] = ordered(row[t]);
          sh.cand_i[slot] = (uint32_t)t;
        }
      }
    } else {
      for (int64_t b0 = (int64_t)warp * 32; b0 < L; b0 += (int64_t)kTkThreads * kTkUnroll) {
        float f[kTkUnroll];
#pragma unroll
        for (int u = 0; u < kTkUnroll; ++u) {
          const int64_t t = b0 + (int64_t)u * kTkThreads + lane;
          f[u] = t < L ? row[t * p.s1] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kTkUnroll; ++u) {
          const int64_t t = b0 + (int64_t)u * kTkThreads + lane;
          const bool c = t < L && f[u] >= f0;
          const int slot = tk_warp_slot(&sh.ncand, c);
          if (c && slot < kTkCand) {
            sh.cand_k[slot] = ordered(f[u]);
            sh.cand_i[slot] = (uint32_t)t;
          }
        }
      }
    }
    __syncthreads();
    n = sh.ncand;
  }
  if (n >= K && n <= kTkCand) {
    uint32_t need, tcount;
    const uint32_t T = tk_select(sh, sh.cand_k, n, (uint32_t)K, &need, &tcount);
    const bool all_ties = need == tcount;
    if (tid == 0) sh.cnt_above = 0;
    __syncthreads();
    for (int i0 = warp * 32; i0 < n; i0 += kTkThreads) {
      const int i = i0 + lane;
      const uint32_t k = i < n ? sh.cand_k[i] : 0u;
      const uint32_t col = i < n ? sh.cand_i[i] : 0u;
      const bool c = i < n && (k > T || (all_ties && k == T));
      const int slot = tk_warp_slot(&sh.cnt_above, c);
      if (c) sh.sel[slot] = pair(k, col);
      // for the column select: a tie's key becomes 2^32-1 - column (> 0,
      // columns being < 2^31), every other key 0
      if (!all_ties && i < n) sh.cand_k[i] = k == T ? 0xFFFFFFFFu - col : 0u;
    }
    if (!all_ties) {                                     // block-uniform
      __syncthreads();
      uint32_t cn, cc;
      const uint32_t C = tk_select(sh, sh.cand_k, n, need, &cn, &cc);   // the need-th smallest tie column
      for (int i0 = warp * 32; i0 < n; i0 += kTkThreads) {
        const int i = i0 + lane;
        const uint32_t kc = i < n ? sh.cand_k[i] : 0u;
        const bool c = kc != 0u && kc >= C;
        const int slot = tk_warp_slot(&sh.cnt_above, c);
        if (c) sh.sel[slot] = pair(T, 0xFFFFFFFFu - kc);
      }
    }
  } else {                                      // select over the row in global memory
    uint32_t prefix = 0, mask = 0, need = (uint32_t)K;
    const int shifts[3] = {21, 10, 0};
    const int widths[3] = {11, 11, 10};
    for (int ps = 0; ps < 3; ++ps) {
      const int nb = 1 << widths[ps];
      for (int i = tid; i < 2048; i += kTkThreads) sh.hist[i] = 0;
      __syncthreads();
      for (int64_t b0 = (int64_t)warp * 32; b0 < L; b0 += (int64_t)kTkThreads * kTkUnroll) {
        uint32_t kv[kTkUnroll];
#pragma unroll
        for (int u = 0; u < kTkUnroll; ++u) {
          const int64_t t = b0 + (int64_t)u * kTkThreads + lane;
          kv[u] = t < L ? ordered(row[t * p.s1]) : 0u;
        }
#pragma unroll
        for (int u = 0; u < kTkUnroll; ++u) {
          const int64_t t = b0 + (int64_t)u * kTkThreads + lane;
          const uint32_t k = kv[u];
          if (t < L && (k & mask) == prefix)
            atomicAdd(&sh.hist[(k >> shifts[ps]) & (uint32_t)(nb - 1)], 1u);
        }
      }
      __syncthreads();
      tk_find_digit(sh, nb < 1024 ? 1024 : nb, need);
      prefix |= sh.digit << shifts[ps];
      mask |= (uint32_t)(nb - 1) << shifts[ps];
      need -= sh.above;
      __syncthreads();
    }
    const uint32_t T = prefix;                 // the K-th largest key; `need` ties kept
    // warp segments of seg columns (a multiple of 32), in column order
    const int64_t seg = ((L + kTkWarps - 1) / kTkWarps + 31) & ~(int64_t)31;
    const int64_t s_lo = (int64_t)warp * seg;
    const int64_t s_hi = s_lo + seg < L ? s_lo + seg : L;
    uint32_t ties = 0;
    for (int64_t b0 = s_lo + lane; b0 < s_hi; b0 += 32 * kTkUnroll) {
      uint32_t kv[kTkUnroll];
#pragma unroll
      for (int u = 0; u < kTkUnroll; ++u) {
        const int64_t t = b0 + 32 * u;
        kv[u] = t < s_hi ? ordered(row[t * p.s1]) : 0u;
      }
#pragma unroll
      for (int u = 0; u < kTkUnroll; ++u) ties += kv[u] == T && b0 + 32 * u < s_hi;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ties += __shfl_xor_sync(0xffffffffu, ties, o);
    if (lane == 0) sh.wties[warp] = ties;
    if (tid == 0) sh.cnt_above = 0;
    __syncthreads();
    uint32_t rank = 0;                         // ties in the segments before this warp's
    for (int w2 = 0; w2 < warp; ++w2) rank += sh.wties[w2];
    for (int64_t c0 = s_lo; c0 < s_hi; c0 += 32 * kTkUnroll) {
      uint32_t kv[kTkUnroll];
#pragma unroll
      for (int u = 0; u < kTkUnroll; ++u) {
        const int64_t t = c0 + 32 * u + lane;
        kv[u] = t < s_hi ? ordered(row[t * p.s1]) : 0u;
      }
#pragma unroll
      for (int u = 0; u < kTkUnroll; ++u) {              // in column order
        const int64_t t = c0 + 32 * u + lane;
        const uint32_t k = kv[u];
        const bool above = t < s_hi && k > T;
        const int slot = tk_warp_slot(&sh.cnt_above, above);
        if (above) sh.sel[slot] = pair(k, t);
        const bool tie = t < s_hi && k == T;
        const uint32_t bal = __ballot_sync(0xffffffffu, tie);
        const uint32_t rk = rank + __popc(bal & ((1u << lane) - 1u));
        if (tie && rk < need) sh.sel[(uint32_t)K - need + rk] = pair(k, t);
        rank += __popc(bal);
      }
    }
  }
  // bitonic sort, descending, over the next power of two >= K
  int size = 64;
  while (size < K) size <<= 1;
  for (int i = K + tid; i < size; i += kTkThreads) sh.sel[i] = 0ull;
  __syncthreads();
  for (int kk = 2; kk <= size; kk <<= 1) {
    for (int jj = kk >> 1; jj > 0; jj >>= 1) {
      for (int pi = tid; pi < (size >> 1); pi += kTkThreads) {
        const int lo = ((pi & ~(jj - 1)) << 1) | (pi & (jj - 1));
        const int hi = lo + jj;
        const unsigned long long x = sh.sel[lo], y = sh.sel[hi];
        const bool desc_order = (lo & kk) == 0;
        if (desc_order ? (x < y) : (x > y)) {
          sh.sel[lo] = y;
          sh.sel[hi] = x;
        }
      }
      __syncthreads();
    }
  }
  for (int i = tid; i < p.topk; i += kTkThreads)
    out[i] = i < K ? (int32_t)(0xFFFFFFFFu - (uint32_t)(sh.sel[i] & 0xFFFFFFFFull)) : -1;
}

// --- host side -----------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

struct DevInfo {
  int sms = 0;
  bool ready = false;
};

cudaError_t dev_info(DevInfo** out) {
  static std::mutex mu;
  static DevInfo info[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  DevInfo& d = info[dev];
  if (!d.ready) {
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kLogitSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(topk_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(TkShared));
    if (e != cudaSuccess) return e;
    d.ready = true;
  }
  *out = &d;
  return cudaSuccess;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
struct Span {
  uintptr_t lo, hi;
};
Span span(const void* p, int64_t bytes) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return Span{lo, lo + (uintptr_t)(bytes > 0 ? bytes : 0)};
}
bool overlaps(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi && a.hi > a.lo && b.hi > b.lo; }

}  // namespace
}  // namespace qsa

extern "C" qsa_status qsa_paged_mqa_logits(
    const void* q, qsa_dtype q_dtype, int64_t num_rows, int64_t num_heads, const void* kv_cache,
    qsa_dtype kv_dtype, int64_t num_blocks, int64_t block_size, const void* weights,
    qsa_dtype weights_dtype, const void* context_lens, qsa_dtype ctx_dtype, int64_t batch,
    const void* block_tables, qsa_dtype bt_dtype, int64_t bt_cols, int64_t bt_stride0,
    int64_t next_n, void* logits, qsa_dtype logits_dtype, int64_t max_model_len,
    int64_t logits_stride0, uint32_t* error_word, qsa_stream_t stream) {
  using namespace qsa;
  if (q_dtype != QSA_DT_F8E4M3 || kv_dtype != QSA_DT_F8E4M3) return QSA_ERR_DTYPE;
  if (weights_dtype != QSA_DT_F32 || logits_dtype != QSA_DT_F32) return QSA_ERR_DTYPE;
  if (ctx_dtype != QSA_DT_I32 || bt_dtype != QSA_DT_I32) return QSA_ERR_DTYPE;
  if (num_heads != 16 && num_heads != 32 && num_heads != 64 && num_heads != 128)
    return QSA_ERR_SHAPE;
  if (next_n < 1 || next_n > 4 || num_heads * next_n > kMaxN) return QSA_ERR_SHAPE;
  if (block_size != 8 && block_size != 16 && block_size != 32 && block_size != 64 &&
      block_size != 128)
    return QSA_ERR_SHAPE;
  if (batch < 0 || num_rows != batch * next_n || num_rows > INT32_MAX / 256) return QSA_ERR_SHAPE;
  if (num_blocks < 0 || num_blocks > INT32_MAX || bt_cols < 0 || bt_cols > INT32_MAX ||
      max_model_len < 0 || max_model_len > INT32_MAX)
    return QSA_ERR_SHAPE;
  if (bt_stride0 < bt_cols || logits_stride0 < max_model_len) return QSA_ERR_STRIDE;
  if (num_rows == 0 || max_model_len == 0) return QSA_OK;
  if (!q || !weights || !context_lens || !logits) return QSA_ERR_NULL;
  if (num_blocks > 0 && !kv_cache) return QSA_ERR_NULL;
  if (bt_cols > 0 && !block_tables) return QSA_ERR_NULL;
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(weights, 16) ||
      !aligned(context_lens, 4) || !aligned(block_tables, 4) || !aligned(logits, 4) ||
      !aligned(error_word, 4))
    return QSA_ERR_ALIGN;
  const int64_t H = num_heads, N = H * next_n;
  const Span out = span(logits, ((num_rows - 1) * logits_stride0 + max_model_len) * 4);
  const Span ins[5] = {span(q, num_rows * H * kDim),
                       span(kv_cache, num_blocks * block_size * (kDim + 4)),
                       span(weights, num_rows * H * 4), span(context_lens, batch * 4),
                       span(block_tables, bt_cols > 0 ? ((batch - 1) * bt_stride0 + bt_cols) * 4 : 0)};
  for (const Span& s : ins)
    if (overlaps(out, s)) return QSA_ERR_ALIAS;
  if (error_word && (overlaps(span(error_word, 4), out))) return QSA_ERR_ALIAS;

  DevInfo* di = nullptr;
  bind_calling_thread();
  if (dev_info(&di) != cudaSuccess) return QSA_ERR_CUDA;
  auto fn = encode_fn();
  if (!fn) return QSA_ERR_CUDA;
  cudaStream_t st = (cudaStream_t)stream;
  CUtensorMap kmap, qmap;
  memset(&kmap, 0, sizeof(kmap));
  memset(&qmap, 0, sizeof(qmap));
  if (num_blocks > 0) {
    cuuint64_t dims[3] = {(cuuint64_t)kDim, (cuuint64_t)block_size, (cuuint64_t)num_blocks};
    cuuint64_t strides[2] = {(cuuint64_t)kDim, (cuuint64_t)(block_size * (kDim + 4))};
    cuuint32_t box[3] = {(cuuint32_t)kDim, (cuuint32_t)block_size, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (fn(&kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(kv_cache), dims, strides,
           box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return QSA_ERR_CUDA;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)kDim, (cuuint64_t)(num_rows * H)};
    cuuint64_t strides[1] = {(cuuint64_t)kDim};
    cuuint32_t box[2] = {(cuuint32_t)kDim, (cuuint32_t)N};
    cuuint32_t es[2] = {1, 1};
    if (fn(&qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(q), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return QSA_ERR_CUDA;
  }
  const int32_t* ctx = static_cast<const int32_t*>(context_lens);
  float* lg = static_cast<float*>(logits);
  fill_kernel<<<(unsigned)num_rows, 256, 0, st>>>(lg, logits_stride0, ctx, (int)next_n,
                                                  max_model_len);
  const int stage_bytes = (kTile * kDim + kTile * 4 + 1023) & ~1023;
  const int qslot_bytes = (int)((N * kDim + N * 4 + 1023) & ~1023);
  const int stages = (int)std::min<int64_t>(
      kMaxStages,
      (int64_t)(kLogitSmem - 1024 - 2 * qslot_bytes - kMiscBytes - kTablesBytes) / stage_bytes);
  const int nacc = N <= 128 ? 4 : 2;       // accumulators of N fp32 columns in 512
  uint32_t cols = 32;
  while (cols < (uint32_t)(nacc * N)) cols <<= 1;
  const int64_t tiles_per_req = (max_model_len + kTile - 1) / kTile;
  for (int64_t b0 = 0; b0 < batch; b0 += kMaxBatch) {
    const int nb = (int)std::min<int64_t>(kMaxBatch, batch - b0);
    LogitParams p{};
    p.kv = static_cast<const uint8_t*>(kv_cache);
    p.w = static_cast<const float*>(weights) + b0 * N;
    p.ctx = ctx + b0;
    p.bt = static_cast<const int32_t*>(block_tables) + (bt_cols > 0 ? b0 * bt_stride0 : 0);
    p.num_blocks = num_blocks;
    p.bt_cols = bt_cols;
    p.bt_s0 = bt_stride0;
    p.logits = lg + b0 * next_n * logits_stride0;
    p.ld = logits_stride0;
    p.max_len = max_model_len;
    p.err = error_word;
    p.bs = (int)block_size;
    p.H = (int)H;
    p.next_n = (int)next_n;
    p.N = (int)N;
    p.batch = nb;
    p.qrow0 = (int)(b0 * N);
    p.stage_bytes = stage_bytes;
    p.stages = stages;
    p.qslot_bytes = qslot_bytes;
    p.nacc = nacc;
    p.bs_log2 = __builtin_ctzll((unsigned long long)block_size);
    p.tmem_cols = cols;
    const int64_t items = (int64_t)nb * tiles_per_req;
    const int grid = (int)std::min<int64_t>(items, di->sms);
    logits_kernel<<<grid, kLogitThreads, kLogitSmem, st>>>(p, kmap, qmap);
  }
  return cudaGetLastError() == cudaSuccess ? QSA_OK : QSA_ERR_CUDA;
}

extern "C" qsa_status qsa_top_k_per_row_decode(
    const void* logits, qsa_dtype logits_dtype, int64_t num_rows, int64_t num_cols,
    int64_t stride0, int64_t stride1, int64_t next_n, const void* seq_lens,
    qsa_dtype seq_lens_dtype, int64_t batch, int64_t topk_tokens, void* indices,
    qsa_dtype idx_dtype, int64_t idx_stride0, qsa_stream_t stream) {
  using namespace qsa;
  if (logits_dtype != QSA_DT_F32 || seq_lens_dtype != QSA_DT_I32 || idx_dtype != QSA_DT_I32)
    return QSA_ERR_DTYPE;
  if (next_n < 1 || batch < 0 || num_rows != batch * next_n || num_rows > INT32_MAX)
    return QSA_ERR_SHAPE;
  if (num_cols < 0 || num_cols > INT32_MAX) return QSA_ERR_SHAPE;
  if (topk_tokens < 1 || topk_tokens > kTkMax) return QSA_ERR_CONTRACT;
  if (stride1 < 1 || stride0 < 0 || idx_stride0 < topk_tokens) return QSA_ERR_STRIDE;
  if (num_rows > 1 && stride0 < 1) return QSA_ERR_STRIDE;
  if (num_rows == 0) return QSA_OK;
  if (!seq_lens || !indices || (num_cols > 0 && !logits)) return QSA_ERR_NULL;
  if (!aligned(logits, 4) || !aligned(seq_lens, 4) || !aligned(indices, 4)) return QSA_ERR_ALIGN;
  const Span out = span(indices, ((num_rows - 1) * idx_stride0 + topk_tokens) * 4);
  const int64_t lg_extent =
      num_cols > 0 ? ((num_rows - 1) * stride0 + (num_cols - 1) * stride1 + 1) * 4 : 0;
  if (overlaps(out, span(logits, lg_extent)) || overlaps(out, span(seq_lens, batch * 4)))
    return QSA_ERR_ALIAS;
  DevInfo* di = nullptr;
  bind_calling_thread();
  if (dev_info(&di) != cudaSuccess) return QSA_ERR_CUDA;
  TkParams p{};
  p.logits = static_cast<const float*>(logits);
  p.s0 = stride0;
  p.s1 = stride1;
  p.num_cols = num_cols;
  p.seq_lens = static_cast<const int32_t*>(seq_lens);
  p.next_n = (int)next_n;
  p.topk = (int)topk_tokens;
  p.out = static_cast<int32_t*>(indices);
  p.out_s0 = idx_stride0;
  topk_rows_kernel<<<(unsigned)num_rows, kTkThreads, sizeof(TkShared), (cudaStream_t)stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? QSA_OK : QSA_ERR_CUDA;
}
