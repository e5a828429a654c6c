// qsa_metadata.cu -- per-forward metadata of one QSA side cache, declared in
// include/qsa_metadata.h.
//
// Restates qsa_cache.py (_build_qsa_metadata_kernel): for each scheduled
// token its request, logical position, visible compressed blocks and side-cache
// slot; optionally the pre-indexer's per-request work list.  One launch of
// 256-thread CTAs; CTA b handles tokens [256b, 256b+256) and work items
// [256b, 256b+256).
//
// Token -> request: the request table (query_start_loc) is staged in shared
// memory when it fits (kStagedReqs entries), else searched in global memory;
// either way a descending power-of-two search finds the last request whose
// query starts at or before the token, never leaving [0, num_reqs).
//
// Work list: each work CTA scans the per-request item counts 256 requests at
// a time (block-wide prefix sum) and places its items by binary search in
// the chunk that holds them, so CTAs write disjoint tiles without a grid-wide
// barrier and shared memory stays fixed for any number of requests.
#include "qsa.h"
#include "qsa_metadata.h"
#include "qsa_device.cuh"
#include "qsa_host.h"

#include <cstdint>
#include <cuda_runtime.h>

namespace qsa {
namespace {

constexpr int kMetaThreads = 256;
constexpr int kStagedReqs = 8192;     // query_start_loc entries staged in smem

struct MetaParams {
  const int32_t* qsl;         // [num_reqs + 1]
  const int32_t* seq_lens;    // [num_reqs]
  const int64_t* common;      // [num_tokens] or null (circular mode)
  const int32_t* bt;          // block table
  int64_t bt_s0, bt_s1;
  int bt_cols;
  int num_reqs;
  int num_mapped;
  int num_tokens;
  int64_t sbs, cr, cbs;       // storage block size, compress ratio, ring size
  int32_t* t2r;
  int64_t* lpos;
  int32_t* vis;
  int64_t* slot;
  int32_t* work;              // [max_work][2] or null
  int max_work;
};

// the last i in [0, n) with starts[i] <= t (0 if none), for non-decreasing starts
template <typename Ptr>
__device__ __forceinline__ int last_start_at_or_before(Ptr starts, int n, int t) {
  int req = 0;
  int step = 1;
  while (step < n) step <<= 1;
  for (step >>= 1; step > 0; step >>= 1) {
    const int cand = req + step;
    if (cand < n && starts[cand] <= t) req = cand;
  }
  return req;
}

__device__ __forceinline__ int64_t work_items(const MetaParams& p, int i) {
  const int64_t q0 = p.qsl[i], q1 = p.qsl[i + 1];
  const int64_t ql = q1 - q0;
  if (ql <= 0) return 0;
  const int64_t L = p.seq_lens[i];
  const int64_t groups = floor_div(L, p.cr) - floor_div(L - ql, p.cr);
  return groups > 1 ? groups : 1;
}

__global__ void __launch_bounds__(kMetaThreads)
metadata_kernel(const MetaParams p) {
  __shared__ int32_t s_qsl[kStagedReqs];
  __shared__ int64_t s_end[kMetaThreads];
  __shared__ int64_t s_warp[kMetaThreads / 32];
  const int tid = threadIdx.x;

  // ---- tokens ----
  const int64_t t0 = (int64_t)blockIdx.x * kMetaThreads;
  if (t0 < p.num_tokens) {
    const bool staged = p.num_reqs <= kStagedReqs;
    if (staged) {
      for (int i = tid; i < p.num_reqs; i += kMetaThreads) s_qsl[i] = p.qsl[i];
    }
    __syncthreads();
    const int t = (int)t0 + tid;
    if (t < p.num_tokens) {
      const bool mapped = t < p.num_mapped;
      int req = 0;
      int64_t q1 = 0, L = 0, lp = -1;
      if (mapped) {
        req = staged ? last_start_at_or_before(s_qsl, p.num_reqs, t)
                     : last_start_at_or_before(p.qsl, p.num_reqs, t);
        const int64_t q0 = staged ? s_qsl[req] : p.qsl[req];
        q1 = p.qsl[req + 1];
        L = p.seq_lens[req];
        lp = L - (q1 - q0) + ((int64_t)t - q0);
      }
      p.t2r[t] = req;
      p.lpos[t] = lp;
      int64_t v = floor_div(lp + 1, p.cr);
      const int64_t vmax = floor_div(L, p.cr);
      v = v < vmax ? v : vmax;
      p.vis[t] = (int32_t)(v > 0 ? v : 0);

      int64_t slot = -1;
      if (p.cbs > 0) {
        // the request's ring block (column 0): the query's last cbs tokens
        if (mapped && lp >= 0 && (int64_t)t + p.cbs >= q1 && p.bt_cols > 0) {
          const int64_t blk = p.bt[(int64_t)req * p.bt_s0];
          if (blk >= 0) slot = blk * p.cbs + lp % p.cbs;
        }
      } else if (p.cr != 1) {
        // a compression group's closing token writes the group's key
        const int64_t g = (lp > 0 ? lp : 0) / p.cr;
        const int64_t col = g / p.sbs;
        if (mapped && lp >= 0 && (lp + 1) % p.cr == 0 && col < p.bt_cols) {
          const int64_t blk = p.bt[(int64_t)req * p.bt_s0 + col * p.bt_s1];
          if (blk >= 0 && p.common[t] >= 0) slot = blk * p.sbs + g % p.sbs;
        }
      } else {
        slot = p.common[t];
      }
      p.slot[t] = slot;
    }
  }

  // ---- work list ----
  const int64_t w0 = (int64_t)blockIdx.x * kMetaThreads;
  if (p.work != nullptr && w0 < p.max_work) {
    const int64_t w = w0 + tid;
    const int64_t w_last = min((int64_t)p.max_work, w0 + kMetaThreads) - 1;
    int32_t out_req = -1, out_idx = -1;
    int64_t running = 0;                    // items of the chunks already scanned
    for (int c0 = 0; c0 < p.num_reqs && running <= w_last; c0 += kMetaThreads) {
      const int i = c0 + tid;
      const int64_t cnt = i < p.num_reqs ? work_items(p, i) : 0;
      // block-wide inclusive prefix sum of cnt
      int64_t incl = cnt;
      const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) s_warp[warp] = incl;
      __syncthreads();
      int64_t before = 0;
      for (int k = 0; k < warp; ++k) before += s_warp[k];
      s_end[tid] = running + before + incl;
      __syncthreads();
      const int64_t chunk_end = s_end[kMetaThreads - 1];
      if (w <= w_last && w >= running && w < chunk_end) {
        // first j with s_end[j] > w: its request holds item w
        int lo = 0, hi = kMetaThreads - 1;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (s_end[mid] > w) hi = mid; else lo = mid + 1;
        }
        const int64_t start = lo == 0 ? running : s_end[lo - 1];
        out_req = c0 + lo;
        out_idx = (int32_t)(w - start);
      }
      running = chunk_end;
      __syncthreads();                      // s_end / s_warp reused next chunk
    }
    if (w <= w_last) {
      p.work[2 * w] = out_req;
      p.work[2 * w + 1] = out_idx;
    }
  }
  pdl_trigger();
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

extern "C" qsa_status qsa_build_metadata(
    const void* query_start_loc, qsa_dtype qsl_dtype, const void* seq_lens,
    qsa_dtype seq_lens_dtype, const void* common_slot_mapping, qsa_dtype common_dtype,
    const void* block_table, qsa_dtype bt_dtype, int64_t bt_rows, int64_t bt_cols,
    int64_t bt_stride0, int64_t bt_stride1, int64_t num_reqs, int64_t num_mapped_tokens,
    int64_t num_tokens, int64_t storage_block_size, int64_t compress_ratio,
    int64_t circular_buffer_size, int32_t* token_to_req, int64_t* logical_positions,
    int32_t* visible_blocks, int64_t* slot_mapping, int32_t* work_metadata,
    int64_t max_num_work, qsa_stream_t stream) {
  using namespace qsa;
  constexpr int64_t kI32Max = INT32_MAX;
  const bool circular = circular_buffer_size > 0;
  if (qsl_dtype != QSA_DT_I32 || seq_lens_dtype != QSA_DT_I32 || bt_dtype != QSA_DT_I32)
    return QSA_ERR_DTYPE;
  if (!circular && common_dtype != QSA_DT_I64) return QSA_ERR_DTYPE;
  if (num_reqs < 1 || num_reqs >= kI32Max || num_tokens < 0 || num_tokens >= kI32Max ||
      num_mapped_tokens < 0 || num_mapped_tokens >= kI32Max || max_num_work < 0 ||
      max_num_work >= kI32Max)
    return QSA_ERR_SHAPE;
  if (storage_block_size <= 0 || storage_block_size > kI32Max || compress_ratio <= 0 ||
      compress_ratio > kI32Max || circular_buffer_size < 0 || circular_buffer_size > kI32Max)
    return QSA_ERR_CONTRACT;
  if (bt_rows < num_reqs || bt_rows >= kI32Max || bt_cols < 0 || bt_cols >= kI32Max)
    return QSA_ERR_SHAPE;
  if (bt_cols > 0 && (bt_stride0 < 1 || bt_stride1 < 1 || bt_stride0 > ((int64_t)1 << 32) ||
                      bt_stride1 > ((int64_t)1 << 32)))
    return QSA_ERR_STRIDE;
  if (!query_start_loc || !seq_lens) return QSA_ERR_NULL;
  if (num_tokens > 0 && (!token_to_req || !logical_positions || !visible_blocks || !slot_mapping))
    return QSA_ERR_NULL;
  if (bt_cols > 0 && !block_table) return QSA_ERR_NULL;
  if (!circular && num_tokens > 0 && !common_slot_mapping) return QSA_ERR_NULL;
  if (max_num_work > 0 && !work_metadata) return QSA_ERR_NULL;
  if (!aligned(query_start_loc, 4) || !aligned(seq_lens, 4) || !aligned(block_table, 4) ||
      !aligned(common_slot_mapping, 8) || !aligned(token_to_req, 4) ||
      !aligned(logical_positions, 8) || !aligned(visible_blocks, 4) ||
      !aligned(slot_mapping, 8) || !aligned(work_metadata, 4))
    return QSA_ERR_ALIGN;
  // aliasing: the outputs against each other and every input
  const int64_t T = num_tokens;
  const int64_t bt_span = bt_cols > 0 ? ((bt_rows - 1) * bt_stride0 + (bt_cols - 1) * bt_stride1 + 1) * 4 : 0;
  const Span outs[5] = {span(token_to_req, T * 4), span(logical_positions, T * 8),
                        span(visible_blocks, T * 4), span(slot_mapping, T * 8),
                        span(work_metadata, max_num_work > 0 ? max_num_work * 8 : 0)};
  const Span ins[4] = {span(query_start_loc, (num_reqs + 1) * 4), span(seq_lens, num_reqs * 4),
                       span(circular ? nullptr : common_slot_mapping, circular ? 0 : T * 8),
                       span(block_table, bt_span)};
  for (int a = 0; a < 5; ++a) {
    for (int b = a + 1; b < 5; ++b)
      if (overlaps(outs[a], outs[b])) return QSA_ERR_ALIAS;
    for (int b = 0; b < 4; ++b)
      if (overlaps(outs[a], ins[b])) return QSA_ERR_ALIAS;
  }
  const int64_t work = max_num_work > 0 ? max_num_work : 0;
  const int64_t units = T > work ? T : work;
  if (units == 0) return QSA_OK;

  MetaParams p{};
  p.qsl = static_cast<const int32_t*>(query_start_loc);
  p.seq_lens = static_cast<const int32_t*>(seq_lens);
  p.common = circular ? nullptr : static_cast<const int64_t*>(common_slot_mapping);
  p.bt = static_cast<const int32_t*>(block_table);
  p.bt_s0 = bt_stride0;
  p.bt_s1 = bt_stride1;
  p.bt_cols = (int)bt_cols;
  p.num_reqs = (int)num_reqs;
  p.num_mapped = (int)num_mapped_tokens;
  p.num_tokens = (int)num_tokens;
  p.sbs = storage_block_size;
  p.cr = compress_ratio;
  p.cbs = circular_buffer_size;
  p.t2r = token_to_req;
  p.lpos = logical_positions;
  p.vis = visible_blocks;
  p.slot = slot_mapping;
  p.work = max_num_work > 0 ? work_metadata : nullptr;
  p.max_work = (int)max_num_work;
  const int64_t grid = (units + kMetaThreads - 1) / kMetaThreads;
  qsa::bind_calling_thread();
  metadata_kernel<<<(unsigned)grid, kMetaThreads, 0, (cudaStream_t)stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? QSA_OK : QSA_ERR_CUDA;
}
