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
//   score_kernel  streams every visible compressed key of every row once
//                 (the dominant HBM stream: 256 B per key) and writes a 32-bit
//                 ordered score key per block to the workspace;
//   topk_kernel   one CTA per row: exact radix select of the top-512 keys over
//                 the row's scores (L2-resident), bitonic sort of the winners,
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

namespace qsa {
namespace {

constexpr int kScoreThreads = 256;                 // 8 warps
constexpr int kKeysPerWarpIter = 8;                // 4 lanes per key
constexpr int kScoreIters = 4;
constexpr int kKeysPerCta = (kScoreThreads / 32) * kKeysPerWarpIter * kScoreIters;  // 256

constexpr int kTopkThreads = 512;

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

__global__ void __launch_bounds__(kScoreThreads)
score_kernel(const SelectParams p) {
  const int r = blockIdx.y;
  const RowSetup rs = row_setup(p, r);
  if (!rs.ok) return;
  const int64_t Vs = rs.V < p.vcap ? rs.V : p.vcap;
  const int64_t cta_base = (int64_t)blockIdx.x * kKeysPerCta;
  if (cta_base >= Vs) return;

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int t = lane & 3;          // 32-dim slice of the key
  const int kslot = lane >> 2;     // key within the warp's group of 8

  // query slice [32t, 32t+32) of each head, as (even, odd) binary32 pairs
  float2 q[kSelHeads][16];
  {
    const uint4* qp = reinterpret_cast<const uint4*>(p.q_sel + (int64_t)r * kSelHeads * kSelDim);
#pragma unroll
    for (int h = 0; h < kSelHeads; ++h) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint4 v = qp[h * 16 + t * 4 + i];
        q[h][4 * i + 0] = h2f2(v.x);
        q[h][4 * i + 1] = h2f2(v.y);
        q[h][4 * i + 2] = h2f2(v.z);
        q[h][4 * i + 3] = h2f2(v.w);
      }
    }
  }
  const int32_t* ptrow = p.pt + (int64_t)rs.req * p.pt_stride0;
  uint32_t* srow = p.scores + (int64_t)r * p.vcap;

#pragma unroll 1
  for (int it = 0; it < kScoreIters; ++it) {
    const int64_t b = cta_base + warp * (kKeysPerWarpIter * kScoreIters) + it * kKeysPerWarpIter + kslot;
    const bool inb = b < Vs;
    bool valid = false;
    uint4 kv[4] = {};
    if (inb) {
      const int32_t pg = ptrow[b >> 7];
      valid = pg >= 0 && pg < p.num_pages;
      if (valid) {
        const __half* kp = p.cmp + (int64_t)pg * kCmpPageHalves + (b & 127) * kSelDim + 32 * t;
#pragma unroll
        for (int i = 0; i < 4; ++i) kv[i] = ld_stream16(kp + 8 * i);
      } else if (t == 0) {
        report(p.err, kErrCmpPage);
      }
    }
    float2 acc[kSelHeads];
#pragma unroll
    for (int h = 0; h < kSelHeads; ++h) acc[h] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t w[4] = {kv[i].x, kv[i].y, kv[i].z, kv[i].w};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float2 kf = h2f2(w[m]);
#pragma unroll
        for (int h = 0; h < kSelHeads; ++h) acc[h] = ffma2(q[h][4 * i + m], kf, acc[h]);
      }
    }
    float P[kSelHeads];
#pragma unroll
    for (int h = 0; h < kSelHeads; ++h) P[h] = __fadd_rn(acc[h].x, acc[h].y);

    // quad reduce-scatter: lanes t, t^2 first (slices 0+2, 1+3), then t^1;
    // lane t ends with head t's d = (P0 + P2) + (P1 + P3).
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
    const float s = __fadd_rn(u, __shfl_xor_sync(0xffffffffu, u, 2));
    if (inb && t == 0) srow[b] = valid ? (__float_as_uint(s) + 1u) : 0u;
  }
}

// ---------------------------------------------------------------------------
// top-k: exact radix select over 32-bit ordered score keys
// ---------------------------------------------------------------------------

__device__ __forceinline__ void warp_hist_add(uint32_t* hist, uint32_t bin, int lane) {
  const unsigned m = __match_any_sync(0xffffffffu, bin);
  if (bin < 256u && lane == __ffs(m) - 1) atomicAdd(&hist[bin], (uint32_t)__popc(m));
}

__global__ void __launch_bounds__(kTopkThreads)
topk_kernel(const SelectParams p) {
  const int r = blockIdx.x;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  constexpr int kWarps = kTopkThreads / 32;

  __shared__ uint32_t hist[256];
  __shared__ unsigned long long keys[kTopkBlocks];
  __shared__ uint32_t warp_cnt[kWarps];
  __shared__ uint32_t s_prefix, s_krem, s_nvalid;
  __shared__ int s_count;

  const RowSetup rs = row_setup(p, r);
  int32_t* out = p.out + (int64_t)r * p.out_stride0;
  if (!rs.ok) {
    for (int j = tid; j < kOutWidth; j += kTopkThreads) out[j] = -1;
    if (tid == 0) report(p.err, kErrRequest);
    return;
  }
  if (tid == 0 && rs.V > p.vcap) report(p.err, kErrCmpPage);
  const int64_t Vs = rs.V < p.vcap ? rs.V : p.vcap;
  const uint32_t* sc = p.scores + (int64_t)r * p.vcap;

  uint32_t prefix = 0, pmask = 0, K = 0, krem = 0;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    for (int64_t base = 0; base < Vs; base += kTopkThreads) {
      const int64_t i = base + tid;
      const uint32_t x = i < Vs ? sc[i] : 0u;
      const bool match = x != 0u && (x & pmask) == prefix;
      warp_hist_add(hist, match ? (x >> shift) & 255u : 256u, lane);
    }
    __syncthreads();
    if (tid == 0) {
      if (pass == 0) {
        uint32_t n = 0;
        for (int d = 0; d < 256; ++d) n += hist[d];
        s_nvalid = n;
        s_krem = n < (uint32_t)kTopkBlocks ? n : (uint32_t)kTopkBlocks;
      }
      uint32_t need = s_krem, above = 0;
      int dsel = 0;
      if (need > 0) {
        for (int d = 255; d >= 0; --d) {
          if (above + hist[d] >= need) { dsel = d; break; }
          above += hist[d];
        }
      }
      s_krem = need - above;
      s_prefix = prefix | ((uint32_t)dsel << shift);
    }
    __syncthreads();
    if (pass == 0) K = s_nvalid < (uint32_t)kTopkBlocks ? s_nvalid : (uint32_t)kTopkBlocks;
    if (K == 0) break;
    prefix = s_prefix;
    pmask |= 255u << shift;
    krem = s_krem;
    __syncthreads();
  }

  if (K > 0) {
    const uint32_t T = prefix;   // the K-th largest key value
    if (tid == 0) s_count = 0;
    __syncthreads();
    // every key strictly above T is in
    for (int64_t i = tid; i < Vs; i += kTopkThreads) {
      const uint32_t x = sc[i];
      if (x > T) {
        const int slot = atomicAdd(&s_count, 1);
        keys[slot] = ((unsigned long long)x << 32) | (0xffffffffu - (uint32_t)i);
      }
    }
    // among keys equal to T, the krem with the smallest block index
    uint32_t taken = 0;
    for (int64_t base = 0; base < Vs && taken < krem; base += kTopkThreads) {
      const int64_t i = base + tid;
      const bool eq = i < Vs && sc[i] == T;
      const unsigned bal = __ballot_sync(0xffffffffu, eq);
      if (lane == 0) warp_cnt[warp] = __popc(bal);
      __syncthreads();
      uint32_t off = 0, tot = 0;
      for (int w = 0; w < kWarps; ++w) {
        const uint32_t c = warp_cnt[w];
        off += (w < warp) ? c : 0u;
        tot += c;
      }
      const uint32_t rank = taken + off + __popc(bal & ((1u << lane) - 1u));
      if (eq && rank < krem) {
        const int slot = atomicAdd(&s_count, 1);
        keys[slot] = ((unsigned long long)T << 32) | (0xffffffffu - (uint32_t)i);
      }
      taken += tot;
      __syncthreads();
    }
    __syncthreads();
  }
  for (int i = (int)K + tid; i < kTopkBlocks; i += kTopkThreads) keys[i] = 0ull;
  __syncthreads();

  // bitonic sort, descending (score desc, then block asc via the ~index)
  for (int k = 2; k <= kTopkBlocks; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < kTopkBlocks; i += kTopkThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long a = keys[i], c = keys[ixj];
          const bool desc = (i & k) == 0;
          if (desc ? (a < c) : (a > c)) { keys[i] = c; keys[ixj] = a; }
        }
      }
      __syncthreads();
    }
  }

  // expand kept blocks, then tail, then -1
  for (int j = tid; j < (int)K; j += kTopkThreads) {
    const int32_t b = (int32_t)(0xffffffffu - (uint32_t)(keys[j] & 0xffffffffull));
    const int32_t tok = b * kRatio;
    out[4 * j + 0] = tok;
    out[4 * j + 1] = tok + 1;
    out[4 * j + 2] = tok + 2;
    out[4 * j + 3] = tok + 3;
  }
  const int64_t tail0 = rs.V * kRatio;
  const int64_t tail_len = rs.tail_end >= tail0 ? rs.tail_end - tail0 + 1 : 0;
  for (int j = 4 * (int)K + tid; j < kOutWidth; j += kTopkThreads) {
    const int64_t tt = j - 4 * (int64_t)K;
    out[j] = tt < tail_len ? (int32_t)(tail0 + tt) : -1;
  }
}

}  // namespace

size_t select_workspace_bytes(int64_t R, int64_t pt_cols) {
  const size_t n = (size_t)R * (size_t)pt_cols * kCmpPageKeys * sizeof(uint32_t);
  return (n + 255) & ~(size_t)255;
}

cudaError_t launch_select(const SelectParams& p, cudaStream_t stream) {
  if (p.R == 0) return cudaSuccess;
  const int64_t ctas = (p.vcap + kKeysPerCta - 1) / kKeysPerCta;
  if (ctas > 0) {
    dim3 grid((unsigned)ctas, (unsigned)p.R);
    score_kernel<<<grid, kScoreThreads, 0, stream>>>(p);
  }
  topk_kernel<<<p.R, kTopkThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace qsa
