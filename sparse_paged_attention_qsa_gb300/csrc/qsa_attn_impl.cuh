// qsa_attn_impl.cuh -- device code of the sparse attention shared by the
// split kernels (qsa_attention.cu) and the fused select -> attend path
// (qsa_select.cu).
//
// "vLLM: integrate FP16 packed QSA extension", Summary (exact-packed
// attention kernel) and "Exact contracts"/Attention: three FP16 query heads
// share one KV head; each logical index of the row's list (holes = -1,
// duplicates allowed) is mapped through the request's K/V page table to a
// token of the exact-packed cache (1 KiB: K then V); scale 1/sqrt(256);
// FP32 accumulation; FP16 output, round to nearest even; no valid entry
// gives 0.
//
// Split-width flash decoding: a warp walks a run of the index list and keeps
// a running (m, l, acc) per head in base 2; the warps of a CTA merge into one
// partial per split; one pass per row merges the splits by log-sum-exp.
#pragma once

#include "qsa_internal.h"
#include "qsa_device.cuh"

#include <math_constants.h>

namespace qsa {
namespace attn {

constexpr int kBatch = 8;            // tokens per warp step
constexpr int kPartFloats = kAttHeads * 2 + kAttHeads * kAttDim;   // m[3], l[3], acc[3][256]

// acc + a*b with fp16 operands and a binary32 accumulator
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

__device__ __forceinline__ void to_f32x8(const uint4 v, float* f) {
  const float2 a = h2f2(v.x), b = h2f2(v.y), c = h2f2(v.z), d = h2f2(v.w);
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
  f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

// Sum 32 per-lane values over the warp, reduce-scatter style: on return
// x[0] of lane l holds the warp-wide sum of value l (31 shuffles).
__device__ __forceinline__ float reduce_scatter32(float (&x)[32], int lane) {
#pragma unroll
  for (int level = 0; level < 5; ++level) {
    const int half = 16 >> level;            // values kept after this level
    const int bit = 16 >> level;             // partner lane distance
    const bool upper = (lane & bit) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? x[i] : x[i + half];
      const float keep = upper ? x[i + half] : x[i];
      x[i] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
    }
  }
  return x[0];
}

// A warp's running softmax state: lane h < 3 holds head h's m and l (base 2);
// lane l holds dims [8l, 8l+8) of each head's accumulator.
struct WarpState {
  float m_run, l_run;
  float acc[kAttHeads][8];
};

__device__ __forceinline__ void init_state(WarpState& st) {
  st.m_run = -CUDART_INF_F;
  st.l_run = 0.f;
#pragma unroll
  for (int h = 0; h < kAttHeads; ++h)
#pragma unroll
    for (int d = 0; d < 8; ++d) st.acc[h][d] = 0.f;
}

// query dims [8*lane, 8*lane+8) of each head of row r, fp16 pairs
__device__ __forceinline__ void load_query(const AttentionParams& p, int r, int lane,
                                           uint32_t (&qh)[kAttHeads][4]) {
  const uint4* qp = reinterpret_cast<const uint4*>(p.q + (int64_t)r * kAttHeads * kAttDim);
#pragma unroll
  for (int h = 0; h < kAttHeads; ++h) {
    const uint4 v = qp[h * 32 + lane];
    qh[h][0] = v.x; qh[h][1] = v.y; qh[h][2] = v.z; qh[h][3] = v.w;
  }
}

// Resolve entries [j0, j0 + kEntries) of row r's index list (those < width)
// to tokens (page*512 + slot), dropping holes and unmapped pages, compacted
// in order into tok[]; returns how many.  kEntries is 16 or a multiple of
// 32.  All index loads are issued before the page-table loads that depend on
// them, so the list costs two memory round trips however long it is.
template <int kEntries>
__device__ __forceinline__ int resolve_entries(const AttentionParams& p, int r, int req, bool rok,
                                               int64_t j0, uint32_t* tok, int lane) {
  static_assert(kEntries == 16 || kEntries % 32 == 0, "entries per warp");
  constexpr int kIter = (kEntries + 31) / 32;
  int32_t iv[kIter];
#pragma unroll
  for (int c = 0; c < kIter; ++c) {
    const int64_t j = j0 + 32 * c + lane;
    iv[c] = rok && 32 * c + lane < kEntries && j < p.width
                ? p.idx[(int64_t)r * p.idx_stride0 + j] : -1;
  }
  int32_t pg[kIter];
#pragma unroll
  for (int c = 0; c < kIter; ++c) {
    const int64_t col = iv[c] >> 9;
    pg[c] = iv[c] >= 0 && col < p.pt_cols ? p.pt[(int64_t)req * p.pt_stride0 + col] : -1;
  }
  int nvalid = 0;
#pragma unroll
  for (int c = 0; c < kIter; ++c) {
    const bool valid = iv[c] >= 0 && pg[c] >= 0 && pg[c] < p.num_pages;
    if (iv[c] >= 0 && !valid) report(p.err, kErrKvPage);
    const unsigned vmask = __ballot_sync(0xffffffffu, valid);
    if (valid)
      tok[nvalid + __popc(vmask & ((1u << lane) - 1u))] =
          (uint32_t)pg[c] * kKvPageTokens + (uint32_t)(iv[c] & 511);
    nvalid += __popc(vmask);
  }
  __syncwarp();
  return nvalid;
}

// Walk tokens tok[0..n) kBatch at a time: lane l owns dims [8l, 8l+8) of K
// and V, so a token's 1 KiB (K then V) is two coalesced 512-byte warp loads
// and a batch keeps 8 KiB in flight.  The 24 head logits of a batch are
// reduced with one reduce-scatter, after which lane l holds token l/4, head
// l%4 (head 3 is padding); the online softmax runs in base 2 with one exp2
// per lane per batch.
__device__ __forceinline__ void attend_tokens(const AttentionParams& p, const uint32_t* tok, int n,
                                              const uint32_t (&qh)[kAttHeads][4], WarpState& st,
                                              int lane) {
  const int hh = lane & 3;         // head of this lane's logit after the reduce
  for (int b0 = 0; b0 < n; b0 += kBatch) {
    uint4 kr[kBatch], vr[kBatch];
#pragma unroll
    for (int t = 0; t < kBatch; ++t) {
      if (b0 + t < n) {
        const __half* tp = p.kv + (int64_t)tok[b0 + t] * kKvTokenHalves;
        kr[t] = ld_stream16(tp + 8 * lane);
        vr[t] = ld_stream16(tp + kAttDim + 8 * lane);
      } else {
        kr[t] = make_uint4(0, 0, 0, 0);
        vr[t] = make_uint4(0, 0, 0, 0);
      }
    }
    // partial logits over this lane's 8 dims: x[4t + h]
    float x[32];
#pragma unroll
    for (int t = 0; t < kBatch; ++t) {
      const uint32_t w[4] = {kr[t].x, kr[t].y, kr[t].z, kr[t].w};
#pragma unroll
      for (int h = 0; h < kAttHeads; ++h) {
        float a = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          a = fma_h(qh[h][m], w[m], false, a);
          a = fma_h(qh[h][m], w[m], true, a);
        }
        x[4 * t + h] = a;
      }
      x[4 * t + 3] = 0.f;
    }
    const float dot = reduce_scatter32(x, lane);
    const int tt = lane >> 2;
    const bool live = hh < kAttHeads && b0 + tt < n;
    const float z = live ? dot * p.scale_log2 : -CUDART_INF_F;
    // batch max per head over the 8 tokens (lanes with the same l%4)
    float mb = z;
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 4));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 8));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 16));
    const float m_new = fmaxf(st.m_run, mb);
    const bool any = m_new != -CUDART_INF_F;
    const float c = any ? exp2f(st.m_run - m_new) : 1.f;
    const float pz = any ? exp2f(z - m_new) : 0.f;
    float ps = pz;
    ps += __shfl_xor_sync(0xffffffffu, ps, 4);
    ps += __shfl_xor_sync(0xffffffffu, ps, 8);
    ps += __shfl_xor_sync(0xffffffffu, ps, 16);
    st.l_run = fmaf(st.l_run, c, ps);
    st.m_run = m_new;
    // P.V over the batch: every lane needs all 24 weights and 3 scales
    float ch[kAttHeads];
#pragma unroll
    for (int h = 0; h < kAttHeads; ++h) ch[h] = __shfl_sync(0xffffffffu, c, h);
#pragma unroll
    for (int h = 0; h < kAttHeads; ++h)
#pragma unroll
      for (int d = 0; d < 8; ++d) st.acc[h][d] *= ch[h];
#pragma unroll
    for (int t = 0; t < kBatch; ++t) {
      float vf[8];
      to_f32x8(vr[t], vf);
#pragma unroll
      for (int h = 0; h < kAttHeads; ++h) {
        const float pw = __shfl_sync(0xffffffffu, pz, 4 * t + h);
#pragma unroll
        for (int d = 0; d < 8; ++d) st.acc[h][d] = fmaf(pw, vf[d], st.acc[h][d]);
      }
    }
  }
}

// Shared memory of a CTA merge: per warp m[3], l[3], acc[3][256].
template <int kWarps>
struct MergeSmem {
  float m[kWarps][kAttHeads], l[kWarps][kAttHeads];
  float acc[kWarps][kAttHeads][kAttDim];
};

// Merge the kWarps warp states stored in sm into one partial (m, l,
// acc[256]) per head at `part` (kPartFloats floats).  Every thread of the
// CTA calls this after the warps stored their states; it starts with a block
// barrier and ends without one, after its reads of shared memory.
template <int kWarps>
__device__ __forceinline__ void merge_stored(MergeSmem<kWarps>& sm, float* part, int tid) {
  __syncthreads();
  for (int o = tid; o < kAttHeads * kAttDim; o += kWarps * 32) {
    const int h = o / kAttDim, d = o % kAttDim;
    float M = sm.m[0][h];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) M = fmaxf(M, sm.m[w][h]);
    float A = 0.f, Lsum = 0.f;
    if (M != -CUDART_INF_F) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float cw = exp2f(sm.m[w][h] - M);
        A = fmaf(cw, sm.acc[w][h][d], A);
        Lsum = fmaf(cw, sm.l[w][h], Lsum);
      }
    }
    part[kAttHeads * 2 + o] = A;
    if (d == 0) {
      part[h] = M;
      part[kAttHeads + h] = Lsum;
    }
  }
}

// Merge the CTA's kWarps warp states (WarpState layout) into one partial.
template <int kWarps>
__device__ __forceinline__ void merge_warps(const WarpState& st, MergeSmem<kWarps>& sm, float* part,
                                            int tid, int warp, int lane) {
#pragma unroll
  for (int h = 0; h < kAttHeads; ++h)
#pragma unroll
    for (int d = 0; d < 8; ++d) sm.acc[warp][h][8 * lane + d] = st.acc[h][d];
  if (lane < kAttHeads) {
    sm.m[warp][lane] = st.m_run;
    sm.l[warp][lane] = st.l_run;
  }
  merge_stored<kWarps>(sm, part, tid);
}

template <int kMaxSplits>
struct CombineSmem {
  float m[kMaxSplits][kAttHeads], l[kMaxSplits][kAttHeads];
  float w[kMaxSplits][kAttHeads];
  float inv_l[kAttHeads];
};

// Log-sum-exp merge of row r's ns <= kMaxSplits partials (at part,
// kPartFloats apart) into the FP16 output, round to nearest even.  Threads
// d in [0, 256) each own dim d of every head; all threads of the CTA must
// call this (it holds block barriers); threads >= 256 only take part in the
// barriers.
template <int kMaxSplits>
__device__ __forceinline__ void combine_row(const AttentionParams& p, int r, const float* part,
                                            int ns, CombineSmem<kMaxSplits>& sm, int tid) {
  const int d = tid;
  if (d < ns * kAttHeads) {
    const int s = d / kAttHeads, h = d % kAttHeads;
    sm.m[s][h] = part[s * kPartFloats + h];
    sm.l[s][h] = part[s * kPartFloats + kAttHeads + h];
  }
  // this thread's accumulators of every split, loaded up front
  float a[kAttHeads][kMaxSplits];
  if (d < kAttDim) {
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s)
#pragma unroll
      for (int h = 0; h < kAttHeads; ++h)
        a[h][s] = s < ns ? part[s * kPartFloats + kAttHeads * 2 + h * kAttDim + d] : 0.f;
  }
  __syncthreads();
  if (d < kAttHeads) {
    const int h = d;
    float M = -CUDART_INF_F;
    for (int s = 0; s < ns; ++s) M = fmaxf(M, sm.m[s][h]);
    float L = 0.f;
    for (int s = 0; s < ns; ++s) {
      const float w = M == -CUDART_INF_F ? 0.f : exp2f(sm.m[s][h] - M);
      sm.w[s][h] = w;
      L = fmaf(w, sm.l[s][h], L);
    }
    sm.inv_l[h] = L > 0.f ? 1.f / L : 0.f;
  }
  __syncthreads();
  if (d < kAttDim) {
#pragma unroll
    for (int h = 0; h < kAttHeads; ++h) {
      float A = 0.f;
#pragma unroll
      for (int s = 0; s < kMaxSplits; ++s)
        if (s < ns) A = fmaf(sm.w[s][h], a[h][s], A);
      p.out[((int64_t)r * kAttHeads + h) * kAttDim + d] = __float2half_rn(A * sm.inv_l[h]);
    }
  }
}

}  // namespace attn
}  // namespace qsa
