// qsa_attention.cu -- qsa_sparse_attention on sm_103a.
//
// "vLLM: integrate FP16 packed QSA extension", Summary (exact-packed
// attention kernel) and "Exact contracts"/Attention: FP16 Q/out [R,3,256];
// FP16 K/V exact-packed with strides [262144,512,256,1] and V at storage
// offset 256 (one KV head shared by the three query heads); logical indices
// [R,2051] int32 with holes and duplicates; caller-owned output.
//
// Split-width flash decoding:
//   attn_partial_kernel  grid (splits, R); each CTA takes kSplit = 256
//                        consecutive entries of one row's index list (a
//                        2051-wide row: 9 CTAs); each warp compacts its 64
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

#include <math_constants.h>

namespace qsa {
namespace {

#ifndef QSA_ATT_SPLIT
#define QSA_ATT_SPLIT 256
#endif
constexpr int kSplit = QSA_ATT_SPLIT;  // index entries per CTA
constexpr int kAttWarps = 4;
constexpr int kWarpEntries = kSplit / kAttWarps;   // 32 or 64 entries per warp
constexpr int kAttThreads = kAttWarps * 32;
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

// One CTA = kSplit consecutive entries of one row's index list; each warp
// takes kSplit/4 of them, compacts the valid ones (holes and unmapped pages
// dropped) and walks them kBatch tokens at a time.  256 entries per CTA
// amortise the CTA's fixed costs -- the dependent index -> page-table -> K/V
// loads before streaming and the merge after it -- over 8 batches per warp
// (128 entries: 0.106 ms on 256 x 2048 rows, 256: 0.101, 512: 0.116 with
// too few CTAs to fill the GPU evenly).  Lane l owns dims
// [8l, 8l+8) of K and V, so a token's 1 KiB (K then V) is two coalesced
// 512-byte warp loads; a batch keeps 8 KiB in flight per warp.  The 24 head
// logits of a batch are reduced with one reduce-scatter, after which lane l
// holds token l/4, head l%4 (head 3 is padding); the online softmax runs in
// base 2 with one exp2 per lane per batch.
__global__ void __launch_bounds__(kAttThreads)
attn_partial_kernel(const AttentionParams p) {
  const int split = blockIdx.x;
  const int r = blockIdx.y;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;

  __shared__ float sm_m[kAttWarps][kAttHeads], sm_l[kAttWarps][kAttHeads];
  __shared__ float sm_acc[kAttWarps][kAttHeads][kAttDim];
  __shared__ uint32_t sm_tok[kAttWarps][kWarpEntries];

  pdl_trigger();   // the combine kernel may be scheduled early (it waits)
  pdl_wait();      // launched as a dependent of the previous kernel (the selection's
                   // top-k when called after it): its output is complete and visible
  const int req = p.t2r[r];
  const bool rok = req >= 0 && req < p.num_reqs;
  if (!rok && split == 0 && tid == 0) report(p.err, kErrRequest);

  // query dims [8*lane, 8*lane+8) of each head, fp16 pairs
  uint32_t qh[kAttHeads][4];
  {
    const uint4* qp = reinterpret_cast<const uint4*>(p.q + (int64_t)r * kAttHeads * kAttDim);
#pragma unroll
    for (int h = 0; h < kAttHeads; ++h) {
      const uint4 v = qp[h * 32 + lane];
      qh[h][0] = v.x; qh[h][1] = v.y; qh[h][2] = v.z; qh[h][3] = v.w;
    }
  }

  // resolve this warp's entries to tokens (page*512 + slot), dropping holes,
  // 32 at a time (one per lane), compacted in order
  int nvalid = 0;
#pragma unroll
  for (int c = 0; c < kWarpEntries; c += 32) {
    const int64_t j = (int64_t)split * kSplit + warp * kWarpEntries + c + lane;
    bool valid = false;
    uint32_t tok = 0;
    if (rok && j < p.width) {
      const int32_t i = p.idx[(int64_t)r * p.idx_stride0 + j];
      if (i >= 0) {
        const int64_t col = i >> 9;
        int32_t pg = -1;
        if (col < p.pt_cols) pg = p.pt[(int64_t)req * p.pt_stride0 + col];
        if (pg >= 0 && pg < p.num_pages) {
          valid = true;
          tok = (uint32_t)pg * kKvPageTokens + (uint32_t)(i & 511);
        } else {
          report(p.err, kErrKvPage);
        }
      }
    }
    const unsigned vmask = __ballot_sync(0xffffffffu, valid);
    if (valid) sm_tok[warp][nvalid + __popc(vmask & ((1u << lane) - 1u))] = tok;
    nvalid += __popc(vmask);
  }
  __syncwarp();

  const int hh = lane & 3;         // head of this lane's logit after the reduce
  float m_run = -CUDART_INF_F, l_run = 0.f;
  float acc[kAttHeads][8];
#pragma unroll
  for (int h = 0; h < kAttHeads; ++h)
#pragma unroll
    for (int d = 0; d < 8; ++d) acc[h][d] = 0.f;

  for (int b0 = 0; b0 < nvalid; b0 += kBatch) {
    uint4 kr[kBatch], vr[kBatch];
#pragma unroll
    for (int t = 0; t < kBatch; ++t) {
      if (b0 + t < nvalid) {
        const __half* tp = p.kv + (int64_t)sm_tok[warp][b0 + t] * kKvTokenHalves;
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
    const bool live = hh < kAttHeads && b0 + tt < nvalid;
    const float z = live ? dot * p.scale_log2 : -CUDART_INF_F;
    // batch max per head over the 8 tokens (lanes with the same l%4)
    float mb = z;
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 4));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 8));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 16));
    const float m_new = fmaxf(m_run, mb);
    const bool any = m_new != -CUDART_INF_F;
    const float c = any ? exp2f(m_run - m_new) : 1.f;
    const float pz = any ? exp2f(z - m_new) : 0.f;
    float ps = pz;
    ps += __shfl_xor_sync(0xffffffffu, ps, 4);
    ps += __shfl_xor_sync(0xffffffffu, ps, 8);
    ps += __shfl_xor_sync(0xffffffffu, ps, 16);
    l_run = fmaf(l_run, c, ps);
    m_run = m_new;
    // P.V over the batch: every lane needs all 24 weights and 3 scales
    float ch[kAttHeads];
#pragma unroll
    for (int h = 0; h < kAttHeads; ++h) ch[h] = __shfl_sync(0xffffffffu, c, h);
#pragma unroll
    for (int h = 0; h < kAttHeads; ++h)
#pragma unroll
      for (int d = 0; d < 8; ++d) acc[h][d] *= ch[h];
#pragma unroll
    for (int t = 0; t < kBatch; ++t) {
      float vf[8];
      to_f32x8(vr[t], vf);
#pragma unroll
      for (int h = 0; h < kAttHeads; ++h) {
        const float pw = __shfl_sync(0xffffffffu, pz, 4 * t + h);
#pragma unroll
        for (int d = 0; d < 8; ++d) acc[h][d] = fmaf(pw, vf[d], acc[h][d]);
      }
    }
  }

  // merge the four warps (lane h holds head h's m and l)
#pragma unroll
  for (int h = 0; h < kAttHeads; ++h) {
#pragma unroll
    for (int d = 0; d < 8; ++d) sm_acc[warp][h][8 * lane + d] = acc[h][d];
  }
  if (lane < kAttHeads) {
    sm_m[warp][lane] = m_run;
    sm_l[warp][lane] = l_run;
  }
  __syncthreads();
  float* part = p.part + ((int64_t)r * p.nsplit + split) * kPartFloats;
  for (int o = tid; o < kAttHeads * kAttDim; o += kAttThreads) {
    const int h = o / kAttDim, d = o % kAttDim;
    float M = sm_m[0][h];
#pragma unroll
    for (int w = 1; w < kAttWarps; ++w) M = fmaxf(M, sm_m[w][h]);
    float A = 0.f, Lsum = 0.f;
    if (M != -CUDART_INF_F) {
#pragma unroll
      for (int w = 0; w < kAttWarps; ++w) {
        const float cw = exp2f(sm_m[w][h] - M);
        A = fmaf(cw, sm_acc[w][h][d], A);
        Lsum = fmaf(cw, sm_l[w][h], Lsum);
      }
    }
    part[kAttHeads * 2 + o] = A;
    if (d == 0) {
      part[h] = M;
      part[kAttHeads + h] = Lsum;
    }
  }
}

constexpr int kMaxSplits = (kOutWidth + kSplit - 1) / kSplit;   // 9

// One CTA per row: log-sum-exp merge of the row's split partials, FP16
// round-to-nearest output; thread d handles dim d of every head.  The
// partials' (m, l) are fetched by parallel threads and every per-split load
// is independent, so the merge costs a few memory round trips.
__global__ void __launch_bounds__(kAttDim)
attn_combine_kernel(const AttentionParams p) {
  __shared__ float sm_m[kMaxSplits][kAttHeads], sm_l[kMaxSplits][kAttHeads];
  __shared__ float w_s[kMaxSplits][kAttHeads];
  __shared__ float inv_l[kAttHeads];
  const int r = blockIdx.x;
  const int d = threadIdx.x;
  const int ns = p.nsplit;
  const float* base = p.part + (int64_t)r * ns * kPartFloats;
  pdl_wait();      // every split partial is written and visible
  if (d < ns * kAttHeads) {
    const int s = d / kAttHeads, h = d % kAttHeads;
    sm_m[s][h] = base[s * kPartFloats + h];
    sm_l[s][h] = base[s * kPartFloats + kAttHeads + h];
  }
  // this thread's accumulators of every split, loaded up front
  float a[kAttHeads][kMaxSplits];
#pragma unroll
  for (int s = 0; s < kMaxSplits; ++s)
#pragma unroll
    for (int h = 0; h < kAttHeads; ++h)
      a[h][s] = s < ns ? base[s * kPartFloats + kAttHeads * 2 + h * kAttDim + d] : 0.f;
  __syncthreads();
  if (d < kAttHeads) {
    const int h = d;
    float M = -CUDART_INF_F;
    for (int s = 0; s < ns; ++s) M = fmaxf(M, sm_m[s][h]);
    float L = 0.f;
    for (int s = 0; s < ns; ++s) {
      const float w = M == -CUDART_INF_F ? 0.f : exp2f(sm_m[s][h] - M);
      w_s[s][h] = w;
      L = fmaf(w, sm_l[s][h], L);
    }
    inv_l[h] = L > 0.f ? 1.f / L : 0.f;
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < kAttHeads; ++h) {
    float A = 0.f;
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s)
      if (s < ns) A = fmaf(w_s[s][h], a[h][s], A);
    p.out[((int64_t)r * kAttHeads + h) * kAttDim + d] = __float2half_rn(A * inv_l[h]);
  }
}

}  // namespace

int attention_splits(int64_t width) {
  const int64_t s = (width + kSplit - 1) / kSplit;
  return s > 0 ? (int)s : 1;
}

size_t attention_workspace_bytes(int64_t R, int64_t width) {
  const size_t n = (size_t)R * (size_t)attention_splits(width) * kPartFloats * sizeof(float);
  return (n + 255) & ~(size_t)255;
}

cudaError_t launch_attention(const AttentionParams& p, cudaStream_t stream) {
  if (p.R == 0) return cudaSuccess;
  dim3 grid((unsigned)p.nsplit, (unsigned)p.R);
  // a programmatic dependent of whatever ran before on the stream: after the
  // selection's top-k (which triggers at its start) the launch and CTA
  // scheduling overlap the top-k's tail; the kernel waits before any read
  cudaError_t e = launch_after(attn_partial_kernel, grid, dim3(kAttThreads), 0, stream, p);
  if (e != cudaSuccess) return e;
  return launch_after(attn_combine_kernel, dim3(p.R), dim3(kAttDim), 0, stream, p);
}

}  // namespace qsa
