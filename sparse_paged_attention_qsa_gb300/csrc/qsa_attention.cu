// qsa_attention.cu -- qsa_sparse_attention on sm_103a.
//
// "vLLM: integrate FP16 packed QSA extension", Summary (exact-packed
// attention kernel) and "Exact contracts"/Attention: FP16 Q/out [R,3,256];
// FP16 K/V exact-packed with strides [262144,512,256,1] and V at storage
// offset 256 (one KV head shared by the three query heads); logical indices
// [R,2051] int32 with holes and duplicates; caller-owned output.
//
// Split-width flash decoding:
//   attn_partial_kernel  grid (splits, R); each CTA takes kSplit consecutive
//                        entries of one row's index list; each warp walks 32
//                        of them.  Lane l owns dims [8l, 8l+8) of K and V, so
//                        a token's 1 KiB (K then V) is read as two coalesced
//                        512-byte warp loads.  Logits use an online softmax in
//                        base 2 (q is pre-scaled by scale*log2 e); the four
//                        warps merge in shared memory and the CTA writes one
//                        partial (m, l, acc[256]) per head to the workspace.
//   attn_combine_kernel  one CTA per row merges the splits by log-sum-exp and
//                        rounds to FP16 (nearest even).  No valid entry -> 0.
#include "qsa_internal.h"
#include "qsa_device.cuh"

#include <math_constants.h>

namespace qsa {
namespace {

constexpr int kSplit = 128;          // index entries per CTA
constexpr int kAttThreads = 128;     // 4 warps x 32 entries
constexpr int kPartFloats = kAttHeads * 2 + kAttHeads * kAttDim;   // m[3], l[3], acc[3][256]

__device__ __forceinline__ void to_f32x8(const uint4 v, float* f) {
  const float2 a = h2f2(v.x), b = h2f2(v.y), c = h2f2(v.z), d = h2f2(v.w);
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
  f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

__global__ void __launch_bounds__(kAttThreads)
attn_partial_kernel(const AttentionParams p) {
  const int split = blockIdx.x;
  const int r = blockIdx.y;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;

  __shared__ float sm_m[4][kAttHeads], sm_l[4][kAttHeads];
  __shared__ float sm_acc[4][kAttHeads][kAttDim];

  const int req = p.t2r[r];
  const bool rok = req >= 0 && req < p.num_reqs;
  if (!rok && split == 0 && tid == 0) report(p.err, kErrRequest);

  // query dims [8*lane, 8*lane+8) of each head, scaled to base-2 logits
  float qf[kAttHeads][8];
  {
    const uint4* qp = reinterpret_cast<const uint4*>(p.q + (int64_t)r * kAttHeads * kAttDim);
#pragma unroll
    for (int h = 0; h < kAttHeads; ++h) {
      to_f32x8(qp[h * 32 + lane], qf[h]);
#pragma unroll
      for (int d = 0; d < 8; ++d) qf[h][d] *= p.scale_log2;
    }
  }

  // resolve this lane's entry to a token address (or a hole)
  const int64_t j = (int64_t)split * kSplit + warp * 32 + lane;
  const __half* tok = nullptr;
  if (rok && j < p.width) {
    const int32_t i = p.idx[(int64_t)r * p.idx_stride0 + j];
    if (i >= 0) {
      const int64_t col = i >> 9;
      bool ok = col < p.pt_cols;
      int32_t pg = -1;
      if (ok) {
        pg = p.pt[(int64_t)req * p.pt_stride0 + col];
        ok = pg >= 0 && pg < p.num_pages;
      }
      if (ok) tok = p.kv + (int64_t)pg * kKvPageHalves + (int64_t)(i & 511) * kKvTokenHalves;
      else report(p.err, kErrKvPage);
    }
  }
  unsigned vmask = __ballot_sync(0xffffffffu, tok != nullptr);

  float m[kAttHeads], l[kAttHeads], acc[kAttHeads][8];
#pragma unroll
  for (int h = 0; h < kAttHeads; ++h) {
    m[h] = -CUDART_INF_F;
    l[h] = 0.f;
#pragma unroll
    for (int d = 0; d < 8; ++d) acc[h][d] = 0.f;
  }

  while (vmask) {
    const int src = __ffs(vmask) - 1;
    vmask &= vmask - 1;
    const unsigned long long a =
        __shfl_sync(0xffffffffu, (unsigned long long)tok, src);
    const __half* tp = reinterpret_cast<const __half*>(a);
    const uint4 kraw = ld_stream16(tp + 8 * lane);
    const uint4 vraw = ld_stream16(tp + kAttDim + 8 * lane);
    float kf[8], vf[8];
    to_f32x8(kraw, kf);
    to_f32x8(vraw, vf);
    float z[kAttHeads];
#pragma unroll
    for (int h = 0; h < kAttHeads; ++h) {
      float s = 0.f;
#pragma unroll
      for (int d = 0; d < 8; ++d) s = fmaf(qf[h][d], kf[d], s);
      z[h] = s;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
      for (int h = 0; h < kAttHeads; ++h) z[h] += __shfl_xor_sync(0xffffffffu, z[h], o);
    }
#pragma unroll
    for (int h = 0; h < kAttHeads; ++h) {
      const float mn = fmaxf(m[h], z[h]);
      const float c = exp2f(m[h] - mn);
      const float pz = exp2f(z[h] - mn);
      l[h] = fmaf(l[h], c, pz);
#pragma unroll
      for (int d = 0; d < 8; ++d) acc[h][d] = fmaf(acc[h][d], c, pz * vf[d]);
      m[h] = mn;
    }
  }

  // merge the four warps
#pragma unroll
  for (int h = 0; h < kAttHeads; ++h) {
#pragma unroll
    for (int d = 0; d < 8; ++d) sm_acc[warp][h][8 * lane + d] = acc[h][d];
    if (lane == 0) { sm_m[warp][h] = m[h]; sm_l[warp][h] = l[h]; }
  }
  __syncthreads();
  float* part = p.part + ((int64_t)r * p.nsplit + split) * kPartFloats;
  for (int o = tid; o < kAttHeads * kAttDim; o += kAttThreads) {
    const int h = o / kAttDim, d = o % kAttDim;
    float M = sm_m[0][h];
#pragma unroll
    for (int w = 1; w < 4; ++w) M = fmaxf(M, sm_m[w][h]);
    float A = 0.f, Lsum = 0.f;
    if (M != -CUDART_INF_F) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float c = exp2f(sm_m[w][h] - M);
        A = fmaf(c, sm_acc[w][h][d], A);
        Lsum = fmaf(c, sm_l[w][h], Lsum);
      }
    }
    part[kAttHeads * 2 + o] = A;
    if (d == 0) {
      part[h] = M;
      part[kAttHeads + h] = Lsum;
    }
  }
}

__global__ void __launch_bounds__(kAttDim)
attn_combine_kernel(const AttentionParams p) {
  const int r = blockIdx.x;
  const int d = threadIdx.x;
  const float* base = p.part + (int64_t)r * p.nsplit * kPartFloats;
#pragma unroll
  for (int h = 0; h < kAttHeads; ++h) {
    float M = -CUDART_INF_F;
    for (int s = 0; s < p.nsplit; ++s) M = fmaxf(M, base[s * kPartFloats + h]);
    float o = 0.f;
    if (M != -CUDART_INF_F) {
      float A = 0.f, L = 0.f;
      for (int s = 0; s < p.nsplit; ++s) {
        const float* ps = base + s * kPartFloats;
        const float c = exp2f(ps[h] - M);
        A = fmaf(c, ps[kAttHeads * 2 + h * kAttDim + d], A);
        L = fmaf(c, ps[kAttHeads + h], L);
      }
      o = A / L;
    }
    p.out[((int64_t)r * kAttHeads + h) * kAttDim + d] = __float2half_rn(o);
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
  attn_partial_kernel<<<grid, kAttThreads, 0, stream>>>(p);
  attn_combine_kernel<<<p.R, kAttDim, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace qsa
