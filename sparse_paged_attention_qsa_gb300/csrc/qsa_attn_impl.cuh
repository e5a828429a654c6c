// qsa_attn_impl.cuh -- device code of the sparse attention kernels
// (qsa_attention.cu): resolving index lists, the warp's walk over tokens,
// and the log-sum-exp merges.
//
// "vLLM: integrate FP16 packed QSA extension", Summary (exact-packed
// attention kernel) and "Exact contracts"/Attention: three FP16 query heads
// share one KV head; each logical index of the row's list (holes = -1,
// duplicates allowed) is mapped through the request's K/V page table to a
// token of the exact-packed cache (1 KiB: K then V); scale 1/sqrt(256);
// FP32 accumulation; FP16 output, round to nearest even; no valid entry
// gives 0.
//
// Flash decoding over pieces of the index list: a warp walks a run of the
// list and keeps a running (m, l, acc) per head in base 2; the warps of a
// CTA merge into one partial per piece; one pass per row merges the pieces
// by log-sum-exp.
#pragma once

#include "qsa_internal.h"
#include "qsa_device.cuh"

#include <math_constants.h>

namespace qsa {
namespace attn {

constexpr int kBatch = 8;            // tokens per warp step
constexpr int kPartFloats = kAttHeads * 2 + kAttHeads * kAttDim;   // m[3], l[3], acc[3][256]

// A warp's running softmax state: lane h < 3 holds head h's m and l (base 2;
// lanes 4h..4h+3 while a walk is under way, see attend_tokens_mma); lane l
// holds dims [8l, 8l+8) of each head's accumulator.
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
  for (int c = 0; c < kIter; ++c) {   // issued without waiting for the request id
    const int64_t j = j0 + 32 * c + lane;
    iv[c] = 32 * c + lane < kEntries && j < p.width ? p.idx[(int64_t)r * p.idx_stride0 + j] : -1;
  }
#pragma unroll
  for (int c = 0; c < kIter; ++c) iv[c] = rok ? iv[c] : -1;
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

// --- tensor-core logits --------------------------------------------------------
//
// The batch's 3 x 8 logits as one warp-level MMA chain, Q (16 rows: the 3
// heads, zero padding) x K^T (8 tokens): 16 mma.m16n8k16 (fp16 operands,
// binary32 accumulation) over the 256 dims.  A dot product does not depend
// on the order of its dims, so each lane takes a fixed set of 64 dims of its
// token -- lane l (token l/4, c = l%4) dims 32i + 8c .. 32i + 8c + 7, i < 8:
// four lanes read 64 contiguous bytes of a token's K per load -- and slice
// (i, u) of the MMA chain maps the fragment's k = 2c + {0,1} to dims
// 32i + 8c + 4u + {0,1} and k = 2c + 8 + {0,1} to 32i + 8c + 4u + 2 + {0,1},
// in the K operand and, through QFrag, in the Q operand alike.  The
// accumulator fragment then holds in lane l the logits of head l/4 (rows
// >= 3 are padding) for tokens 2c and 2c + 1.

// Q operand of a row: entry [i][l] holds dims 32i + 8c .. 32i + 8c + 7 of
// head l/4 for l/4 < 3 (c = l%4), zeros for the padding rows.
struct QFrag {
  uint4 v[8][32];
};

// Every thread of the CTA calls this (nthreads of them); the caller
// synchronises before the fragments are read.
__device__ __forceinline__ void stage_query(const AttentionParams& p, int r, QFrag& qf, int tid,
                                            int nthreads) {
  const uint4* qp = reinterpret_cast<const uint4*>(p.q + (int64_t)r * kAttHeads * kAttDim);
  for (int e = tid; e < 8 * 32; e += nthreads) {
    const int i = e >> 5, l = e & 31, g = l >> 2, c = l & 3;
    qf.v[i][l] = g < kAttHeads ? qp[g * (kAttDim / 8) + 4 * i + c] : make_uint4(0, 0, 0, 0);
  }
}

// A fragment read from shared memory that the compiler may not hoist out of
// the token loop (it would hold 32 more registers per thread).
__device__ __forceinline__ uint4 lds_frag(const uint4* a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"((uint32_t)__cvta_generic_to_shared(a)));
  return v;
}

// d += A x B for one 16 x 8 x 16 slice; A rows 8..15 are zero
__device__ __forceinline__ void mma_slice(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0,
                                          uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

// Batch b0's operands (tokens tok[b0 .. b0+8) of tok[0..n)): kr = this
// lane's 128 bytes of token b0 + l/4's K (the MMA operand), vr = dims
// [8l, 8l+8) of every token's V (this lane's share of the P.V
// accumulators); zeros past n.
__device__ __forceinline__ void mma_load(const AttentionParams& p, const uint32_t* tok, int n,
                                         int b0, uint4 (&kr)[8], uint4 (&vr)[kBatch], int lane) {
  const int g = lane >> 2, c = lane & 3;
  const bool kl = b0 + g < n;
  const __half* kp = p.kv + (int64_t)tok[kl ? b0 + g : b0] * kKvTokenHalves + 8 * c;
#pragma unroll
  for (int i = 0; i < 8; ++i) kr[i] = kl ? ld_stream16(kp + 32 * i) : make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int t = 0; t < kBatch; ++t)
    vr[t] = b0 + t < n
                ? ld_stream16(p.kv + (int64_t)tok[b0 + t] * kKvTokenHalves + kAttDim + 8 * lane)
                : make_uint4(0, 0, 0, 0);
}

// Logits, online softmax and P.V of batch b0 (operands from mma_load).
__device__ __forceinline__ void mma_batch(const AttentionParams& p, int n, int b0,
                                          const uint4 (&kr)[8], const uint4 (&vr)[kBatch],
                                          const QFrag& qf, WarpState& st, int lane) {
  const int g = lane >> 2, c = lane & 3;
  // two accumulator chains (even / odd i), summed at the end
  float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint4 q = lds_frag(&qf.v[i][lane]);   // re-read per batch: no registers held
    float(&d)[4] = (i & 1) ? d1 : d0;
    mma_slice(d, q.x, q.y, kr[i].x, kr[i].y);
    mma_slice(d, q.z, q.w, kr[i].z, kr[i].w);
  }
  const bool hv = g < kAttHeads;
  const float z0 = hv && b0 + 2 * c < n ? (d0[0] + d1[0]) * p.scale_log2 : -CUDART_INF_F;
  const float z1 = hv && b0 + 2 * c + 1 < n ? (d0[1] + d1[1]) * p.scale_log2 : -CUDART_INF_F;
  // batch max and sum per head over the four lanes of the head
  float mb = fmaxf(z0, z1);
  mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
  mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
  const float m_new = fmaxf(st.m_run, mb);
  const bool any = m_new != -CUDART_INF_F;
  const float cs = any ? exp2f(st.m_run - m_new) : 1.f;
  const float p0 = any ? exp2f(z0 - m_new) : 0.f;
  const float p1 = any ? exp2f(z1 - m_new) : 0.f;
  float ps = p0 + p1;
  ps += __shfl_xor_sync(0xffffffffu, ps, 1);
  ps += __shfl_xor_sync(0xffffffffu, ps, 2);
  st.l_run = fmaf(st.l_run, cs, ps);
  st.m_run = m_new;
  // P.V: weight (head h, token t) is in lane 4h + t/2 (p0 for even t)
#pragma unroll
  for (int h = 0; h < kAttHeads; ++h) {
    const float ch = __shfl_sync(0xffffffffu, cs, 4 * h);
#pragma unroll
    for (int d = 0; d < 8; ++d) st.acc[h][d] *= ch;
  }
#pragma unroll
  for (int t = 0; t < kBatch; ++t) {
    const float2 v01 = h2f2(vr[t].x), v23 = h2f2(vr[t].y), v45 = h2f2(vr[t].z),
                 v67 = h2f2(vr[t].w);
#pragma unroll
    for (int h = 0; h < kAttHeads; ++h) {
      const float pw = __shfl_sync(0xffffffffu, (t & 1) ? p1 : p0, 4 * h + (t >> 1));
      const float2 pp = make_float2(pw, pw);
      float2 a;
      a = ffma2(pp, v01, make_float2(st.acc[h][0], st.acc[h][1]));
      st.acc[h][0] = a.x; st.acc[h][1] = a.y;
      a = ffma2(pp, v23, make_float2(st.acc[h][2], st.acc[h][3]));
      st.acc[h][2] = a.x; st.acc[h][3] = a.y;
      a = ffma2(pp, v45, make_float2(st.acc[h][4], st.acc[h][5]));
      st.acc[h][4] = a.x; st.acc[h][5] = a.y;
      a = ffma2(pp, v67, make_float2(st.acc[h][6], st.acc[h][7]));
      st.acc[h][6] = a.x; st.acc[h][7] = a.y;
    }
  }
}

// The warp's walk over tok[0..n), 8 tokens at a time.  While it runs,
// lanes 4g..4g+3 keep head g's running (m, l) (g < 3); the state may be
// carried over several walks, and finish_mma_state() moves it to the
// WarpState layout for the merge.
__device__ __forceinline__ void attend_tokens_mma(const AttentionParams& p, const uint32_t* tok,
                                                  int n, const QFrag& qf, WarpState& st,
                                                  int lane) {
  for (int b0 = 0; b0 < n; b0 += kBatch) {
    uint4 kr[8], vr[kBatch];
    mma_load(p, tok, n, b0, kr, vr, lane);
    mma_batch(p, n, b0, kr, vr, qf, st, lane);
  }
}

// Keeps the compiler from sinking a batch's arithmetic below the loads of
// the batches after it (which would hold a third operand set in registers):
// the state must be final here, before any later volatile load is issued.
__device__ __forceinline__ void pin_state(WarpState& st) {
  asm volatile("" : "+f"(st.acc[0][0]), "+f"(st.acc[0][1]), "+f"(st.acc[0][2]),
               "+f"(st.acc[0][3]), "+f"(st.acc[0][4]), "+f"(st.acc[0][5]), "+f"(st.acc[0][6]),
               "+f"(st.acc[0][7]), "+f"(st.m_run), "+f"(st.l_run));
  asm volatile("" : "+f"(st.acc[1][0]), "+f"(st.acc[1][1]), "+f"(st.acc[1][2]),
               "+f"(st.acc[1][3]), "+f"(st.acc[1][4]), "+f"(st.acc[1][5]), "+f"(st.acc[1][6]),
               "+f"(st.acc[1][7]));
  asm volatile("" : "+f"(st.acc[2][0]), "+f"(st.acc[2][1]), "+f"(st.acc[2][2]),
               "+f"(st.acc[2][3]), "+f"(st.acc[2][4]), "+f"(st.acc[2][5]), "+f"(st.acc[2][6]),
               "+f"(st.acc[2][7]));
}

// attend_tokens_mma with the next batch's loads issued before the current
// batch is computed (two operand sets in registers): a warp always has a
// batch of K/V in flight.
__device__ __forceinline__ void attend_tokens_mma_pipe(const AttentionParams& p,
                                                       const uint32_t* tok, int n,
                                                       const QFrag& qf, WarpState& st, int lane) {
  if (n <= 0) return;
  uint4 ka[8], va[kBatch], kb[8], vb[kBatch];
  mma_load(p, tok, n, 0, ka, va, lane);
  for (int b0 = 0; b0 < n; b0 += 2 * kBatch) {
    if (b0 + kBatch < n) mma_load(p, tok, n, b0 + kBatch, kb, vb, lane);
    mma_batch(p, n, b0, ka, va, qf, st, lane);
    pin_state(st);
    if (b0 + kBatch >= n) break;
    if (b0 + 2 * kBatch < n) mma_load(p, tok, n, b0 + 2 * kBatch, ka, va, lane);
    mma_batch(p, n, b0 + kBatch, kb, vb, qf, st, lane);
    pin_state(st);
  }
}

// head h's (m, l) from lane 4h to lane h
__device__ __forceinline__ void finish_mma_state(WarpState& st, int lane) {
  const int src = lane < kAttHeads ? 4 * lane : 0;
  st.m_run = __shfl_sync(0xffffffffu, st.m_run, src);
  st.l_run = __shfl_sync(0xffffffffu, st.l_run, src);
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
