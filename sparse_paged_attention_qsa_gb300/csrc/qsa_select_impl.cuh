// qsa_select_impl.cuh -- device code shared by the selection kernels
// (qsa_select.cu) and the fused small-batch decode kernel (qsa_fused.cu):
// row setup, the canonical score of a key by a quad of lanes, and the exact
// top-512 of one row by a 512-thread CTA.
//
// "vLLM: integrate FP16 packed QSA extension", Summary (fused selection) and
// "Exact contracts"/Selection; visible blocks from qsa_cache.py,
// _build_qsa_metadata_kernel.  The score order is described in qsa_select.cu.
#pragma once

#include "qsa_internal.h"
#include "qsa_device.cuh"

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
// The score kernel also keeps the largest key of each run of 16 blocks (one
// warp step: two groups of 8 keys), so the top-k reads 1/16 of a row first.
constexpr int kUnitKeys = 16;

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

// Where topk_row writes the row's 2051 output entries: out(j, value).
struct RowOut {
  int32_t* row;   // the row of p.out
  __device__ __forceinline__ void operator()(int j, int32_t v) const { row[j] = v; }
};

// Top-k of row r by the CTA's kTopkThreads threads into `sh`, written
// through `out`.  In the top-k kernel the CTA is a programmatic dependent of
// the score kernel and waits for it after the row's setup (in the fused
// kernel that wait is a no-op: a cluster barrier precedes the call).
// kDense: every row of the launch has at most kCandCap blocks (the page
// table is at most kCandCap / 128 columns wide), and all of a row's keys are
// its candidates.  Ends after its last output write (no final barrier).

template <bool kDense, typename Out>
__device__ __forceinline__ void topk_row(const SelectParams& p, int r, TopkShared& sh,
                                         const Out& out) {
  const int tid = threadIdx.x, lane = tid & 31;
  const RowSetup rs = row_setup(p, r);
  if (!rs.ok) {
    pdl_wait();
    for (int j = tid; j < kOutWidth; j += kTopkThreads) out(j, -1);
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
      // four lanes per hit unit, 16 bytes (4 keys) each: one warp load covers
      // 8 whole units (a lane per unit made every load touch 32 lines; more
      // loads in flight per thread measured slower)
      constexpr int kQuadUnits = kTopkThreads / 4;            // units per round
      const int q = tid & 3;
      for (int base = 0; base < nhit; base += kQuadUnits) {
        const int h = base + (tid >> 2);
        const int64_t g = h < nhit ? (int64_t)hit[h] : -1;
        const uint4 v = g >= 0 ? ld_cg16(sc + kUnitKeys * g + 4 * q) : make_uint4(0, 0, 0, 0);
        const int64_t k0 = kUnitKeys * g + 4 * q;               // this lane's first block
        uint32_t mask = 0;                                     // bit j: block k0 + j
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t x = g >= 0 && k0 + j < Vs ? u4_at(v, j) : 0u;
          mask |= (uint32_t)(x >= lo) << j;
        }
        int slot = warp_reserve(&sh.ncand, __popc(mask), lane);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (mask >> j & 1u) {
            if (slot < kCandCap) {
              sh.cand_x[slot] = u4_at(v, j);
              sh.cand_i[slot] = (uint32_t)(k0 + j);
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
  // a row of at most 512 blocks keeps every key: no select, only the ordering
  const bool all_kept = kDense && Vs <= kTopkThreads;

  if (K > 0 && !all_kept) {
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
  if (all_kept) {          // slot tid: block tid's (key, ~index); blocks without a key last
    const uint32_t x = tid < Vs ? sh.cand_x[tid] : 0u;
    a = x ? ((unsigned long long)x << 32) | (0xffffffffu - (uint32_t)tid) : 0ull;
  }
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
    out(4 * tid + 0, tok);
    out(4 * tid + 1, tok + 1);
    out(4 * tid + 2, tok + 2);
    out(4 * tid + 3, tok + 3);
  }
  // then the tail, then -1
  const int64_t tail0 = rs.V * kRatio;
  const int64_t tail_len = rs.tail_end >= tail0 ? rs.tail_end - tail0 + 1 : 0;
  for (int j = 4 * (int)K + tid; j < kOutWidth; j += kTopkThreads) {
    const int64_t tt = j - 4 * (int64_t)K;
    out(j, tt < tail_len ? (int32_t)(tail0 + tt) : -1);
  }
}

}  // namespace

}  // namespace qsa
