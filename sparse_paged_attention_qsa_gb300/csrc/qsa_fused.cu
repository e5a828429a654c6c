// qsa_fused.cu -- the one-call decode step for batches that fit in one wave
// on sm_103a: one kernel, one thread-block cluster per row, the selected
// index list handed from the top-k to the attention in shared memory.
//
// "vLLM: integrate FP16 packed QSA extension", Summary (fused selection and
// the exact-packed attention kernel) and "Exact contracts"/Selection and
// Attention; the decode rows of qsa_cache.py (_logical_positions,
// _build_qsa_metadata_kernel).  For a few rows the chained kernels of the
// two calls are bound by their launch and dependent-load latencies, not by
// bytes, and up to a wave of rows their stages do not overlap; here a row's
// whole step is one cluster's work, every row's cluster resident at once
// (which batches take it: qsa_fused.h):
//
//  A. scoring -- CTA c of the row's cluster (CS = 1 .. 16 CTAs of 512
//     threads: the most for which the GPU holds a cluster per row) streams
//     the row's compressed pages c, c + CS, ... through a TMA ring and
//     scores every visible key in the canonical order (the score kernel's
//     quad code, so the keys are bit-identical), writing the ordered keys
//     and the unit maxima to the workspace.  Warps 9..15 stage the
//     attention query and the row's K/V page-table entries meanwhile, and
//     attend what needs no ranking: the tail tokens, and -- in a row of at
//     most 512 scored blocks, which keeps every block that has a key, and a
//     cluster of at least 4 CTAs -- all of the row's tokens.
//  B. after a cluster barrier every CTA runs the row's exact top-512 (the
//     top-k kernel's code) into its own shared memory; CTA 0 also writes
//     out_indices.  (A short row is ranked by CTA 0 alone, while the others
//     go straight to the merge.)
//  C. CTA c attends over its ceil(2048/CS) of the selected blocks' entries (16
//     warps, 8 to 128 entries each, walked 32 at a time with the tensor-core
//     walk of the attention kernels), merges its
//     warps into one partial (m, l, acc) per head and pushes each owner CTA
//     its slice of the outputs (remote stores into the owner's shared
//     memory); after a cluster barrier each owner merges its slice over the
//     senders and writes FP16.
//
// Every mbarrier wait is bounded (QSA_DERR_TIMEOUT); every cluster barrier
// is reached by every thread of every CTA of the cluster (the short-row
// choice is the same on every CTA of a row).
#include "qsa_internal.h"
#include "qsa_device.cuh"
#include "qsa_select_impl.cuh"
#include "qsa_fused.h"
#include "qsa_attn_impl.cuh"

#include <mutex>

namespace qsa {
namespace {

constexpr int kFThreads = 512;
constexpr int kFWarps = kFThreads / 32;
constexpr int kFProducerWarp = kScoreWarps;                          // warps 0..7 score
constexpr int kFHelperThreads = kFThreads - (kScoreWarps + 1) * 32;  // warps 9..15
constexpr int kFRingBytes = 4 * kCmpPageKeys * kSelDim * 2;          // 128 KiB in flight
constexpr int kFMaxStages = 8;
constexpr int kFMinCluster = 1;     // CTAs per row's cluster: 1 .. 16, as many as fit
constexpr int kFMaxCluster = 16;
// A short row (at most 512 scored blocks) is attended during the scoring by
// the helper warps of CTAs 1 .. CS-1 when there are at least this many CTAs;
// in smaller clusters it takes the ranked path (phase C on every warp).
constexpr int kFShortRowMinCluster = 4;
// Phase C covers list positions [0, 2048): the expanded blocks.  The tail
// tokens (values >= 4V, at most 3, after the blocks) are attended in phase
// A by one helper warp, so with 16 CTAs every warp walks one 8-token batch.
constexpr int kFBlockEntries = kTokenTopk;
constexpr int kFHelperWarps = kFHelperThreads / 32;   // 7
constexpr int kFTailWarp = kScoreWarps + 1;   // the helper warp that attends the tail
constexpr int kStateFloats = 2 + kAttHeads * 8;   // a lane's WarpState
// Each owner CTA (f0 .. CS-1; f0 = 1 when CTA 0 ranks a short row alone)
// holds a slice of `per` of the row's 3 x 256 outputs, and every sender
// pushes its partial for it into the owner's inbox: m[3], l[3], acc[per]
// at floats [c * stride, (c + 1) * stride), stride = 6 + per.
__host__ __device__ constexpr int inbox_slice(int cs, int f0) {
  return (kAttHeads * kAttDim + (cs - f0) - 1) / (cs - f0);
}
constexpr int inbox_floats_max() {
  int m = 0;
  for (int cs = kFMinCluster; cs <= kFMaxCluster; ++cs)
    for (int f0 = 0; f0 <= (cs >= kFShortRowMinCluster ? 1 : 0); ++f0) {
      const int n = cs * (2 * kAttHeads + inbox_slice(cs, f0));
      m = n > m ? n : m;
    }
  return m;
}
constexpr int kInboxFloats = inbox_floats_max();   // 1048 (4 CTAs, short row)
static_assert(kTopkThreads == kFThreads, "the top-k runs on the whole CTA");
static_assert(kFShortRowMinCluster >= 2, "a short row needs a merging CTA besides CTA 0");
constexpr int kKvPtStaged = 2048;          // K/V page-table entries staged per row

template <bool kFp8>
struct FCfg {
  static constexpr int kPageBytes = KeyCfg<kFp8>::kPageBytes;
  static constexpr int kStages = kFRingBytes / kPageBytes;          // 4 fp16, 8 E4M3 pages
};
static_assert(FCfg<true>::kStages <= kFMaxStages && FCfg<false>::kStages <= kFMaxStages,
              "stage barriers");

// Phase C's shared memory (reuses the ring, as the top-k does in phase B).
struct FusedAttnSmem {
  attn::MergeSmem<kFWarps> merge;
  uint32_t tok[kFWarps][32];
};
static_assert(sizeof(TopkShared) <= (size_t)kFRingBytes, "top-k fits in the ring");
static_assert(sizeof(FusedAttnSmem) <= (size_t)kFRingBytes, "attention fits in the ring");

// Shared memory after the ring (offsets from the 1024-aligned base).
constexpr size_t kOffIdx = kFRingBytes;                                   // int32 [2052]
constexpr size_t kOffQf = kOffIdx + 2052 * 4;                             // QFrag
constexpr size_t kOffKvPt = kOffQf + sizeof(attn::QFrag);                 // int32 [2048]
constexpr size_t kOffInbox = kOffKvPt + kKvPtStaged * 4;                 // float [kInboxFloats]
constexpr size_t kOffState = (kOffInbox + kInboxFloats * 4 + 15) & ~(size_t)15;   // float [7][26][32]
constexpr size_t kOffHTok = kOffState + kFHelperWarps * kStateFloats * 32 * 4;   // uint32 [7][32]
constexpr size_t kOffBars = (kOffHTok + kFHelperWarps * 32 * 4 + 7) & ~(size_t)7;
constexpr size_t kOffCols = kOffBars + 2 * kFMaxStages * 8;               // int [8]
constexpr size_t kFSmem = 1024 + kOffCols + kFMaxStages * 4;
static_assert(kOffQf % 16 == 0 && kOffKvPt % 16 == 0 && kOffInbox % 16 == 0 &&
              kOffState % 16 == 0 && kOffHTok % 16 == 0, "alignment");
static_assert(kFSmem <= 227 * 1024, "fused kernel shared memory");

// --- clusters (sm_90+ PTX) ---------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster; orders each thread's earlier
// memory accesses (shared and global) before the others' later ones.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
// The two halves of cluster_sync_all, for a CTA with work of its own between
// its arrival and the barrier's completion.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The address of this CTA's shared-memory word `local` in CTA `rank`.
__device__ __forceinline__ uint32_t dsmem_map(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_dsmem(uint32_t a, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}

// A lane's WarpState to and from shared memory (column `lane` of [26][32]).
__device__ __forceinline__ void store_state(const attn::WarpState& st, float* sm, int lane) {
  sm[0 * 32 + lane] = st.m_run;
  sm[1 * 32 + lane] = st.l_run;
#pragma unroll
  for (int h = 0; h < kAttHeads; ++h)
#pragma unroll
    for (int d = 0; d < 8; ++d) sm[(2 + 8 * h + d) * 32 + lane] = st.acc[h][d];
}
__device__ __forceinline__ void load_state(attn::WarpState& st, const float* sm, int lane) {
  st.m_run = sm[0 * 32 + lane];
  st.l_run = sm[1 * 32 + lane];
#pragma unroll
  for (int h = 0; h < kAttHeads; ++h)
#pragma unroll
    for (int d = 0; d < 8; ++d) st.acc[h][d] = sm[(2 + 8 * h + d) * 32 + lane];
}

// Resolve a warp's list entries (one per lane, -1 = none) to tokens of the
// K/V cache, compacted in order into tok[]; returns how many.  Holes, tokens
// of unmapped pages and, with skip_from >= 0, entries >= skip_from are left out.
__device__ __forceinline__ int resolve_lane_entries(const AttentionParams& a, int req, bool rok,
                                                    int32_t iv, const int32_t* kvpt_s,
                                                    int64_t skip_from, uint32_t* tok, int lane) {
  if (!rok || (skip_from >= 0 && iv >= skip_from)) iv = -1;
  int32_t pg = -1;
  const int64_t kcol = iv >> 9;
  if (iv >= 0 && kcol < a.pt_cols)
    pg = kcol < kKvPtStaged && kvpt_s ? kvpt_s[kcol]
                                      : __ldg(a.pt + (int64_t)req * a.pt_stride0 + kcol);
  const bool valid = iv >= 0 && pg >= 0 && pg < a.num_pages;
  if (iv >= 0 && !valid) report(a.err, kErrKvPage);
  const unsigned vmask = __ballot_sync(0xffffffffu, valid);
  if (valid)
    tok[__popc(vmask & ((1u << lane) - 1u))] = (uint32_t)pg * kKvPageTokens + (uint32_t)(iv & 511);
  __syncwarp();
  return __popc(vmask);
}

// The CTA's 16 warp states (WarpState layout, in sm) merged into one partial
// per head and pushed to the owners of the output elements -- the cluster's
// CTAs f0 .. CS-1, which are also the senders: element o of the row's
// 3 x 256 goes to CTA f0 + o / per, sender slot c of its inbox; each head's
// (m, l) goes to every owner.  The merge is the log-sum-exp one
// (M = max m_w, weights 2^(m_w - M)).  Every thread of the CTA calls this
// after the warps stored their states; a cluster barrier must follow before
// an owner reads its inbox.
__device__ __forceinline__ void merge_push(attn::MergeSmem<kFWarps>& sm, uint32_t inbox, int c,
                                           int f0, int CS, int tid) {
  const int per = inbox_slice(CS, f0);
  const int stride = 2 * kAttHeads + per;
  __syncthreads();
  if (tid < kAttHeads) {   // head tid: the CTA's (m, l), pushed to every owner, and the
    const int h = tid;     // warps' weights 2^(m_w - M), left in sm.m
    float M = sm.m[0][h];
#pragma unroll
    for (int w = 1; w < kFWarps; ++w) M = fmaxf(M, sm.m[w][h]);
    float Lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kFWarps; ++w) {
      const float cw = M == -CUDART_INF_F ? 0.f : exp2f(sm.m[w][h] - M);
      Lsum = fmaf(cw, sm.l[w][h], Lsum);
      sm.m[w][h] = cw;
    }
    for (int q = f0; q < CS; ++q) {
      st_dsmem(dsmem_map(inbox + 4u * (c * stride + h), (uint32_t)q), M);
      st_dsmem(dsmem_map(inbox + 4u * (c * stride + kAttHeads + h), (uint32_t)q), Lsum);
    }
  }
  __syncthreads();
  for (int o = tid; o < kAttHeads * kAttDim; o += kFThreads) {
    const int h = o / kAttDim, d = o % kAttDim;
    float A = 0.f;
#pragma unroll
    for (int w = 0; w < kFWarps; ++w) A = fmaf(sm.m[w][h], sm.acc[w][h][d], A);
    const int q = o / per;
    st_dsmem(dsmem_map(inbox + 4u * (c * stride + 2 * kAttHeads + (o - q * per)),
                       (uint32_t)(f0 + q)), A);
  }
}

// The owner's slice of the row's output: log-sum-exp merge of the senders'
// (CTAs f0 .. CS-1) partials in its inbox, FP16 round to nearest even.
__device__ __forceinline__ void owner_write(const AttentionParams& a, int r, const float* inbox,
                                            int c, int f0, int CS, int tid) {
  const int per = inbox_slice(CS, f0);
  const int stride = 2 * kAttHeads + per;
  for (int o = (c - f0) * per + tid, t = tid; t < per && o < kAttHeads * kAttDim;
       o += kFThreads, t += kFThreads) {
    const int h = o / kAttDim;
    float M = -CUDART_INF_F;
    for (int q = f0; q < CS; ++q) M = fmaxf(M, inbox[q * stride + h]);
    float A = 0.f, L = 0.f;
    if (M != -CUDART_INF_F) {
      for (int q = f0; q < CS; ++q) {
        const float w = exp2f(inbox[q * stride + h] - M);
        L = fmaf(w, inbox[q * stride + kAttHeads + h], L);
        A = fmaf(w, inbox[q * stride + 2 * kAttHeads + t], A);
      }
    }
    const float inv_l = L > 0.f ? 1.f / L : 0.f;
    a.out[(int64_t)r * kAttHeads * kAttDim + o] = __float2half_rn(A * inv_l);
  }
}

// The warp's state into the CTA's merge space (WarpState layout).
__device__ __forceinline__ void stash_warp(const attn::WarpState& st,
                                           attn::MergeSmem<kFWarps>& sm, int warp, int lane) {
#pragma unroll
  for (int h = 0; h < kAttHeads; ++h)
#pragma unroll
    for (int d = 0; d < 8; ++d) sm.acc[warp][h][8 * lane + d] = st.acc[h][d];
  if (lane < kAttHeads) {
    sm.m[warp][lane] = st.m_run;
    sm.l[warp][lane] = st.l_run;
  }
}

// topk_row's output: the CTA's shared-memory index list, and out_indices
// for the cluster's first CTA.
struct FusedOut {
  int32_t* smem;
  int32_t* global;   // nullptr: shared memory only
  __device__ __forceinline__ void operator()(int j, int32_t v) const {
    smem[j] = v;
    if (global) global[j] = v;
  }
};

template <bool kFp8>
__global__ void __launch_bounds__(kFThreads, 1)
fused_decode_kernel(const SelectParams p, const AttentionParams a,
                    const __grid_constant__ CUtensorMap tmap) {
  constexpr int kPageBytes = FCfg<kFp8>::kPageBytes;
  constexpr int kStages = FCfg<kFp8>::kStages;
  extern __shared__ unsigned char smem_raw[];
  __shared__ int s_abort;
  const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  const uint32_t base = raw + pad;
  unsigned char* gbase = smem_raw + pad;
  TopkShared& tsh = *reinterpret_cast<TopkShared*>(gbase);
  FusedAttnSmem& ash = *reinterpret_cast<FusedAttnSmem*>(gbase);
  int32_t* idx_s = reinterpret_cast<int32_t*>(gbase + kOffIdx);
  attn::QFrag& qf = *reinterpret_cast<attn::QFrag*>(gbase + kOffQf);
  int32_t* kvpt_s = reinterpret_cast<int32_t*>(gbase + kOffKvPt);
  float* inbox_s = reinterpret_cast<float*>(gbase + kOffInbox);
  float* hstate_s = reinterpret_cast<float*>(gbase + kOffState);
  uint32_t* htok_s = reinterpret_cast<uint32_t*>(gbase + kOffHTok);
  int* s_col = reinterpret_cast<int*>(gbase + kOffCols);
  const uint32_t bar_full = base + (uint32_t)kOffBars;
  const uint32_t bar_empty = bar_full + kFMaxStages * 8;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int CS = (int)cluster_size();
  const int c = (int)cluster_rank();
  const int r = (int)cluster_index();            // one cluster per row

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kScoreWarps);
    }
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  const RowSetup rs = row_setup(p, r);
  const int64_t Vs = rs.ok ? (rs.V < p.vcap ? rs.V : p.vcap) : 0;
  const int npages = (int)((Vs + kCmpPageKeys - 1) / kCmpPageKeys);
  const int nmine = c < npages ? (npages - c + CS - 1) / CS : 0;   // pages c, c + CS, ...
  // at most 512 scored blocks: the top-512 keeps every block that has a key,
  // so the attention does not wait for the ranking (the same on every CTA)
  const bool short_row = Vs <= kTopkBlocks && CS >= kFShortRowMinCluster;
  __syncthreads();
  volatile int* abort_flag = &s_abort;
  int issued = 0;
  int withheld = -1;    // test build: the fill that got no copy (never drained)

  // ---- A. scoring --------------------------------------------------------
  if (warp == kFProducerWarp) {
    if (lane == 0) {
      const uint64_t policy = evict_first_policy();
      for (int i = 0; i < nmine; ++i) {
        const int s = i % kStages;
        const uint32_t ph = (uint32_t)((i / kStages) & 1);
        if (i >= kStages && !mbar_wait(bar_empty + 8 * s, ph ^ 1u)) {
          *abort_flag = 1;
          report(p.err, kErrTimeout);
          break;
        }
        if (*abort_flag) break;
        const int col = c + i * CS;
        const int32_t pg = __ldg(p.pt + (int64_t)rs.req * p.pt_stride0 + col);
        issued = i + 1;
        if (pg >= 0 && pg < p.num_pages) {
          s_col[s] = col;
#ifdef QSA_WAIT_TEST
          // test build: leave this fill without a copy (the failure-detection test)
          if (blockIdx.x == 0 && i == p.test_withhold) {
            withheld = i;
            continue;
          }
#endif
          mbar_expect_tx(bar_full + 8 * s, kPageBytes);
          tma_load_2d(base + s * kPageBytes, &tmap, 0,
                      pg * KeyCfg<kFp8>::kRowsPerKey * kCmpPageKeys, bar_full + 8 * s, policy);
        } else {                    // no key for this page's blocks
          s_col[s] = -1 - col;
          report(p.err, kErrCmpPage);
          mbar_arrive(bar_full + 8 * s);
        }
      }
    }
  } else if (warp < kScoreWarps) {
    // warp w scores key groups 2w, 2w + 1 (one unit of 16 keys) of each page
    const int t = lane & 3;
    const int kslot = lane >> 2;
    const int g0 = 2 * warp;
    uint32_t q[kSelHeads][16];
    uint32_t* srow = p.scores + (int64_t)r * p.vcap;
    uint32_t* urow = p.umax + (int64_t)r * (p.vcap / kUnitKeys);
    if (nmine > 0) load_query_slice(p.q_sel + (int64_t)r * kSelHeads * kSelDim, t, q);
    for (int i = 0; i < nmine; ++i) {
      const int s = i % kStages;
      const uint32_t ph = (uint32_t)((i / kStages) & 1);
      if (!mbar_wait(bar_full + 8 * s, ph)) {
        *abort_flag = 1;
        report(p.err, kErrTimeout);
        break;
      }
      const int col = s_col[s];
      const int64_t b0 = (int64_t)(col >= 0 ? col : -1 - col) * kCmpPageKeys;
      const int nk = (int)(Vs - b0 < kCmpPageKeys ? Vs - b0 : kCmpPageKeys);
      if (col >= 0) {
        uint4 kv[2][4];
        load_key_groups<kFp8, 2>(base + s * kPageBytes, g0, t, kslot, kv);
        if (nk > 8 * g0) {
          uint32_t um = 0;
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            const uint32_t key = quad_score(q, kv[g], t);
            const int k = (g0 + g) * 8 + kslot;
            if (k < nk) {
              if (t == 0) srow[b0 + k] = key;
              um = key > um ? key : um;
            }
          }
          um = __reduce_max_sync(0xffffffffu, um);
          if (lane == 0) urow[(b0 + 8 * g0) / kUnitKeys] = um;
        }
      } else if (nk > 8 * g0) {      // an absent page: its blocks get no key
        if (lane < kUnitKeys && 8 * g0 + lane < nk) srow[b0 + 8 * g0 + lane] = 0u;
        if (lane == 0) urow[(b0 + 8 * g0) / kUnitKeys] = 0u;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);
      if (*abort_flag) break;
    }
  } else {
    // helpers: the attention's query fragments and the row's K/V page table;
    // then attention that needs no ranking: the tail tokens (4V .. tail end,
    // known before the selection; the cluster's last CTA) and, in a short
    // row (at most 512 scored blocks, so the top-512 keeps every block whose
    // page is mapped), the tokens of every such block
    const int ht = tid - (kScoreWarps + 1) * 32;
    const int hw = warp - (kScoreWarps + 1);
    attn::stage_query(a, r, qf, ht, kFHelperThreads);
    const bool rok = rs.ok && rs.req < a.num_reqs;
    const int64_t ncols = a.pt_cols < kKvPtStaged ? a.pt_cols : kKvPtStaged;
    for (int64_t j = ht; j < ncols; j += kFHelperThreads)
      kvpt_s[j] = rok ? __ldg(a.pt + (int64_t)rs.req * a.pt_stride0 + j) : -1;
    asm volatile("bar.sync 2, %0;" ::"r"(kFHelperThreads) : "memory");   // qf is staged
    attn::WarpState st;
    attn::init_state(st);
    uint32_t* tok = htok_s + 32 * hw;
    if (short_row && c > 0) {
      // batch i = blocks 2i, 2i + 1 (tokens 8i .. 8i + 7); helper warp gh of
      // CTAs 1 .. CS-1 (CTA 0 ranks the row meanwhile) takes batches gh,
      // gh + (CS - 1) * 7, ...
      const int nb = (int)((Vs + 1) / 2);
      for (int i = (c - 1) * kFHelperWarps + hw; i < nb; i += (CS - 1) * kFHelperWarps) {
        const int64_t b = 2 * (int64_t)i + (lane >> 2);
        bool keyed = false;
        if (lane < 8 && b < Vs) {
          const int32_t pg = __ldg(p.pt + (int64_t)rs.req * p.pt_stride0 + (b >> 7));
          keyed = pg >= 0 && pg < p.num_pages;
        }
        const int32_t iv = keyed ? (int32_t)(8 * i + lane) : -1;
        const int n = resolve_lane_entries(a, rs.req, rok, iv, kvpt_s, -1, tok, lane);
        attn::attend_tokens_mma(a, tok, n, qf, st, lane);
      }
    }
    if (warp == kFTailWarp && c == CS - 1) {
      const int64_t tail0 = rs.V * kRatio;
      const int64_t tail_len = rs.tail_end >= tail0 ? rs.tail_end - tail0 + 1 : 0;
      const int32_t iv = lane < tail_len ? (int32_t)(tail0 + lane) : -1;
      const int n = resolve_lane_entries(a, rs.req, rok, iv, kvpt_s, -1, tok, lane);
      attn::attend_tokens_mma(a, tok, n, qf, st, lane);
    }
    store_state(st, hstate_s + kStateFloats * 32 * hw, lane);
  }
  __syncthreads();
  // After a timeout, let every copy this CTA issued land before the ring's
  // memory is reused.
  if (*abort_flag && warp == kFProducerWarp && lane == 0) {
    for (int n = issued > kStages ? issued - kStages : 0; n < issued; ++n)
      if (n != withheld)
        mbar_wait(bar_full + 8 * (n % kStages), (uint32_t)((n / kStages) & 1), kDrainLimitNs);
  }
  __syncthreads();
  cluster_sync_all();               // every CTA's keys are written and visible

  const uint32_t inbox_a = base + (uint32_t)kOffInbox;
  if (short_row) {
    // ---- B'. every entry is attended already.  CTA 0 ranks the row
    // (out_indices) while CTAs 1 .. CS-1 merge their partials and write the
    // output; it arrives on the merge's cluster barrier first (it sends and
    // owns nothing) and waits on it at the end.
    if (c == 0) {
      cluster_arrive();
      const RowOut out{p.out + (int64_t)r * p.out_stride0};
      if (p.vcap <= kCandCap)
        topk_row<true>(p, r, tsh, out);
      else
        topk_row<false>(p, r, tsh, out);
      cluster_wait();
      return;
    }
    attn::WarpState st;
    if (warp > kScoreWarps)
      load_state(st, hstate_s + kStateFloats * 32 * (warp - kScoreWarps - 1), lane);
    else
      attn::init_state(st);
    attn::finish_mma_state(st, lane);
    stash_warp(st, ash.merge, warp, lane);
    merge_push(ash.merge, inbox_a, c, 1, CS, tid);
    cluster_sync_all();             // every partial is in its owner's inbox
    owner_write(a, r, inbox_s, c, 1, CS, tid);
    return;
  }

  // ---- B. the row's top-512, into shared memory --------------------------
  const FusedOut out{idx_s, c == 0 ? p.out + (int64_t)r * p.out_stride0 : nullptr};
  if (p.vcap <= kCandCap)
    topk_row<true>(p, r, tsh, out);
  else
    topk_row<false>(p, r, tsh, out);
  __syncthreads();                  // the index list is complete

  // ---- C. attention over this CTA's share of the blocks' entries ----------
  // CTA c: entries [c * chunk, (c + 1) * chunk), per_warp of them per warp
  // (8 at CS = 16, 64 at CS = 2), walked 32 at a time
  const int chunk = (kFBlockEntries + CS - 1) / CS;
  const int per_warp = (chunk + kFWarps - 1) / kFWarps;
  const int e1 = min(kFBlockEntries, (c + 1) * chunk);
  const int w0 = c * chunk + warp * per_warp;
  const int w1 = min(e1, w0 + per_warp);
  const bool rok = rs.ok && rs.req < a.num_reqs;
  attn::WarpState st;
  if (warp > kScoreWarps)
    load_state(st, hstate_s + kStateFloats * 32 * (warp - kScoreWarps - 1), lane);
  else
    attn::init_state(st);
  for (int j = w0; j < w1; j += 32) {
    __syncwarp();                   // the last walk has read tok[]
    const int32_t iv = lane < w1 - j ? idx_s[j + lane] : -1;
    // the tail (values >= 4V) was attended in phase A
    const int n = resolve_lane_entries(a, rs.req, rok, iv, kvpt_s, rs.V * kRatio, ash.tok[warp],
                                       lane);
    attn::attend_tokens_mma(a, ash.tok[warp], n, qf, st, lane);
  }
  attn::finish_mma_state(st, lane);
  stash_warp(st, ash.merge, warp, lane);
  merge_push(ash.merge, inbox_a, c, 0, CS, tid);
  cluster_sync_all();               // every partial is in its owner's inbox
  owner_write(a, r, inbox_s, c, 0, CS, tid);
}

template <bool kFp8>
cudaError_t fused_attrs() {
  cudaError_t e = cudaFuncSetAttribute(fused_decode_kernel<kFp8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(fused_decode_kernel<kFp8>,
                              cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

template <bool kFp8>
cudaLaunchConfig_t fused_config(int R, int cs, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(R * cs));
  cfg.blockDim = dim3(kFThreads);
  cfg.dynamicSmemBytes = kFSmem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Per device and key type: how many clusters of cs CTAs the GPU holds at
// once, cs = kFMinCluster .. kFMaxCluster.
struct FusedInfo {
  bool ready = false;
  int maxc[2][kFMaxCluster + 1] = {};
};

cudaError_t fused_info(const FusedInfo** out) {
  static std::mutex mu;
  static FusedInfo info[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  FusedInfo& d = info[dev];
  if (!d.ready) {
    if ((e = fused_attrs<false>()) != cudaSuccess) return e;
    if ((e = fused_attrs<true>()) != cudaSuccess) return e;
    for (int f = 0; f < 2; ++f) {
      for (int cs = kFMinCluster; cs <= kFMaxCluster; ++cs) {
        cudaLaunchAttribute attr[1];
        int n = 0;
        cudaLaunchConfig_t cfg = f ? fused_config<true>(1, cs, nullptr, attr)
                                   : fused_config<false>(1, cs, nullptr, attr);
        e = f ? cudaOccupancyMaxActiveClusters(&n, fused_decode_kernel<true>, &cfg)
              : cudaOccupancyMaxActiveClusters(&n, fused_decode_kernel<false>, &cfg);
        if (e != cudaSuccess) {   // a size the device cannot run: not offered
          cudaGetLastError();
          n = 0;
        }
        d.maxc[f][cs] = n;
      }
    }
    d.ready = true;
  }
  *out = &d;
  return cudaSuccess;
}

}  // namespace

int fused_decode_max_rows(bool key_fp8) {
  const FusedInfo* d = nullptr;
  if (fused_info(&d) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  const int f = key_fp8 ? 1 : 0;
  int n = 0;
  for (int cs = kFMinCluster; cs <= kFMaxCluster; ++cs) n = d->maxc[f][cs] > n ? d->maxc[f][cs] : n;
  return n < kFusedMaxRows ? n : kFusedMaxRows;
}

int fused_decode_cluster(int R, int64_t pt_cols, bool key_fp8) {
  if (R <= 0 || R > kFusedMaxRows) return 0;
  if (pt_cols > (int64_t)kFusedColsPerRow * R) return 0;
  const FusedInfo* d = nullptr;
  if (fused_info(&d) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  const int f = key_fp8 ? 1 : 0;
  for (int cs = kFMaxCluster; cs >= kFMinCluster; --cs) {   // the largest cluster that fits
    if (d->maxc[f][cs] >= R) {
      const int64_t fused = kFusedBaseCost + kFusedPageCost * ((pt_cols + cs - 1) / cs);
      const int64_t chain = kChainBaseCost + kChainPageCost * R * pt_cols;
      return fused <= chain ? cs : 0;
    }
  }
  return 0;
}

cudaError_t launch_fused_decode(const SelectParams& p, const AttentionParams& a,
                                const CUtensorMap& map, int cs, cudaStream_t stream) {
  if (p.R == 0) return cudaSuccess;
  if (cs < kFMinCluster || cs > kFMaxCluster) return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[1];
  cudaError_t e;
  if (p.key_fp8) {
    const cudaLaunchConfig_t cfg = fused_config<true>(p.R, cs, stream, attr);
    e = cudaLaunchKernelEx(&cfg, fused_decode_kernel<true>, p, a, map);
  } else {
    const cudaLaunchConfig_t cfg = fused_config<false>(p.R, cs, stream, attr);
    e = cudaLaunchKernelEx(&cfg, fused_decode_kernel<false>, p, a, map);
  }
  return e;
}

}  // namespace qsa
