"""Seeded synthetic inputs shaped like the QSA decode workloads.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no visible-block rule, no scoring, no paging).  Both the
CUDA path and the CPU oracle receive the same tensors from here.

Layouts follow "vLLM: integrate FP16 packed QSA extension", "Exact contracts":
  q_sel       FP16 [R,4,128]
  cmp_cache   FP16 [P,128,1,128]       (128 compressed keys per page)
  q_attn      FP16 [R,3,256]
  kv_cache    FP16 [Pkv,512,2,256]     exact-packed: per token K = halves
                                       0..255, V = halves 256..511 (the same
                                       bytes as [Pkv,512,1,512]); the op sees
                                       K/V as the views kv[:,:,0:1] and
                                       kv[:,:,1:2], strides [262144,512,256,1],
                                       V at storage offset 256
  page tables int32 [num_reqs, cols] (-1 = unused column)
  token_to_request int32 [R], seq_lens int32 [num_reqs],
  query_positions int64 [R]
  query_start_loc int32 [num_reqs+1] (batches with several query tokens per
                  request: request i owns rows query_start_loc[i] ..
                  query_start_loc[i+1]-1; its token_to_request and
                  query_positions are then left to the metadata builder)

Structure (sequence lengths, page tables, premade index lists) is drawn from
a CPU generator seeded with ``seed``; values (queries, keys, K/V) from a
generator on the target device seeded with ``seed + 1``.  Structure is
therefore identical on every device; values depend on the device's RNG.
Large pools are filled in fixed-size chunks so the draw is reproducible.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

CMP_PAGE = 128          # compressed keys per page
KV_PAGE = 512           # tokens per K/V page
SEL_HEADS, SEL_DIM = 4, 128
ATT_HEADS, ATT_DIM = 3, 256
OUT_WIDTH = 2051
_CHUNK = 1 << 26        # elements per fill chunk


@dataclass
class Workload:
    name: str
    R: int
    q_sel: torch.Tensor
    cmp_cache: torch.Tensor
    cmp_page_table: torch.Tensor
    token_to_request: torch.Tensor | None
    seq_lens: torch.Tensor
    query_positions: torch.Tensor | None
    q_attn: torch.Tensor
    kv_cache: torch.Tensor
    kv_page_table: torch.Tensor
    indices: torch.Tensor | None = None    # premade attention index lists
    meta: dict = field(default_factory=dict)
    query_start_loc: torch.Tensor | None = None   # multi-token batches

    @property
    def k_view(self) -> torch.Tensor:
        """K view [Pkv,512,1,256], strides [262144,512,256,1], offset 0."""
        return self.kv_cache[:, :, 0:1, :]

    @property
    def v_view(self) -> torch.Tensor:
        """V view [Pkv,512,1,256], strides [262144,512,256,1], offset 256."""
        return self.kv_cache[:, :, 1:2, :]

    def to(self, device) -> "Workload":
        kw = {}
        for k, v in self.__dict__.items():
            kw[k] = v.to(device) if isinstance(v, torch.Tensor) else v
        return Workload(**kw)


def _fill_normal(shape, std: float, gen: torch.Generator, device,
                 dtype=torch.float16) -> torch.Tensor:
    """fp32 N(0, std^2) draws rounded to `dtype`, filled chunk by chunk."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        x = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        flat[s:e].copy_(x)
    return out


def _randint(lo: int, hi: int, n: int, gen: torch.Generator) -> list[int]:
    """n integers uniform in [lo, hi] inclusive."""
    return torch.randint(lo, hi + 1, (n,), generator=gen).tolist()


def _pages_for(n_items: int, per_page: int) -> int:
    return (n_items + per_page - 1) // per_page


def build(name: str, seq_lens: list[int], *, positions: list[int] | None = None,
          cmp_pool: int | None = None, kv_pool: int | None = None,
          cmp_cols: int | None = None, kv_cols: int | None = None,
          cmp_std: float = 0.1, distinct_keys: int = 0,
          dup_mapping: bool = False, premade_widths: list[int] | None = None,
          hole_frac: float = 0.10, dup_frac: float = 0.05,
          cmp_dtype: str = "fp16", query_lens: list[int] | None = None,
          seed: int = 0, device="cpu") -> Workload:
    """General builder: one request per row (token_to_request = arange(R)).

    ``query_lens`` instead gives request i query_lens[i] consecutive rows
    (speculative / multi-token decode and prefill chunks; 0 = a request with
    no rows): R = sum(query_lens), ``query_start_loc`` is their running sum,
    and token_to_request / query_positions stay None for the metadata
    builder to fill.

    ``positions`` default to seq_len-1 (plain decode).  Each request gets the
    compressed pages its seq_len needs (seq_len // 4 keys, 128 per page) and
    the K/V pages its tokens need (512 per page), drawn without replacement
    from one random permutation of each pool.  ``distinct_keys`` > 0 fills the
    compressed pool with copies of that many random vectors (exact score
    ties).  ``dup_mapping`` makes request 0 map one physical compressed and
    K/V page into two of its logical columns and request 1 map one page that
    request 0 also uses.  ``premade_widths`` builds attention index lists
    (valid widths cycled over rows; holes and duplicates as in the stress
    workload) instead of relying on the selection output.  ``cmp_dtype``
    "fp8" stores the compressed keys as FP8 E4M3 (torch.float8_e4m3fn, the
    same draws rounded to E4M3) -- the optional e4m3 compressed indexer
    cache.
    """
    if cmp_dtype not in ("fp16", "fp8"):
        raise ValueError("cmp_dtype must be 'fp16' or 'fp8'")
    kdt = torch.float8_e4m3fn if cmp_dtype == "fp8" else torch.float16
    nreq = len(seq_lens)
    if query_lens is not None:
        if len(query_lens) != nreq or positions is not None or premade_widths:
            raise ValueError("query_lens: one per request, no positions / premade lists")
        R = int(sum(query_lens))
    else:
        R = nreq
    sg = torch.Generator().manual_seed(seed)
    if positions is None and query_lens is None:
        positions = [L - 1 for L in seq_lens]
    cmp_need = [_pages_for(max(L, 0) // 4, CMP_PAGE) for L in seq_lens]
    kv_need = [_pages_for(max(L, 0), KV_PAGE) for L in seq_lens]
    extra = 2 if dup_mapping else 0
    cmp_cols = cmp_cols or max(1, max(cmp_need) + extra)
    kv_cols = kv_cols or max(1, max(kv_need) + extra)
    cmp_pool = cmp_pool or max(1, sum(cmp_need))
    kv_pool = kv_pool or max(1, sum(kv_need))
    if sum(cmp_need) > cmp_pool or sum(kv_need) > kv_pool:
        raise ValueError("pool too small for the requested sequence lengths")

    def tables(need, pool, cols):
        perm = torch.randperm(pool, generator=sg).tolist()
        pt = torch.full((nreq, cols), -1, dtype=torch.int32)
        at = 0
        for r, n in enumerate(need):
            if n:
                pt[r, :n] = torch.tensor(perm[at:at + n], dtype=torch.int32)
            at += n
        return pt

    cmp_pt = tables(cmp_need, cmp_pool, cmp_cols)
    kv_pt = tables(kv_need, kv_pool, kv_cols)
    if dup_mapping and nreq >= 2:
        for pt, need in ((cmp_pt, cmp_need), (kv_pt, kv_need)):
            if need[0] >= 2:
                pt[0, 1] = pt[0, 0]              # request 0: one page, two columns
            if need[0] >= 1 and need[1] >= 1:
                pt[1, 0] = pt[0, 0]              # request 1 shares request 0's page

    indices = None
    if premade_widths:
        indices = torch.full((R, OUT_WIDTH), -1, dtype=torch.int32)
        for r in range(R):
            L = seq_lens[r]
            w = premade_widths[r % len(premade_widths)]
            if w == 0 or L <= 0:
                continue
            ndist = min(w, L)
            toks = torch.randperm(L, generator=sg)[:ndist]
            if ndist < w:
                fill = toks[torch.randint(0, ndist, (w - ndist,), generator=sg)]
                toks = torch.cat([toks, fill])
            toks = toks[torch.randperm(w, generator=sg)].to(torch.int32)
            n_dup = int(round(dup_frac * w))
            if n_dup and w > 1:
                dst = torch.randperm(w, generator=sg)[:n_dup]
                src = torch.randint(0, w, (n_dup,), generator=sg)
                toks[dst] = toks[src]
            n_hole = int(round(hole_frac * w))
            if n_hole:
                toks[torch.randperm(w, generator=sg)[:n_hole]] = -1
            indices[r, :w] = toks

    vg = torch.Generator(device=device).manual_seed(seed + 1)
    q_sel = _fill_normal((R, SEL_HEADS, SEL_DIM), 1.0, vg, device)
    if distinct_keys:
        vecs = _fill_normal((distinct_keys, SEL_DIM), cmp_std, vg, device, kdt)
        pick = torch.randint(0, distinct_keys, (cmp_pool * CMP_PAGE,), generator=sg)
        cmp = vecs.view(torch.uint8 if kdt != torch.float16 else kdt)[pick.to(device)]
        cmp = cmp.view(kdt).view(cmp_pool, CMP_PAGE, 1, SEL_DIM).contiguous()
    else:
        cmp = _fill_normal((cmp_pool, CMP_PAGE, 1, SEL_DIM), cmp_std, vg, device, kdt)
    q_attn = _fill_normal((R, ATT_HEADS, ATT_DIM), 1.0, vg, device)
    kv = _fill_normal((kv_pool, KV_PAGE, 2, ATT_DIM), 1.0, vg, device)

    qsl = None
    if query_lens is not None:
        qsl = torch.zeros(nreq + 1, dtype=torch.int32)
        qsl[1:] = torch.tensor(query_lens, dtype=torch.int32).cumsum(0)
    return Workload(
        name=name, R=R, q_sel=q_sel, cmp_cache=cmp,
        cmp_page_table=cmp_pt.to(device),
        token_to_request=None if qsl is not None else
        torch.arange(R, dtype=torch.int32).to(device),
        seq_lens=torch.tensor(seq_lens, dtype=torch.int32).to(device),
        query_positions=None if qsl is not None else
        torch.tensor(positions, dtype=torch.int64).to(device),
        q_attn=q_attn, kv_cache=kv, kv_page_table=kv_pt.to(device),
        indices=indices.to(device) if indices is not None else None,
        meta={"seed": seed, "cmp_pool": cmp_pool, "kv_pool": kv_pool},
        query_start_loc=qsl.to(device) if qsl is not None else None)


# --- the five named workloads ------------------------------------------------

CONFIG_NAMES = {
    0: "R1_L519_cross_page_tail",
    1: "R1_L9215_P8192_saturated",
    2: "R64_L512-65536_decode_batch",
    3: "R16_L300-20000_tie_dup_hole_stress",
    4: "R256_L131072_long_context",
}


def config(cfg: int, device="cpu", seed: int | None = None, rows: int | None = None,
           cmp_dtype: str = "fp16") -> Workload:
    """The five workloads (seed 1000+cfg unless given).  ``rows`` truncates a
    multi-row workload to its first rows (structure drawn for all rows first,
    so the kept rows are identical to the full workload's structure) -- only
    used to size CPU-side checks; values are drawn for the kept rows only."""
    seed = 1000 + cfg if seed is None else seed
    name = CONFIG_NAMES[cfg]
    if cfg == 0:
        # 519 tokens: 129 visible blocks over 2 compressed pages + 3-token tail;
        # pools of 8 compressed / 4 K/V pages, tables a permutation of the pool.
        return _permuted_single(name, 519, 8, 4, seed, device, cmp_dtype)
    if cfg == 1:
        # 9215 tokens: 2303 visible blocks (18 pages) in a pool of 8192;
        # K/V pool of 64 pages, 18 in use.
        return build(name, [9215], cmp_pool=8192, kv_pool=64, cmp_dtype=cmp_dtype, seed=seed,
                     device=device)
    if cfg == 2:
        sg = torch.Generator().manual_seed(seed + 7)
        L = _randint(512, 65536, 64, sg)
        if rows:
            L = L[:rows]
        return build(name, L, cmp_pool=16384, kv_pool=8192, cmp_cols=128, kv_cols=128,
                     cmp_dtype=cmp_dtype, seed=seed, device=device)
    if cfg == 3:
        sg = torch.Generator().manual_seed(seed + 7)
        L = _randint(300, 20000, 16, sg)
        if rows:
            L = L[:rows]
        need_c = sum(_pages_for(x // 4, CMP_PAGE) for x in L)
        need_k = sum(_pages_for(x, KV_PAGE) for x in L)
        return build(name, L, cmp_pool=need_c + 16, kv_pool=need_k + 16, distinct_keys=4,
                     dup_mapping=True, premade_widths=[0, 1, 32, 1024, 2051],
                     cmp_dtype=cmp_dtype, seed=seed, device=device)
    if cfg == 4:
        R = rows or 256
        return build(name, [131072] * R, cmp_pool=256 * R, kv_pool=256 * R,
                     cmp_dtype=cmp_dtype, seed=seed, device=device)
    raise ValueError(f"unknown workload {cfg}")


def _permuted_single(name, L, cmp_pool, kv_pool, seed, device, cmp_dtype="fp16") -> Workload:
    """One row whose page tables are full random permutations of small pools."""
    sg = torch.Generator().manual_seed(seed)
    cmp_pt = torch.randperm(cmp_pool, generator=sg).to(torch.int32).view(1, -1)
    kv_pt = torch.randperm(kv_pool, generator=sg).to(torch.int32).view(1, -1)
    vg = torch.Generator(device=device).manual_seed(seed + 1)
    q_sel = _fill_normal((1, SEL_HEADS, SEL_DIM), 1.0, vg, device)
    kdt = torch.float8_e4m3fn if cmp_dtype == "fp8" else torch.float16
    cmp = _fill_normal((cmp_pool, CMP_PAGE, 1, SEL_DIM), 0.1, vg, device, kdt)
    q_attn = _fill_normal((1, ATT_HEADS, ATT_DIM), 1.0, vg, device)
    kv = _fill_normal((kv_pool, KV_PAGE, 2, ATT_DIM), 1.0, vg, device)
    return Workload(
        name=name, R=1, q_sel=q_sel, cmp_cache=cmp, cmp_page_table=cmp_pt.to(device),
        token_to_request=torch.zeros(1, dtype=torch.int32, device=device),
        seq_lens=torch.tensor([L], dtype=torch.int32, device=device),
        query_positions=torch.tensor([L - 1], dtype=torch.int64, device=device),
        q_attn=q_attn, kv_cache=kv, kv_page_table=kv_pt.to(device),
        meta={"seed": seed, "cmp_pool": cmp_pool, "kv_pool": kv_pool})



# --- weighted paged MQA indexer (DeepSeek-V3.2 style) -----------------------

IDX_DIM = 128


@dataclass
class IndexerBatch:
    """Inputs of the indexer decode step: rows r = b*next_n + j.

    q             float8_e4m3fn [rows, heads, 128]
    kv_cache      uint8 [num_blocks, block_size*132]: per block the tokens'
                  128 E4M3 value bytes, then their fp32 scales
    weights       float32 [rows, heads]
    context_lens  int32 [batch]
    block_tables  int32 [batch, cols] (-1 = unused column)
    """
    name: str
    q: torch.Tensor
    kv_cache: torch.Tensor
    weights: torch.Tensor
    context_lens: torch.Tensor
    block_tables: torch.Tensor
    next_n: int
    block_size: int
    max_model_len: int
    meta: dict = field(default_factory=dict)


def indexer_batch(name: str, context_lens: list[int], *, next_n: int = 1, heads: int = 64,
                  block_size: int = 64, max_model_len: int | None = None,
                  extra_blocks: int = 3, tie_values: int = 0, seed: int = 0,
                  device="cpu") -> IndexerBatch:
    """Seeded indexer inputs.  Query values ~ N(0, 2^2), key values
    ~ N(0, 16^2), both rounded to E4M3; key scales ~ U[0.005, 0.05]; head
    weights ~ N(0, 1/8^2).  Each request's blocks are drawn without
    replacement from one random permutation of the pool (``extra_blocks``
    spare blocks).  ``tie_values`` > 0 draws every key from that many random
    vectors with one common scale (exact logit ties)."""
    B = len(context_lens)
    rows = B * next_n
    sg = torch.Generator().manual_seed(seed)
    need = [(max(c, 0) + block_size - 1) // block_size for c in context_lens]
    nblocks = max(1, sum(need) + extra_blocks)
    cols = max(1, max(need))
    perm = torch.randperm(nblocks, generator=sg)
    bt = torch.full((B, cols), -1, dtype=torch.int32)
    at = 0
    for b, n in enumerate(need):
        if n:
            bt[b, :n] = perm[at:at + n].to(torch.int32)
        at += n
    vg = torch.Generator(device=device).manual_seed(seed + 1)
    q = (torch.randn((rows, heads, IDX_DIM), generator=vg, device=device) * 2.0).to(
        torch.float8_e4m3fn)
    w = torch.randn((rows, heads), generator=vg, device=device) / 8.0
    ntok = nblocks * block_size
    if tie_values:
        vecs = (torch.randn((tie_values, IDX_DIM), generator=vg, device=device) * 16.0).to(
            torch.float8_e4m3fn)
        pick = torch.randint(0, tie_values, (ntok,), generator=sg).to(device)
        vals = vecs.view(torch.uint8)[pick]
        scales = torch.full((ntok,), 0.02, dtype=torch.float32, device=device)
    else:
        vals = (torch.randn((ntok, IDX_DIM), generator=vg, device=device) * 16.0).to(
            torch.float8_e4m3fn).view(torch.uint8)
        scales = torch.rand((ntok,), generator=vg, device=device) * 0.045 + 0.005
    cache = torch.empty((nblocks, block_size * (IDX_DIM + 4)), dtype=torch.uint8, device=device)
    cache[:, :block_size * IDX_DIM] = vals.view(nblocks, block_size * IDX_DIM)
    cache[:, block_size * IDX_DIM:] = scales.view(nblocks, block_size).contiguous().view(
        torch.uint8).view(nblocks, block_size * 4)
    mml = max_model_len or max(1, max(context_lens))
    return IndexerBatch(name=name, q=q, kv_cache=cache, weights=w,
                        context_lens=torch.tensor(context_lens, dtype=torch.int32).to(device),
                        block_tables=bt.to(device), next_n=next_n, block_size=block_size,
                        max_model_len=mml, meta={"seed": seed, "blocks": nblocks})
