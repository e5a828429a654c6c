"""GPU parity for the weighted paged MQA indexer (qsa_paged_mqa_logits, FP8
tensor-core MMAs) and its per-row top-k (qsa_top_k_per_row_decode), through
the C ABI, against oracle/indexer.py.

Logits: every column compared with the binary64 oracle.  The tensor cores
form each q_h . k in fp32 from exact E4M3 products and the head sum is an
fp32 chain, so an element may differ from the oracle by at most
2^-16 x scale x sum_h |w_h| sum_i |q_hi k_i| (a few hundred times the fp32
rounding of a 128-term dot and a 128-term head sum); a wrong lane, head,
block or scale is off by the element's whole size.  -inf columns must match
exactly.  Top-k: bit-exact against the oracle's ranking of the same fp32
logits (the GPU's), on indexer outputs and on synthetic rows with heavy ties,
-inf entries, short rows and a column stride."""
import numpy as np
import pytest
import torch

import sparse_paged_attention_qsa_gb300 as qsa
from oracle import indexer as X
from sparse_paged_attention_qsa_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _gpu_logits(ib, err=None):
    out = qsa.qsa_paged_mqa_logits(ib.q, ib.kv_cache, ib.weights, ib.context_lens,
                                   ib.block_tables, ib.next_n, ib.max_model_len,
                                   block_size=ib.block_size, error_word=err)
    torch.cuda.synchronize()
    return out


def _magnitude(ib, rows):
    """scale_t * sum_h |w_h| * sum_i |q_hi k_i| for the oracle rows."""
    qv = X.e4m3_decode(ib.q.view(torch.uint8).cpu().numpy())
    cache = ib.kv_cache.cpu().numpy()
    bt = ib.block_tables.cpu().numpy()
    w = np.abs(ib.weights.cpu().numpy().astype(np.float64))
    ctx = ib.context_lens.cpu().numpy()
    out = np.zeros((len(rows), ib.max_model_len))
    for i, r in enumerate(rows):
        b = r // ib.next_n
        L = X.row_length(ctx, r, ib.next_n)
        L = min(L, ib.max_model_len)
        for c in range((L + ib.block_size - 1) // ib.block_size):
            blk = int(bt[b, c]) if c < bt.shape[1] else -1
            if not (0 <= blk < cache.shape[0]):
                continue
            vals, sc = X.split_block(cache[blk], ib.block_size, 128)
            t0, t1 = c * ib.block_size, min(L, (c + 1) * ib.block_size)
            k = np.abs(X.e4m3_decode(vals[:t1 - t0]))
            out[i, t0:t1] = np.abs(sc[:t1 - t0]) * ((k @ np.abs(qv[r]).T) @ w[r])
    return out


def _check_logits(ib, rows=None, expect_err=0):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = _gpu_logits(ib, err).cpu().numpy()
    rows = list(range(got.shape[0])) if rows is None else list(rows)
    exp, oerr = X.paged_mqa_logits(ib.q.view(torch.uint8).cpu().numpy(), ib.kv_cache.cpu().numpy(),
                                   ib.weights.cpu().numpy(), ib.context_lens.cpu().numpy(),
                                   ib.block_tables.cpu().numpy(), ib.next_n, ib.max_model_len,
                                   ib.block_size, rows=rows)
    g = got[rows]
    assert np.array_equal(np.isneginf(g), np.isneginf(exp)), \
        np.nonzero(np.isneginf(g) != np.isneginf(exp))
    fin = np.isfinite(exp)
    tol = 2.0 ** -16 * _magnitude(ib, rows) + 1e-30
    diff = np.zeros_like(exp)
    diff[fin] = np.abs(g[fin] - exp[fin])
    bad = fin & (diff > tol)
    assert not bad.any(), (np.argwhere(bad)[:5], g[bad][:5], exp[bad][:5])
    assert (int(err.item()) != 0) == (oerr != 0) and (int(err.item()) & ~16) == 0
    return got


@pytest.mark.parametrize("heads,next_n,bs", [(64, 1, 64), (64, 2, 64), (16, 4, 8), (128, 2, 128),
                                             (32, 3, 16), (128, 1, 32)])
def test_logits_ragged_contexts(heads, next_n, bs):
    ctx = [1, 63, 64, 65, 127, 128, 129, 700, 4, 1500]
    ib = W.indexer_batch("ragged", ctx, next_n=next_n, heads=heads, block_size=bs,
                         max_model_len=1600, seed=heads + next_n + bs, device=DEV)
    _check_logits(ib)


def test_logits_empty_and_short_requests():
    ctx = [0, 1, 2, 3, 0, 200]
    ib = W.indexer_batch("short", ctx, next_n=3, heads=64, block_size=64, max_model_len=256,
                         seed=7, device=DEV)
    _check_logits(ib)


def test_logits_bad_blocks_and_short_tables():
    ib = W.indexer_batch("bad", [300, 500, 257], next_n=2, heads=64, block_size=64,
                         max_model_len=600, seed=8, device=DEV)
    bt = ib.block_tables.clone()
    bt[0, 1] = -1
    bt[1, 3] = ib.kv_cache.shape[0] + 7
    ib2 = W.IndexerBatch(**{**ib.__dict__, "block_tables": bt[:, :5].contiguous()})
    ib2.context_lens[1] = 500                      # needs 8 columns: 5..7 are past the table
    _check_logits(ib2)


def test_logits_many_tiles_and_requests():
    # more tiles than CTAs: the per-CTA ranges cross requests; sampled rows
    rng = np.random.default_rng(3)
    ctx = [int(x) for x in rng.integers(1, 9000, size=40)]
    ib = W.indexer_batch("many", ctx, next_n=2, heads=64, block_size=64, max_model_len=9000,
                         seed=9, device=DEV)
    _check_logits(ib, rows=[0, 1, 17, 38, 51, 79])


def test_logits_long_context_sampled_rows():
    ib = W.indexer_batch("long", [65536, 40000, 65536, 1], next_n=1, heads=64, block_size=64,
                         max_model_len=65536, seed=10, device=DEV)
    _check_logits(ib, rows=[0, 1, 3])


# ---- top-k ------------------------------------------------------------------

def _check_topk(logits, next_n, seq_lens, topk, rows=None):
    got = qsa.qsa_top_k_per_row_decode(logits, next_n, seq_lens, topk)
    torch.cuda.synchronize()
    lg = logits.float().cpu().numpy()
    exp = X.top_k_per_row(lg, next_n, seq_lens.cpu().numpy(), topk, rows=rows)
    g = got.cpu().numpy()
    g = g if rows is None else g[rows]
    for i in range(exp.shape[0]):
        assert np.array_equal(g[i], exp[i]), (i, np.nonzero(g[i] != exp[i])[0][:5])
    return got


def test_topk_on_indexer_logits():
    ib = W.indexer_batch("tk", [5000, 2048, 2047, 30000, 1, 0], next_n=2, heads=64,
                         block_size=64, max_model_len=30000, seed=11, device=DEV)
    lg = _gpu_logits(ib)
    _check_topk(lg, 2, ib.context_lens, 2048)
    _check_topk(lg, 2, ib.context_lens, 1)
    _check_topk(lg, 2, ib.context_lens, 777)


def test_topk_on_tied_indexer_logits():
    ib = W.indexer_batch("tk_ties", [9000, 4000], next_n=1, heads=16, block_size=64,
                         max_model_len=9000, tie_values=5, seed=12, device=DEV)
    lg = _gpu_logits(ib)
    _check_topk(lg, 1, ib.context_lens, 2048)


@pytest.mark.parametrize("distinct,cols,topk", [(0, 70000, 2048), (3, 10000, 2048), (1, 5000, 100),
                                                (50, 4096, 2048), (0, 2100, 2048),
                                                # heavy ties on long rows: more candidates than the
                                                # kernel keeps on chip (its fallback path)
                                                (2, 30000, 2048), (1, 12000, 64), (0, 131072, 1)])
def test_topk_synthetic_rows(distinct, cols, topk):
    g = torch.Generator(device=DEV).manual_seed(distinct + cols)
    rows, next_n = 6, 3
    if distinct:
        vals = torch.randn(distinct, device=DEV, generator=g)
        lg = vals[torch.randint(0, distinct, (rows, cols), device=DEV, generator=g)]
    else:
        lg = torch.randn(rows, cols, device=DEV, generator=g)
    lg[0, ::7] = -float("inf")
    lg[1, :100] = 0.0
    lg[1, 100:200] = -0.0
    seq = torch.tensor([cols, cols // 2], dtype=torch.int32, device=DEV)
    _check_topk(lg.contiguous(), next_n, seq, topk)


def test_topk_strided_columns_and_short_rows():
    g = torch.Generator(device=DEV).manual_seed(5)
    base = torch.randn(4, 6000, device=DEV, generator=g)
    view = base[:, ::2]                                  # stride1 = 2
    seq = torch.tensor([3000, 10, 1, 2500], dtype=torch.int32, device=DEV)
    _check_topk(view, 1, seq, 2048)
    _check_topk(view, 1, seq, 5)


def test_topk_sample_skew_and_alignment():
    # Rows built against the kernel's sampled threshold (32-column chunks at
    # multiples of L // 256): large logits exactly on the sampled chunks
    # (too few candidates), large logits only between them (too many), an
    # increasing row, and a row whose start is not 16-byte aligned.
    L = 65536
    g = torch.Generator(device=DEV).manual_seed(21)
    lg = torch.randn(5, L + 3, device=DEV, generator=g) * 0.01
    stride = L // 256
    cols = (torch.arange(256, device=DEV)[:, None] * stride + torch.arange(32, device=DEV)).flatten()
    lg[0, cols] += 10.0
    off = torch.ones(L + 3, dtype=torch.bool, device=DEV)
    off[cols] = False
    lg[1, off] += 10.0
    lg[2] = torch.arange(L + 3, device=DEV, dtype=torch.float32) * 1e-3
    seq = torch.full((5,), L, dtype=torch.int32, device=DEV)
    _check_topk(lg[:, :L], 1, seq, 2048)                  # row stride L + 3: rows 1.. misaligned
    _check_topk(lg[:, :L].contiguous(), 1, seq, 2048)
    seq_t = torch.tensor([L - 1, L - 2, L - 3, 40000, 10241], dtype=torch.int32, device=DEV)
    _check_topk(lg[:, :L].contiguous(), 1, seq_t, 2048)   # float4 tails of 1..3 columns
    _check_topk(lg[:, :L].contiguous(), 1, seq_t, 3)
