"""Pins for the weighted paged MQA indexer oracle (oracle/indexer.py).

Independent checks:
  * E4M3 decoding against torch.float8_e4m3fn (a library routine);
  * the cache-block layout against a block assembled by hand;
  * closed forms: one-hot queries/keys, keys that encode their own logical
    index (pins the block-table lookup, the slot and the per-row causal
    length), scale and weight linearity, sign of weights;
  * exact rational arithmetic (fractions) on random small cases: the
    binary64 logits agree to rounding of the final head sum;
  * reduction to the QSA selection score: 4 heads, unit weights and scale,
    exactly summable values give the canonical binary32 score bit for bit;
  * top-k: brute-force rank (no sort) with heavy ties, short rows, -inf
    entries, per-row causal lengths.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import indexer as X

D = 128


def _e4m3(x) -> np.ndarray:
    """float values exactly representable in E4M3 -> codes."""
    t = torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    assert torch.equal(t.to(torch.float32), torch.tensor(np.asarray(x, dtype=np.float32)))
    return t.view(torch.uint8).numpy()


def _block(vals_codes, scales):
    """Assemble one cache block by hand: value rows, then fp32 scales."""
    vals_codes = np.asarray(vals_codes, dtype=np.uint8)
    return np.concatenate([vals_codes.reshape(-1),
                           np.asarray(scales, dtype=np.float32).view(np.uint8)])


def test_e4m3_decode_matches_library():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = X.e4m3_decode(codes)
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok]) and np.isnan(got[~ok]).all()


def test_block_layout():
    bs = 4
    vals = np.stack([np.full(D, t + 1, np.uint8) for t in range(bs)])
    blk = _block(vals, [0.5, 1.5, 2.5, 3.5])
    assert blk.size == bs * (D + 4)
    v, s = X.split_block(blk, bs, D)
    assert np.array_equal(v, vals) and s.tolist() == [0.5, 1.5, 2.5, 3.5]


def _cache_from_keys(keys_codes, scales, block_size, perm):
    """Logical tokens -> blocks placed at physical ids perm[c]; returns the
    cache [num_blocks, block_size*(D+4)] and one request's block table."""
    n = len(keys_codes)
    nb = (n + block_size - 1) // block_size
    cache = np.zeros((max(perm) + 1, block_size * (D + 4)), np.uint8)
    for c in range(nb):
        v = np.zeros((block_size, D), np.uint8)
        s = np.zeros(block_size, np.float32)
        seg = keys_codes[c * block_size:(c + 1) * block_size]
        v[:len(seg)] = seg
        s[:len(seg)] = scales[c * block_size:(c + 1) * block_size]
        cache[perm[c]] = _block(v, s)
    return cache, np.array([perm[:nb]], dtype=np.int32)


@pytest.mark.parametrize("block_size,next_n", [(64, 1), (64, 2), (16, 3)])
def test_keys_encoding_their_index_pin_paging_and_lengths(block_size, next_n):
    # token t: key = one-hot at dim t % D with value 1, scale t + 1; q all
    # ones, one head, weight w_r -> logit(r, t) = (t + 1) * w_r for t < L_r
    L = 300
    keys = np.zeros((L, D), np.float32)
    keys[np.arange(L), np.arange(L) % D] = 1.0
    scales = np.arange(1, L + 1, dtype=np.float32)
    rng = np.random.default_rng(block_size + next_n)
    nb = (L + block_size - 1) // block_size
    perm = rng.permutation(nb + 5)[:nb].tolist()
    cache, bt = _cache_from_keys(_e4m3(keys), scales, block_size, perm)
    q = _e4m3(np.ones((next_n, 1, D), np.float32))
    w = np.array([[2.0 + j] for j in range(next_n)], np.float32)
    lg, err = X.paged_mqa_logits(q, cache, w, [L], bt, next_n, 400, block_size)
    assert err == 0
    for j in range(next_n):
        Lr = L - next_n + j + 1
        assert np.array_equal(lg[j, :Lr], (np.arange(Lr) + 1) * (2.0 + j))
        assert np.isneginf(lg[j, Lr:]).all()


def test_one_hot_closed_form_and_linearity():
    H = 5
    q = np.zeros((1, H, D), np.float32)
    k = np.zeros((1, D), np.float32)
    q[0, np.arange(H), [3, 3, 7, 100, 3]] = [2.0, -1.5, 4.0, 0.25, 448.0]
    k[0, [3, 7, 100]] = [0.5, -3.0, 8.0]
    w = np.array([[1.0, 2.0, -0.5, 3.0, 0.125]], np.float32)
    cache, bt = _cache_from_keys(_e4m3(k), np.array([0.75], np.float32), 64, [0])
    lg, _ = X.paged_mqa_logits(_e4m3(q), cache, w, [1], bt, 1, 1, 64)
    dots = [2.0 * 0.5, -1.5 * 0.5, 4.0 * -3.0, 0.25 * 8.0, 448.0 * 0.5]
    exp = 0.75 * sum(wh * max(d, 0.0) for wh, d in zip(w[0], dots))
    assert lg[0, 0] == exp
    # scale and weights enter linearly
    cache2, _ = _cache_from_keys(_e4m3(k), np.array([1.5], np.float32), 64, [0])
    lg2, _ = X.paged_mqa_logits(_e4m3(q), cache2, 2 * w, [1], bt, 1, 1, 64)
    assert lg2[0, 0] == 4 * exp


@pytest.mark.parametrize("seed", range(4))
def test_exact_rational_reference(seed):
    rng = np.random.default_rng(seed)
    H, L, bs = 3, 70, 32
    qf = torch.randn(1, H, D, generator=torch.Generator().manual_seed(seed)).to(
        torch.float8_e4m3fn)
    kf = (torch.randn(L, D, generator=torch.Generator().manual_seed(seed + 50)) * 0.3).to(
        torch.float8_e4m3fn)
    scales = rng.uniform(0.01, 2.0, size=L).astype(np.float32)
    w = rng.normal(size=(1, H)).astype(np.float32)
    cache, bt = _cache_from_keys(kf.view(torch.uint8).numpy(), scales, bs,
                                 rng.permutation(3).tolist())
    lg, _ = X.paged_mqa_logits(qf.view(torch.uint8).numpy(), cache, w, [L], bt, 1, L, bs)
    qd, kd = qf.to(torch.float64).numpy(), kf.to(torch.float64).numpy()
    for t in range(L):
        dots = [sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(qd[0, h], kd[t]))
                for h in range(H)]
        exact = Fraction(float(scales[t])) * sum(Fraction(float(w[0, h])) * max(dots[h], 0)
                                                 for h in range(H))
        mag = abs(float(scales[t])) * sum(abs(float(w[0, h])) * abs(float(dots[h]))
                                         for h in range(H))
        assert abs(lg[0, t] - float(exact)) <= 8 * 2.0 ** -53 * mag + 1e-300


def test_reduces_to_the_qsa_selection_score():
    # 4 heads, unit weights and scale, small integers (exact in E4M3, fp16
    # and every binary32 partial sum): the canonical binary32 score
    rng = np.random.default_rng(3)
    for _ in range(20):
        q = rng.integers(-4, 5, size=(4, D)).astype(np.float32)
        k = rng.integers(-4, 5, size=(1, D)).astype(np.float32)
        cache, bt = _cache_from_keys(_e4m3(k), np.ones(1, np.float32), 64, [0])
        lg, _ = X.paged_mqa_logits(_e4m3(q[None]), cache, np.ones((1, 4), np.float32),
                                   [1], bt, 1, 1, 64)
        s = oracle.score_e4m3(q.astype(np.float16), _e4m3(k[0]))
        assert np.float32(lg[0, 0]) == s


def test_bad_blocks_give_minus_inf_and_an_error_bit():
    L, bs = 100, 32
    keys = np.ones((L, D), np.float32)
    cache, bt = _cache_from_keys(_e4m3(keys), np.ones(L, np.float32), bs, [0, 1, 2, 3])
    bt = bt.copy()
    bt[0, 1] = -1
    bt[0, 2] = 99
    lg, err = X.paged_mqa_logits(_e4m3(np.ones((1, 1, D), np.float32)), cache,
                                 np.ones((1, 1), np.float32), [L], bt, 1, L, bs)
    assert err == X.ERR_BLOCK
    assert np.isneginf(lg[0, 32:96]).all() and (lg[0, :32] == 128.0).all()
    assert (lg[0, 96:100] == 128.0).all()


# ---- top-k ----------------------------------------------------------------

def _brute_topk(v, topk):
    L = len(v)
    rank = [sum(1 for u in range(L) if v[u] > v[t] or (v[u] == v[t] and u < t))
            for t in range(L)]
    order = sorted((rk, t) for t, rk in enumerate(rank) if rk < topk)
    return [t for _, t in order] + [-1] * (topk - len(order))


@pytest.mark.parametrize("seed,distinct", [(0, 0), (1, 3), (2, 1), (3, 7)])
def test_topk_brute_force_rank(seed, distinct):
    rng = np.random.default_rng(seed)
    R, W, topk, next_n = 6, 90, 17, 2
    lg = rng.normal(size=(R, W)).astype(np.float32)
    if distinct:
        lg = rng.choice(rng.normal(size=distinct).astype(np.float32), size=(R, W))
    lg[0, 5] = -np.inf
    seq = [85, 9, 60]                         # rows: 84, 85 | 8, 9 | 59, 60 columns
    got = X.top_k_per_row(lg, next_n, seq, topk)
    for r in range(R):
        Lr = X.row_length(seq, r, next_n)
        assert Lr == seq[r // 2] - 2 + r % 2 + 1
        assert got[r].tolist() == _brute_topk(lg[r, :Lr].tolist(), topk), r


def test_topk_all_equal_and_short_rows():
    lg = np.zeros((2, 50), np.float32)
    got = X.top_k_per_row(lg, 1, [50, 3], 8)
    assert got[0].tolist() == list(range(8))
    assert got[1].tolist() == [0, 1, 2] + [-1] * 5
    assert (X.top_k_per_row(lg, 1, [0, 0], 4) == -1).all()


def test_rows_map_to_requests_by_next_n():
    # two requests, next_n = 2: rows 0,1 -> request 0; rows 2,3 -> request 1
    bs = 16
    keys = np.zeros((40, D), np.float32)
    keys[:, 0] = 1.0
    c0, bt0 = _cache_from_keys(_e4m3(keys[:20]), np.full(20, 1.0, np.float32), bs, [0, 1])
    c1, bt1 = _cache_from_keys(_e4m3(keys[:40]), np.full(40, 3.0, np.float32), bs, [0, 1, 2])
    cache = np.concatenate([c0, c1])                     # request 1's blocks at 2, 3, 4
    bt = np.full((2, 3), -1, np.int32)
    bt[0, :2] = bt0[0]
    bt[1, :3] = bt1[0] + 2
    q = _e4m3(np.ones((4, 1, D), np.float32))
    lg, err = X.paged_mqa_logits(q, cache, np.ones((4, 1), np.float32), [20, 40], bt, 2, 48, bs)
    assert err == 0
    assert [int(np.isfinite(lg[r]).sum()) for r in range(4)] == [19, 20, 39, 40]
    assert (lg[0, :19] == 1.0).all() and (lg[3, :40] == 3.0).all()
