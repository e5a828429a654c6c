"""Pins for the oracle's sparse attention ("vLLM: integrate FP16 packed QSA
extension", "Exact contracts"/Attention: Q/out [R,3,256], exact-packed K/V,
V at storage offset 256, logical indices with holes and duplicates).

Independent checks:
  * dense brute force: gather the listed tokens with Python's own page lookup
    and run scipy.special.softmax over all of them (a library routine);
  * duplicates = dense softmax over the distinct tokens with weights
    c_t * e^{z_t} (multiplicity c_t), computed with scipy.special.logsumexp;
  * one valid index: the output is that token's V exactly;
  * all keys equal: the output is the multiplicity-weighted mean of V;
  * inserting holes anywhere or permuting the list changes nothing beyond
    rounding; no valid index gives zeros;
  * select -> attend equals full dense attention over the sequence masked to
    the selected token set;
  * bad page ids / request ids are holes with the error bit set.
"""
import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

import oracle
from sparse_paged_attention_qsa_gb300 import workloads as W

SCALE = 1.0 / 16.0


def _kv(w, req, i):
    pt = w.kv_page_table.numpy()
    page = int(pt[req, i // 512])
    tok = w.kv_cache.numpy()[page, i % 512].reshape(-1).astype(np.float64)
    return tok[:256], tok[256:]


def _dense(w, r, idx, scale=SCALE):
    req = int(w.token_to_request[r])
    q = w.q_attn[r].numpy().astype(np.float64)
    valid = [int(i) for i in idx if i >= 0]
    if not valid:
        return np.zeros((3, 256))
    K = np.stack([_kv(w, req, i)[0] for i in valid])
    V = np.stack([_kv(w, req, i)[1] for i in valid])
    p = softmax(q @ K.T * scale, axis=1)
    return p @ V


def _run(w, idx, scale=SCALE):
    return oracle.attention(w.q_attn.numpy(), w.kv_cache.numpy(), w.kv_page_table.numpy(),
                            w.token_to_request.numpy(), idx, scale=scale)


@pytest.mark.parametrize("seed", range(3))
def test_attention_matches_dense_softmax(seed):
    w = W.build("att", [700, 1500, 40], premade_widths=[1024, 2051, 32], seed=seed)
    idx = w.indices.numpy()
    out, err = _run(w, idx)
    assert err == 0
    for r in range(w.R):
        np.testing.assert_allclose(out[r], _dense(w, r, idx[r]), rtol=0, atol=1e-12)


def test_attention_duplicates_are_weighted_terms():
    w = W.build("dup", [300], seed=4)
    rng = np.random.default_rng(4)
    toks = rng.choice(300, size=20, replace=False)
    counts = rng.integers(1, 5, size=20)
    lst = np.repeat(toks, counts)
    rng.shuffle(lst)
    idx = np.full((1, 2051), -1, np.int32)
    idx[0, :len(lst)] = lst
    out, _ = _run(w, idx)
    q = w.q_attn[0].numpy().astype(np.float64)
    K = np.stack([_kv(w, 0, t)[0] for t in toks])
    V = np.stack([_kv(w, 0, t)[1] for t in toks])
    z = q @ K.T * SCALE + np.log(counts)[None, :]
    p = np.exp(z - logsumexp(z, axis=1, keepdims=True))
    np.testing.assert_allclose(out[0], p @ V, rtol=0, atol=1e-12)


def test_attention_single_index_is_exact_v():
    w = W.build("one", [5000], seed=5)
    for t in (0, 511, 512, 4999):
        idx = np.full((1, 2051), -1, np.int32)
        idx[0, 1234] = t
        out, _ = _run(w, idx)
        v = _kv(w, 0, t)[1]
        assert np.array_equal(out[0], np.stack([v] * 3))


def test_attention_equal_keys_give_mean_of_v():
    w = W.build("eq", [1024], seed=6)
    kv = w.kv_cache
    kv[:, :, 0, :] = kv[0, 0, 0, :]            # every K identical
    lst = [3, 3, 3, 700, 12, 1000]
    idx = np.full((1, 2051), -1, np.int32)
    idx[0, :len(lst)] = lst
    out, _ = _run(w, idx)
    mean = np.mean([_kv(w, 0, t)[1] for t in lst], axis=0)
    np.testing.assert_allclose(out[0], np.stack([mean] * 3), rtol=0, atol=1e-12)


def test_attention_hole_and_permutation_invariance():
    w = W.build("perm", [3000], premade_widths=[2051], hole_frac=0.0, dup_frac=0.05, seed=7)
    idx = w.indices.numpy().copy()
    base, _ = _run(w, idx)
    rng = np.random.default_rng(7)
    perm = idx.copy()
    perm[0] = idx[0, rng.permutation(2051)]
    holes = np.full_like(idx, -1)
    keep = np.sort(rng.choice(2051, size=1500, replace=False))
    holes[0, :] = -1
    # same multiset, spread out with holes in between (list truncated to 2051)
    sub = idx[0, :1500]
    holes[0, keep] = sub
    sub_out, _ = _run(w, np.concatenate([sub, -np.ones(551, np.int32)])[None])
    np.testing.assert_allclose(_run(w, perm)[0], base, rtol=0, atol=1e-12)
    np.testing.assert_allclose(_run(w, holes)[0], sub_out, rtol=0, atol=1e-12)


def test_attention_empty_rows_are_zero():
    w = W.build("empty", [100, 0], seed=8)
    idx = np.full((2, 2051), -1, np.int32)
    out, err = _run(w, idx)
    assert err == 0 and (out == 0).all()
    out, err = _run(w, idx[:, :0])         # zero width
    assert (out == 0).all()


def test_attention_bad_ids_are_holes():
    w = W.build("bad", [1500, 1500], seed=9)
    pt = w.kv_page_table.numpy().copy()
    pt[0, 1] = -1                              # tokens 512..1023 of request 0 unmapped
    idx = np.full((2, 2051), -1, np.int32)
    idx[0, :4] = [5, 600, 7, 1400]
    idx[1, :3] = [5, 6, 200000]               # beyond the page table columns
    out, err = oracle.attention(w.q_attn.numpy(), w.kv_cache.numpy(), pt,
                                w.token_to_request.numpy(), idx)
    assert err == oracle.ERR_KV_PAGE
    w2 = W.Workload(**{**w.__dict__, "kv_page_table": torch.from_numpy(pt)})
    np.testing.assert_allclose(out[0], _dense(w2, 0, [5, 7, 1400]), atol=1e-12, rtol=0)
    np.testing.assert_allclose(out[1], _dense(w, 1, [5, 6]), atol=1e-12, rtol=0)
    out, err = oracle.attention(w.q_attn.numpy(), w.kv_cache.numpy(), pt,
                                np.array([0, 7], np.int32), idx)
    assert err & oracle.ERR_REQUEST and (out[1] == 0).all()


def test_select_then_attend_equals_masked_dense():
    w = W.build("e2e", [4 * 600 + 3, 901], seed=10)
    sel, err = oracle.select(w.q_sel.numpy(), w.cmp_cache.numpy(), w.cmp_page_table.numpy(),
                             w.token_to_request.numpy(), w.seq_lens.numpy(),
                             w.query_positions.numpy())
    assert err == 0
    out, err = _run(w, sel)
    assert err == 0
    for r in range(w.R):
        L = int(w.seq_lens[r])
        q = w.q_attn[r].numpy().astype(np.float64)
        K = np.stack([_kv(w, r, i)[0] for i in range(L)])
        V = np.stack([_kv(w, r, i)[1] for i in range(L)])
        mask = np.full(L, -np.inf)
        mask[sel[r][sel[r] >= 0]] = 0.0
        p = softmax(q @ K.T * SCALE + mask[None, :], axis=1)
        np.testing.assert_allclose(out[r], p @ V, rtol=0, atol=1e-12)
