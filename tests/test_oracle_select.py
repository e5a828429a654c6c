"""Pins for the oracle's selection ("vLLM: integrate FP16 packed QSA
extension", Summary bullet 3 and "Exact contracts"/Selection; visible blocks
from qsa_cache.py, _build_qsa_metadata_kernel and compressed_qsa_slot_mapping).

Independent checks:
  * visible blocks == a brute-force count of complete compression groups
    (group g exists once token 4g+3 exists and is at or before the query);
  * the pages' worked sizes (tests/golden/worked_sizes.json);
  * brute-force ranking on small rows: a block's rank is the number of blocks
    that beat it (higher score, or equal score and smaller index); computed
    with Python's own page lookup, no sort;
  * special cases: Q = 0 (all scores +0 -> blocks in index order), V <= 512
    (every block kept), one-hot keys (scores known in closed form);
  * invariants: output width, no duplicates, tokens never past the query,
    -1 only as a suffix, expanded groups of 4 consecutive tokens;
  * error handling: bad request ids and page ids.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from sparse_paged_attention_qsa_gb300 import workloads as W


def test_visible_blocks_brute_force():
    for L in list(range(0, 40)) + [519, 9215, 131072]:
        for pos in list(range(-6, 44)) + [L - 1, L, L + 5]:
            last = min(pos, L - 1)
            groups = sum(1 for g in range(0, max(0, L // 4 + 2)) if 4 * g + 3 <= last)
            assert oracle.visible_blocks(L, pos) == groups, (L, pos)
            # tail = tokens <= last not inside a complete group, contiguous
            te = oracle.tail_end(L, pos)
            covered = set(range(4 * groups)) | set(range(4 * groups, te + 1))
            assert covered == set(range(0, last + 1)), (L, pos)
            assert 0 <= te + 1 - 4 * groups <= 3 or last < 0


def test_worked_sizes(golden_dir):
    d = json.load(open(os.path.join(golden_dir, "worked_sizes.json")))
    for c in d["cases"]:
        L = c["seq_len"]
        V = oracle.visible_blocks(L, L - 1)
        assert V == c["visible_blocks"]
        w = W.build("worked", [L], seed=5)
        out, err = oracle.select(w.q_sel.numpy(), w.cmp_cache.numpy(), w.cmp_page_table.numpy(),
                                 w.token_to_request.numpy(), w.seq_lens.numpy(),
                                 w.query_positions.numpy())
        assert err == 0
        assert int((out[0] >= 0).sum()) == c["valid_tokens"]


def _brute_select(w, r):
    """Independent restatement: score every block with its own page lookup,
    rank by counting, expand, append the tail."""
    q = w.q_sel[r].numpy()
    req = int(w.token_to_request[r])
    L = int(w.seq_lens[req])
    pos = int(w.query_positions[r])
    last = min(pos, L - 1)
    V = sum(1 for g in range(L // 4 + 1) if 4 * g + 3 <= last)
    pt = w.cmp_page_table.numpy()
    pool = w.cmp_cache.numpy()
    scores = {}
    for b in range(V):
        page = int(pt[req, b // 128])
        scores[b] = float(oracle.score(q, pool[page, b % 128, 0]))
    rank = {b: sum(1 for c in scores if scores[c] > scores[b] or
                   (scores[c] == scores[b] and c < b)) for b in scores}
    order = sorted((rk, b) for b, rk in rank.items() if rk < 512)
    toks = [4 * b + i for _, b in order for i in range(4)]
    toks += list(range(4 * V, last + 1))
    return toks + [-1] * (2051 - len(toks))


def _oracle(w):
    return oracle.select(w.q_sel.numpy(), w.cmp_cache.numpy(), w.cmp_page_table.numpy(),
                         w.token_to_request.numpy(), w.seq_lens.numpy(),
                         w.query_positions.numpy())


@pytest.mark.parametrize("seed", range(4))
def test_select_matches_brute_force_rank(seed):
    rng = np.random.default_rng(seed)
    lens = [int(x) for x in rng.integers(0, 180, size=5)] + [3, 4, 7]
    w = W.build("small", lens, seed=seed)
    out, err = _oracle(w)
    assert err == 0
    for r in range(w.R):
        assert out[r].tolist() == _brute_select(w, r), r


def test_select_brute_force_over_512_blocks():
    # V = 700 > 512: the cut at rank 512 is exercised; 6 pages cross
    w = W.build("over", [2803], seed=11)
    out, err = _oracle(w)
    assert err == 0
    assert out[0].tolist() == _brute_select(w, 0)


def test_select_ties_brute_force():
    # only 3 distinct keys: heavy exact ties broken by ascending block index
    w = W.build("ties", [2403, 777], distinct_keys=3, seed=3)
    out, err = _oracle(w)
    assert err == 0
    for r in range(w.R):
        assert out[r].tolist() == _brute_select(w, r)


def test_select_zero_query_gives_index_order():
    w = W.build("zeroq", [4 * 700 + 2, 4 * 100 + 3, 6], seed=1)
    w.q_sel.zero_()
    out, _ = _oracle(w)
    # all scores +0 -> the first min(V,512) blocks in ascending order
    exp0 = [t for b in range(512) for t in range(4 * b, 4 * b + 4)] + [2800, 2801]
    assert out[0, :len(exp0)].tolist() == exp0 and (out[0, len(exp0):] == -1).all()
    exp1 = list(range(403))
    assert out[1, :403].tolist() == exp1 and (out[1, 403:] == -1).all()
    assert out[2, :6].tolist() == [0, 1, 2, 3, 4, 5]


def test_select_one_hot_keys_closed_form():
    # k_b = a_b * e_d: s_b = sum_h max(0, q[h,d] * a_b) exactly (one product)
    w = W.build("onehot", [4 * 300 + 3], seed=2)
    d = 17
    a = torch.linspace(-2, 2, 300).to(torch.float16)
    pool = w.cmp_cache
    pool.zero_()
    pt = w.cmp_page_table
    for b in range(300):
        pool[int(pt[0, b // 128]), b % 128, 0, d] = a[b]
    q = w.q_sel[0].float()
    s = [sum(max(0.0, float(q[h, d]) * float(a[b])) for h in range(4)) for b in range(300)]
    # the closed form sums four exact products in the stated head order
    s32 = [float((np.float32(max(0.0, float(q[0, d]) * float(a[b]))) +
                  np.float32(max(0.0, float(q[1, d]) * float(a[b])))) +
                 (np.float32(max(0.0, float(q[2, d]) * float(a[b]))) +
                  np.float32(max(0.0, float(q[3, d]) * float(a[b]))))) for b in range(300)]
    order = sorted(range(300), key=lambda b: (-s32[b], b))
    out, _, sc = oracle.select(w.q_sel.numpy(), pool.numpy(), pt.numpy(),
                               w.token_to_request.numpy(), w.seq_lens.numpy(),
                               w.query_positions.numpy(), return_scores=True)
    got_blocks = out[0, :1200:4] // 4
    assert got_blocks.tolist() == order
    assert np.allclose(sc[0, :300], [s[b] for b in order], rtol=1e-6, atol=0)


def _invariants(out, w, r):
    req = int(w.token_to_request[r])
    L, pos = int(w.seq_lens[req]), int(w.query_positions[r])
    V = oracle.visible_blocks(L, pos)
    tail = max(0, min(pos, L - 1) - 4 * V + 1)
    width = 4 * min(512, V) + tail
    row = out[r]
    assert (row[:width] >= 0).all() and (row[width:] == -1).all()
    assert len(set(row[:width].tolist())) == width
    assert (row[:width] <= min(pos, L - 1)).all()
    grp = row[:4 * min(512, V)].reshape(-1, 4)
    assert (grp[:, 0] % 4 == 0).all() and (np.diff(grp, axis=1) == 1).all()
    assert row[4 * min(512, V):width].tolist() == list(range(4 * V, 4 * V + tail))


def test_select_invariants_random_rows():
    rng = np.random.default_rng(7)
    lens = [int(x) for x in rng.integers(1, 6000, size=12)]
    pos = [L - 1 - int(rng.integers(0, 3)) for L in lens]   # speculative rows too
    w = W.build("inv", lens, positions=pos, seed=7)
    out, sc_err, sc = oracle.select(w.q_sel.numpy(), w.cmp_cache.numpy(),
                                    w.cmp_page_table.numpy(), w.token_to_request.numpy(),
                                    w.seq_lens.numpy(), w.query_positions.numpy(),
                                    return_scores=True)
    for r in range(w.R):
        _invariants(out, w, r)
        n = min(512, oracle.visible_blocks(lens[r], pos[r]))
        s = sc[r, :n]
        blocks = out[r, :4 * n:4] // 4
        ok = (s[:-1] > s[1:]) | ((s[:-1] == s[1:]) & (blocks[:-1] < blocks[1:]))
        assert ok.all()


def test_select_empty_and_short_rows():
    w = W.build("short", [1, 2, 3, 4, 5, 8], seed=9)
    out, err = _oracle(w)
    assert err == 0
    assert out[0, :2].tolist() == [0, -1]
    assert out[2, :4].tolist() == [0, 1, 2, -1]
    assert out[3, :5].tolist() == [0, 1, 2, 3, -1]        # one block, empty tail
    assert out[4, :5].tolist() == [0, 1, 2, 3, 4]
    # seq_len 0: nothing at all
    w0 = W.build("empty", [0, 5], seed=9)
    out0, _ = _oracle(w0)
    assert (out0[0] == -1).all()


def test_select_multi_request_token_to_request():
    w = W.build("multi", [900, 2500, 30], seed=4)
    base, _ = _oracle(w)
    # rows naming the requests in another order (one request twice) give the
    # same per-row result as the row that owns that request
    perm = [2, 0, 1, 0]
    q2 = np.stack([w.q_sel.numpy()[p] for p in perm])
    qpos = np.array([int(w.query_positions[p]) for p in perm], np.int64)
    out, err = oracle.select(q2, w.cmp_cache.numpy(), w.cmp_page_table.numpy(),
                             np.array(perm, np.int32), w.seq_lens.numpy(), qpos)
    assert err == 0
    for i, p in enumerate(perm):
        assert (out[i] == base[p]).all()


def test_select_bad_request_and_page_ids():
    w = W.build("bad", [1000, 1000], seed=6)   # 250 blocks each, empty tail
    pt = w.cmp_page_table.numpy().copy()
    pt[1, 1] = 10 ** 6                       # page id beyond the pool
    t2r = np.array([5, 1], np.int32)         # row 0 names a request that does not exist
    out, err = oracle.select(w.q_sel.numpy(), w.cmp_cache.numpy(), pt, t2r,
                             w.seq_lens.numpy(), w.query_positions.numpy())
    assert err == (oracle.ERR_REQUEST | oracle.ERR_CMP_PAGE)
    assert (out[0] == -1).all()
    valid = out[1][out[1] >= 0]
    # blocks 128..249 sit on the bad page and are skipped; 0..127 remain
    assert len(valid) == 4 * 128
    assert set((valid // 4).tolist()) == set(range(128))
    assert (out[1, 512:] == -1).all()


def test_select_duplicate_physical_pages():
    w = W.build("dup", [3000, 2000], dup_mapping=True, seed=8)
    out, err = _oracle(w)
    assert err == 0
    for r in range(w.R):
        assert out[r].tolist() == _brute_select(w, r)
        _invariants(out, w, r)
