"""GPU parity for qsa_build_metadata (qsa_cache.py, _build_qsa_metadata_kernel)
and for the multi-token decode chain built on it: the CUDA builder, selection
and attention through the C ABI vs the oracle's builder, selection and
attention -- bit-exact for every integer output, attention within 2e-3.

Batches: plain decode, speculative decode (several query tokens per request
at positions seq_len-n .. seq_len-1), prefill chunks, requests with no query
tokens, padding tokens past query_start_loc[-1], the three slot-map modes
(compressed keys, circular raw-key ring, pass-through), work lists shorter
and longer than the item count, a strided block table, and more requests
than the builder stages on chip."""
import numpy as np
import pytest
import torch

import sparse_paged_attention_qsa_gb300 as qsa
from oracle import metadata as M
from sparse_paged_attention_qsa_gb300 import workloads as W
from tests._util import oracle_attention, oracle_select
from tests.test_oracle_metadata import BT, COMMON, QSL, SL, SLOT_CIRC, SLOT_CMP, WORK7

pytestmark = pytest.mark.gpu
DEV = "cuda"
KEYS = ("token_to_req", "logical_positions", "visible_blocks", "slot_mapping")


def _compare(qsl, sl, bt, T, bt_dev=None, **kw):
    """Run both builders on the same inputs; return the GPU outputs."""
    common = kw.pop("common_slot_mapping", None)
    maxw = kw.pop("max_num_work", 0)
    nm = kw.pop("num_mapped_tokens", None)
    got = qsa.qsa_build_metadata(
        torch.as_tensor(qsl, dtype=torch.int32).to(DEV),
        torch.as_tensor(sl, dtype=torch.int32).to(DEV),
        bt_dev if bt_dev is not None else torch.as_tensor(bt, dtype=torch.int32).to(DEV), T,
        common_slot_mapping=None if common is None else
        torch.as_tensor(common, dtype=torch.int64).to(DEV),
        num_mapped_tokens=nm, max_num_work=maxw, **kw)
    torch.cuda.synchronize()
    exp = M.build_metadata(np.asarray(qsl), np.asarray(sl), np.asarray(bt), T,
                           common_slot_mapping=common, num_mapped_tokens=nm,
                           max_num_work=maxw if maxw else None, **kw)
    for k in KEYS:
        g = got[k][:T].cpu().numpy()
        assert np.array_equal(g, exp[k]), (k, np.nonzero(g != exp[k])[0][:8])
    if maxw:
        g = got["work_metadata"].cpu().numpy()
        assert np.array_equal(g, exp["work_metadata"]), np.nonzero(g != exp["work_metadata"])[0][:8]
    return got


def test_hand_worked_example_all_modes():
    g = _compare(QSL, SL, BT, 14, storage_block_size=2, compress_ratio=4,
                 common_slot_mapping=COMMON, max_num_work=7)
    assert g["slot_mapping"].cpu().tolist() == SLOT_CMP
    assert [tuple(x) for x in g["work_metadata"].cpu().tolist()] == WORK7
    g = _compare(QSL, SL, BT, 14, storage_block_size=2, compress_ratio=4,
                 circular_buffer_size=3)
    assert g["slot_mapping"].cpu().tolist() == SLOT_CIRC
    _compare(QSL, SL, BT, 14, storage_block_size=2, compress_ratio=1,
             common_slot_mapping=COMMON)


def _batch(seed, num_reqs, max_q, max_len, empty_frac=0.15, pad=3):
    rng = np.random.default_rng(seed)
    ql = rng.integers(1, max_q + 1, size=num_reqs)
    ql[rng.random(num_reqs) < empty_frac] = 0
    L = np.array([int(rng.integers(q, max_len + 1)) if q else int(rng.integers(0, max_len + 1))
                  for q in ql], dtype=np.int64)
    qsl = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    T = int(qsl[-1]) + pad
    return rng, qsl, L.astype(np.int32), T


@pytest.mark.parametrize("seed,num_reqs,max_q", [(0, 1, 1), (1, 7, 4), (2, 256, 1), (3, 64, 4),
                                                  (4, 300, 9), (5, 33, 700)])
def test_compressed_slot_map_random(seed, num_reqs, max_q):
    rng, qsl, L, T = _batch(seed, num_reqs, max_q, 40000)
    sbs = 128
    cols = int(L.max()) // 4 // sbs + 1
    bt = rng.permutation(num_reqs * cols + 11)[:num_reqs * cols].astype(np.int32)
    bt = bt.reshape(num_reqs, cols)
    bt[rng.random(bt.shape) < 0.05] = -1
    common = rng.integers(-1, 1 << 40, size=T)
    total = int(sum(max(1, int(L[i]) // 4 - (int(L[i]) - int(qsl[i + 1] - qsl[i])) // 4)
                    for i in range(num_reqs) if qsl[i + 1] > qsl[i]))
    for maxw in (0, max(1, total // 2), total + 300):
        _compare(qsl, L, bt, T, storage_block_size=sbs, compress_ratio=4,
                 common_slot_mapping=common, max_num_work=maxw)


@pytest.mark.parametrize("cbs", [1, 8, 128])
def test_circular_ring_random(cbs):
    rng, qsl, L, T = _batch(10 + cbs, 90, 300, 5000)
    bt = rng.permutation(90).astype(np.int32).reshape(90, 1)
    bt[5, 0] = -1
    _compare(qsl, L, bt, T, storage_block_size=64, compress_ratio=4, circular_buffer_size=cbs,
             max_num_work=50)


def test_passthrough_and_ratio_one():
    rng, qsl, L, T = _batch(20, 40, 6, 3000)
    bt = np.zeros((40, 2), np.int32)
    common = rng.integers(-1, 100000, size=T)
    _compare(qsl, L, bt, T, storage_block_size=16, compress_ratio=1, common_slot_mapping=common,
             max_num_work=200)


def test_strided_block_table_and_extra_rows():
    rng, qsl, L, T = _batch(30, 50, 5, 20000)
    cols = int(L.max()) // 4 // 32 + 1
    big = torch.from_numpy(rng.integers(-1, 5000, size=(64, 2 * cols)).astype(np.int32))
    view = big.to(DEV)[:, ::2]                        # strides (2*cols, 2); 64 >= 50 rows
    common = rng.integers(0, 100, size=T)
    _compare(qsl, L, big[:, ::2].numpy(), T, bt_dev=view, storage_block_size=32,
             compress_ratio=4, common_slot_mapping=common, max_num_work=80)


def test_many_requests_global_search_path():
    # more requests than the builder stages in shared memory
    rng, qsl, L, T = _batch(40, 9000, 3, 600, empty_frac=0.3, pad=0)
    bt = rng.integers(0, 1 << 20, size=(9000, 2)).astype(np.int32)
    common = np.arange(T)
    _compare(qsl, L, bt, T, storage_block_size=128, compress_ratio=4,
             common_slot_mapping=common, max_num_work=T + 9000)


def test_num_mapped_below_and_above_query_end():
    rng, qsl, L, T = _batch(50, 20, 5, 900, pad=6)
    bt = rng.integers(0, 100, size=(20, 3)).astype(np.int32)
    common = np.arange(T)
    for nm in (0, int(qsl[-1]) // 2, T):
        _compare(qsl, L, bt, T, storage_block_size=128, compress_ratio=4,
                 common_slot_mapping=common, num_mapped_tokens=nm)


def test_work_list_only_and_reuse_of_outputs():
    rng, qsl, L, _ = _batch(60, 500, 8, 9000, pad=0)
    bt = np.zeros((500, 1), np.int32)
    # no tokens, only a work list (the builder's second grid role)
    _compare(qsl, L, bt, 0, storage_block_size=128, compress_ratio=4,
             common_slot_mapping=np.zeros(0, np.int64), max_num_work=3000)
    # preallocated outputs are overwritten in full
    T = int(qsl[-1])
    out = {k: torch.full((T,), 77, dtype=dt, device=DEV) for k, dt in
           zip(KEYS, (torch.int32, torch.int64, torch.int32, torch.int64))}
    g = qsa.qsa_build_metadata(torch.from_numpy(qsl).to(DEV), torch.from_numpy(L).to(DEV),
                               torch.from_numpy(bt).to(DEV), T, storage_block_size=128,
                               compress_ratio=4, common_slot_mapping=torch.zeros(
                                   T, dtype=torch.int64, device=DEV), out=out)
    exp = M.build_metadata(qsl, L, bt, T, storage_block_size=128, compress_ratio=4,
                           common_slot_mapping=np.zeros(T, np.int64))
    for k in KEYS:
        assert g[k] is out[k]
        assert np.array_equal(g[k].cpu().numpy(), exp[k])


# ---- multi-token decode chain: builder -> selection -> attention -------------

def _chain(w, rows_checked=None):
    """GPU chain vs oracle chain on a workload with query_start_loc."""
    nreq = w.seq_lens.numel()
    T = w.R
    g = qsa.qsa_build_metadata(w.query_start_loc, w.seq_lens, w.cmp_page_table, T,
                               storage_block_size=128, compress_ratio=4,
                               common_slot_mapping=torch.zeros(T, dtype=torch.int64, device=DEV),
                               num_mapped_tokens=T)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    idx, out = qsa.qsa_decode(w.q_sel, w.cmp_cache, w.cmp_page_table, g["token_to_req"],
                              w.seq_lens, g["logical_positions"], w.q_attn, w.k_view, w.v_view,
                              w.kv_page_table, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    m = M.build_metadata(w.query_start_loc.cpu().numpy(), w.seq_lens.cpu().numpy(),
                         w.cmp_page_table.cpu().numpy(), T, storage_block_size=128,
                         compress_ratio=4, common_slot_mapping=np.zeros(T, np.int64))
    assert np.array_equal(g["token_to_req"].cpu().numpy(), m["token_to_req"])
    assert np.array_equal(g["logical_positions"].cpu().numpy(), m["logical_positions"])
    wo = W.Workload(**{**w.__dict__,
                       "token_to_request": torch.from_numpy(m["token_to_req"]).to(DEV),
                       "query_positions": torch.from_numpy(m["logical_positions"]).to(DEV)})
    rows = list(range(w.R)) if rows_checked is None else list(rows_checked)
    exp_idx, oerr = oracle_select(wo, rows=rows)
    assert oerr == 0
    got_idx = idx.cpu().numpy()
    for i, r in enumerate(rows):
        assert np.array_equal(got_idx[r], exp_idx[i]), r
        # the row's visible blocks are what the builder reported
        vis = int(m["visible_blocks"][r])
        nsel = min(vis, 512)
        assert (got_idx[r][:4 * nsel] >= 0).all() and \
            (got_idx[r][4 * nsel:4 * nsel + 3] < 4 * vis + 3).all()
    full = np.full((w.R, 2051), -1, np.int32)
    full[rows] = exp_idx                    # the oracle's own index lists
    exp_out, _ = oracle_attention(wo, full, rows=rows)
    diff = np.abs(out.float().cpu().numpy()[rows] - exp_out).max()
    assert diff <= 2e-3, diff
    return got_idx


def test_speculative_decode_chain():
    # 12 requests x 4 query tokens (positions L-4 .. L-1), lengths across
    # page boundaries and below / above the 2048-token saturation point
    rng = np.random.default_rng(70)
    L = [int(x) for x in rng.integers(600, 40000, size=12)]
    L[0], L[1], L[2] = 2051, 2052, 9215
    w = W.build("spec4", L, query_lens=[4] * 12, seed=71, device=DEV)
    got = _chain(w)
    # request 0 (L = 2051, positions 2047..2050): every row sees 512 blocks;
    # the tails grow from 0 tokens (position 2047) to 3 (position 2050)
    assert (got[0] >= 0).sum() == 4 * 512 + 0 and (got[3] >= 0).sum() == 4 * 512 + 3


def test_mixed_prefill_chunk_and_decode_chain():
    # a prefill chunk of 40 tokens, two empty requests, decode and spec rows
    L = [5000, 777, 12000, 3, 65536, 9000]
    ql = [40, 0, 1, 3, 5, 0]
    w = W.build("mixed", L, query_lens=ql, seed=72, device=DEV)
    _chain(w, rows_checked=[0, 1, 17, 38, 39, 40, 41, 42, 43, 44, 45, 46, 47, 48])


def _with_positions(w):
    m = M.build_metadata(w.query_start_loc.cpu().numpy(), w.seq_lens.cpu().numpy(),
                         w.cmp_page_table.cpu().numpy(), w.R, storage_block_size=128,
                         compress_ratio=4, common_slot_mapping=np.zeros(w.R, np.int64))
    return W.Workload(**{**w.__dict__,
                         "token_to_request": torch.from_numpy(m["token_to_req"]).to(DEV),
                         "query_positions": torch.from_numpy(m["logical_positions"]).to(DEV)})


def _select_parity(w, pt=None):
    pt = w.cmp_page_table if pt is None else pt
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = qsa.qsa_select_paged_tokens(w.q_sel, w.cmp_cache, pt, w.token_to_request,
                                      w.seq_lens, w.query_positions, error_word=err)
    torch.cuda.synchronize()
    exp, oerr = oracle_select(w, cmp_page_table=pt)
    g = got.cpu().numpy()
    for r in range(w.R):
        assert np.array_equal(g[r], exp[r]), r
    assert int(err.item()) == oerr
    return g


@pytest.mark.parametrize("fp8", [False, True])
def test_row_groups_straddling_pages_and_windows(fp8):
    # rows of one request see different block counts: L = 517 gives 128, 128,
    # 129, 129 visible blocks (1 or 2 pages); L = 2053 crosses the 512-block
    # saturation; query lengths 3, 5, 7, 9 make groups break at the 8-row
    # window edges
    L = [517, 2053, 700, 30000, 131, 5000, 9000]
    ql = [4, 4, 3, 5, 7, 9, 1]
    w = _with_positions(W.build("groups", L, query_lens=ql, cmp_dtype="fp8" if fp8 else "fp16",
                                seed=80, device=DEV))
    _select_parity(w)


def test_row_groups_bad_page_inside_group():
    L = [3000, 6000, 1000]
    w = _with_positions(W.build("groupbad", L, query_lens=[4, 6, 2], seed=81, device=DEV))
    pt = w.cmp_page_table.clone()
    pt[1, 3] = -5                           # a missing page inside request 1's rows
    pt[0, 0] = w.cmp_cache.shape[0] + 1     # and past the pool for request 0
    g = _select_parity(w, pt)
    assert (g[:4] >= 0).sum() > 0


def test_row_groups_ties_and_duplicate_pages():
    w = _with_positions(W.build("groupties", [6003, 4099, 30001], query_lens=[4, 4, 8],
                                distinct_keys=4, dup_mapping=True, seed=82, device=DEV))
    _select_parity(w)
