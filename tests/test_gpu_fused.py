"""GPU parity for qsa_select_attend, the one-call decode step: the selection's
indices must be bit-identical to the oracle's (and to qsa_select_paged_tokens),
and the attention output within 2e-3 of the binary64 oracle over those
indices ("vLLM: integrate FP16 packed QSA extension", Summary and "Exact
contracts"/Selection and Attention; the pages' tie, tail, saturation and
multi-request cases).

Small batches (as many rows as the GPU holds clusters of the fused kernel,
at most 256) run one fused kernel where it is estimated faster; larger ones run the two calls' kernels
from one workspace, so their outputs must equal the two calls' bit for
bit.  The edge cases run both ways (the row list repeated past the fused
limit, which also puts the chained attention past 32 rows, where it cuts
the index lists into equal runs over the batch), and the tests also cover
row chunks (more than 1024 rows), speculative rows that share a request,
every cluster size of the fused kernel, and repeated calls on a dirty
workspace.  Tolerance as in test_gpu_attention.py.
"""
import numpy as np
import pytest
import torch

import sparse_paged_attention_qsa_gb300 as qsa
from sparse_paged_attention_qsa_gb300 import workloads as W
from tests._util import CORES, oracle_attention, oracle_select

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = 2e-3


def _fused(w, pt=None, t2r=None, workspace=None):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    idx, out = qsa.qsa_select_attend(
        w.q_sel, w.cmp_cache, w.cmp_page_table if pt is None else pt,
        w.token_to_request if t2r is None else t2r, w.seq_lens, w.query_positions,
        w.q_attn, w.k_view, w.v_view, w.kv_page_table, workspace=workspace, error_word=err)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), out.float().cpu().numpy(), int(err.item())


def _check(w, rows=None, pt=None, t2r=None):
    got_idx, got_out, gerr = _fused(w, pt=pt, t2r=t2r)
    rows = list(range(w.R)) if rows is None else list(rows)
    exp_idx, oerr = oracle_select(w, rows=rows, cmp_page_table=pt, token_to_request=t2r)
    for i, r in enumerate(rows):
        if not np.array_equal(got_idx[r], exp_idx[i]):
            bad = np.nonzero(got_idx[r] != exp_idx[i])[0]
            raise AssertionError(f"row {r}: {len(bad)} index mismatches, first at {bad[0]}")
    full = np.full((w.R, 2051), -1, np.int32)
    full[rows] = exp_idx                    # the oracle's own index lists
    exp_out, _ = oracle_attention(w, full, rows=rows, token_to_request=t2r)
    diff = np.abs(got_out[rows] - exp_out).max() if rows else 0.0
    assert diff <= TOL, f"max abs error {diff}"
    return got_idx, got_out, gerr, oerr


@pytest.mark.parametrize("cfg", [0, 1, 2, 3])
def test_fused_configs(cfg):
    w = W.config(cfg, device=DEV)
    _, _, gerr, oerr = _check(w)
    assert gerr == oerr == 0


def test_fused_config4_full_size_all_rows():
    # indices of every row bit for bit; attention on at least 32 rows,
    # including every row at an edge of the stream split's runs
    from tests.test_gpu_attention import config4_attention_rows
    w = W.config(4, device=DEV)
    got_idx, got_out, gerr = _fused(w)
    assert gerr == 0
    exp_idx, oerr = oracle_select(w, threads=CORES)
    assert oerr == 0
    bad = [r for r in range(w.R) if not np.array_equal(got_idx[r], exp_idx[r])]
    assert not bad, f"rows differing from the oracle: {bad[:10]}"
    rows = config4_attention_rows(w.R)
    exp_out, _ = oracle_attention(w, exp_idx, rows=rows, threads=CORES)
    assert np.abs(got_out[rows] - exp_out).max() <= TOL
    assert np.isfinite(got_out).all()


def test_fused_matches_two_call_path():
    # a batch above the fused kernel's limit: the chained kernels, bit for
    # bit the two calls' (lengths spread over [512, 65536])
    n = qsa.qsa_select_attend_fused_rows() + 1
    w = W.build("chain", [512 + (i * 40503) % 65025 for i in range(n)], seed=1002, device=DEV)
    idx2, out2 = qsa.qsa_decode(w.q_sel, w.cmp_cache, w.cmp_page_table, w.token_to_request,
                                w.seq_lens, w.query_positions, w.q_attn, w.k_view, w.v_view,
                                w.kv_page_table)
    got_idx, got_out, gerr = _fused(w)
    assert gerr == 0
    assert np.array_equal(got_idx, idx2.cpu().numpy())
    assert np.array_equal(got_out, out2.float().cpu().numpy())     # the same kernels


# --- small batches: one fused kernel, one thread-block cluster per
# row (scoring, top-512 and attention; the index list handed over in shared
# memory).  Indices bit-exact, attention within the tolerance; the fused
# attention cuts a row's list differently from the two calls' kernels, so
# its output is compared with the oracle, not bit for bit with theirs.

@pytest.mark.parametrize("lens", [[131072] * 16, [131072, 519, 9215, 70001, 3, 0, 65536, 4099],
                                  [2051], [300003, 40003]])
def test_fused_small_batch_matches_two_calls_and_oracle(lens):
    w = W.build("small", lens, seed=len(lens) + lens[0] % 97, device=DEV)
    got_idx, got_out, gerr, oerr = _check(w)
    assert gerr == oerr == 0
    idx2, out2 = qsa.qsa_decode(w.q_sel, w.cmp_cache, w.cmp_page_table, w.token_to_request,
                                w.seq_lens, w.query_positions, w.q_attn, w.k_view, w.v_view,
                                w.kv_page_table)
    assert np.array_equal(got_idx, idx2.cpu().numpy())
    assert np.abs(got_out - out2.float().cpu().numpy()).max() <= 2 * TOL


@pytest.mark.parametrize("R", [1, 4, 12, 24])
def test_fused_small_batch_fp8_keys(R):
    # the device picks the cluster size per batch (on a GB300: 16 CTAs for 1
    # and 4 rows, fewer for 12 and 24)
    lens = [9215, 131072, 519, 40000] * 3
    w = W.build("small8", lens[:R], cmp_dtype="fp8", distinct_keys=0, seed=70 + R, device=DEV)
    _, _, gerr, oerr = _check(w)
    assert gerr == oerr == 0


def test_fused_small_batch_ties_bad_pages_and_requests():
    w = W.build("smallbad", [6003, 30001, 515, 131072, 2051, 9000], distinct_keys=2,
                dup_mapping=True, seed=77, device=DEV)
    pt = w.cmp_page_table.clone()
    pt[1, 3] = -1                                 # an unmapped compressed page
    pt[3, 200] = w.cmp_cache.shape[0] + 2         # a page beyond the pool
    t2r = torch.arange(w.R, dtype=torch.int32, device=DEV)
    t2r[4] = 99                                   # a row without a request
    got_idx, got_out, gerr, oerr = _check(w, pt=pt, t2r=t2r)
    assert gerr == oerr == (qsa.DERR_REQUEST | qsa.DERR_CMP_PAGE)
    assert (got_idx[4] == -1).all() and (got_out[4] == 0).all()


def test_fused_small_batch_bad_kv_pages():
    w = W.build("smallkv", [9215, 20000, 3000], seed=78, device=DEV)
    kpt = w.kv_page_table.clone()
    kpt[0, 3] = -1                                # tokens 1536..2047 of row 0: holes
    kpt[2, 1] = w.kv_cache.shape[0] + 7
    w2 = W.Workload(**{**w.__dict__, "kv_page_table": kpt})
    _, _, gerr, oerr = _check(w2)
    assert oerr == 0 and gerr == qsa.DERR_KV_PAGE


def test_fused_rows_query_and_the_boundary():
    # the largest batch the fused kernel takes on this GPU (as many rows as
    # it holds clusters of 4 or more CTAs at once), and one row more (the
    # chained kernels); a lone 131072-token row (256 columns) takes the
    # chained kernels too
    n = qsa.qsa_select_attend_fused_rows()
    assert 1 <= n <= 256
    assert qsa.qsa_select_attend_fused_rows(torch.float8_e4m3fn) >= 1
    assert qsa.qsa_select_attend_fused_rows(torch.float32) == 0
    cyc = [131072, 9215, 519, 3, 70001, 2052]
    for R in (1, 2, n, n + 1):
        w = W.build("bound", [cyc[i % len(cyc)] for i in range(R)], seed=80 + R, device=DEV)
        _, _, gerr, oerr = _check(w)
        assert gerr == oerr == 0


def _fused_wins(R, cols, cs):
    # include/qsa.h, qsa_select_attend_fused_cluster: 25 us + 0.9 us per page
    # of a CTA against 50 us + 6.25 ns per page of the batch (x 1600)
    return 40000 + 1440 * -(-cols // cs) <= 80000 + 10 * R * cols


def test_fused_cluster_query():
    # the cluster size a batch runs with: 1 .. 16 CTAs, never fewer CTAs
    # for fewer rows; 0 above the fused limit, for tables wider than 128
    # columns per row, where the chained kernels are estimated faster, and
    # for other key types
    n = qsa.qsa_select_attend_fused_rows()
    prev = 17
    for R in range(1, n + 1):
        cs = qsa.qsa_select_attend_fused_cluster(R, 2)
        assert 1 <= cs <= 16 and cs <= prev
        prev = cs
        for cols in (1, 64, 128, 200, 256, 512, 128 * R, 128 * R + 1):
            want = cs if cols <= 128 * R and _fused_wins(R, cols, cs) else 0
            assert qsa.qsa_select_attend_fused_cluster(R, cols) == want, (R, cols)
    assert qsa.qsa_select_attend_fused_cluster(1, 256) == 0     # a lone row of 131072 tokens
    assert qsa.qsa_select_attend_fused_cluster(n + 1, 64) == 0
    assert qsa.qsa_select_attend_fused_cluster(0, 64) == 0
    assert qsa.qsa_select_attend_fused_cluster(1, 2, torch.float32) == 0
    assert qsa.qsa_select_attend_fused_cluster(1, 2, torch.float8_e4m3fn) >= 2


@pytest.mark.parametrize("cols", [256, 257])
def test_fused_page_table_width_boundary(cols):
    # two rows of 131072 tokens: a table of 128 columns per row takes the
    # fused kernel, one column more (unused, -1) the chained kernels; both
    # match the oracle
    w = W.build("width", [131072, 9215], cmp_cols=cols, seed=95, device=DEV)
    assert (qsa.qsa_select_attend_fused_cluster(2, cols) > 0) == (cols == 256)
    _, _, gerr, oerr = _check(w)
    assert gerr == oerr == 0


@pytest.mark.parametrize("kdt", ["fp16", "fp8"])
def test_fused_every_cluster_size(kdt):
    # batches of 2 .. n rows of mixed lengths (131072-token rows included:
    # 256 columns) run with every cluster size the device picks for them;
    # each is checked against the oracle
    tdt = torch.float8_e4m3fn if kdt == "fp8" else torch.float16
    n = qsa.qsa_select_attend_fused_rows(tdt)
    cyc = [131072, 9215, 519, 70001, 3, 2052, 40000]
    seen = {}
    for R in range(2, n + 1):
        cs = qsa.qsa_select_attend_fused_cluster(R, 256, tdt)
        if cs == 0 or cs in seen:
            continue
        seen[cs] = R
        w = W.build("csize", [cyc[i % len(cyc)] for i in range(R)], cmp_dtype=kdt,
                    seed=90 + R, device=DEV)
        assert w.cmp_page_table.shape[1] == 256
        _, _, gerr, oerr = _check(w)
        assert gerr == oerr == 0, (R, cs)
    assert len(seen) >= 2, seen


@pytest.mark.parametrize("R", [1, 3, "over"])
def test_fused_empty_compressed_pool(R):
    # a compressed cache of no pages: every page id is out of range, so no
    # block has a key -- each row keeps only its tail tokens (fused kernel
    # for 1 and 3 rows, the chained kernels one row above the fused limit)
    if R == "over":
        R = qsa.qsa_select_attend_fused_rows() + 1
    lens = [519, 9215, 131072] * (R // 3 + 1)
    w = W.build("nopool", lens[:R], seed=83 + R, device=DEV)
    w = W.Workload(**{**w.__dict__, "cmp_cache": w.cmp_cache[:0]})
    got_idx, got_out, gerr, oerr = _check(w)
    assert gerr == oerr == qsa.DERR_CMP_PAGE
    for r, L in enumerate(lens[:R]):
        tail = list(range(4 * (L // 4), L))
        assert got_idx[r, :len(tail)].tolist() == tail and (got_idx[r, len(tail):] == -1).all()


@pytest.mark.parametrize("cfg", [0, 1])
def test_fused_small_batch_deterministic_on_dirty_workspace(cfg):
    # the fused kernel (a short row at 519 tokens, a ranked row at 9215):
    # repeated calls on a dirty workspace give identical indices and outputs
    w = W.config(cfg, device=DEV)
    a_idx, a_out, _ = _fused(w)
    need = qsa.qsa_select_attend_workspace_bytes(w.R, w.cmp_page_table.shape[1])
    ws = torch.full((need,), 0x5A, dtype=torch.uint8, device=DEV)
    for _ in range(3):
        b_idx, b_out, gerr = _fused(w, workspace=ws)
        assert gerr == 0
        assert np.array_equal(a_idx, b_idx) and np.array_equal(a_out, b_out)


def _rows(lens, big):
    """The row list, repeated past the fused kernel's limit (and 32 rows) when
    the chained kernels are wanted."""
    n = max(qsa.qsa_select_attend_fused_rows(), 32) + 1
    return lens * (n // len(lens) + 1) if big else lens


@pytest.mark.parametrize("big", [False, True])
@pytest.mark.parametrize("lens", [[0, 1, 3, 4, 7, 515, 516, 519, 1027], [2051, 2053, 9215, 131072]])
def test_fused_short_empty_and_saturated_rows(lens, big):
    w = W.build("edge", _rows(lens, big), seed=sum(lens) % 1000 + 3, device=DEV)
    _, got_out, gerr, oerr = _check(w)
    assert gerr == oerr == 0
    assert (got_out[0] == 0).all() if lens[0] == 0 else True   # no valid entry -> zeros


@pytest.mark.parametrize("big", [False, True])
def test_fused_heavy_ties_and_duplicate_pages(big):
    w = W.build("ties", _rows([6003, 4099, 30001, 515, 131072], big), distinct_keys=2,
                dup_mapping=True, seed=31, device=DEV)
    _check(w)


def test_fused_speculative_rows_share_pages():
    # 12 requests x 4 query tokens: rows of one request are scored from one
    # pass over its pages; each row still gets its own visible blocks
    from oracle import metadata as M
    rng = np.random.default_rng(90)
    L = [int(x) for x in rng.integers(600, 40000, size=12)]
    L[0], L[1] = 2051, 2052
    w = W.build("spec4", L, query_lens=[4] * 12, seed=91, device=DEV)
    m = M.build_metadata(w.query_start_loc.cpu().numpy(), w.seq_lens.cpu().numpy(),
                         w.cmp_page_table.cpu().numpy(), w.R, storage_block_size=128,
                         compress_ratio=4, common_slot_mapping=np.zeros(w.R, np.int64))
    w = W.Workload(**{**w.__dict__,
                      "token_to_request": torch.from_numpy(m["token_to_req"]).to(DEV),
                      "query_positions": torch.from_numpy(m["logical_positions"]).to(DEV)})
    _, _, gerr, oerr = _check(w)
    assert gerr == oerr == 0


@pytest.mark.parametrize("big", [False, True])
def test_fused_bad_ids_set_error_bits(big):
    w = W.build("bad", _rows([3000, 3000, 3000, 9000], big), seed=36, device=DEV)
    pt = w.cmp_page_table.clone()
    pt[1, 2] = w.cmp_cache.shape[0] + 5         # compressed page beyond the pool
    pt[3, 0] = -1                               # unmapped compressed page
    t2r = torch.arange(w.R, dtype=torch.int32, device=DEV)
    t2r[2] = w.R + 9                            # row 2: no such request
    got_idx, got_out, gerr, oerr = _check(w, pt=pt, t2r=t2r)
    assert gerr == oerr == (qsa.DERR_REQUEST | qsa.DERR_CMP_PAGE)
    assert (got_idx[2] == -1).all() and (got_out[2] == 0).all()


def test_fused_fp8_keys():
    w = W.config(2, device=DEV, cmp_dtype="fp8")
    _, _, gerr, oerr = _check(w, rows=list(range(0, 64, 7)))
    assert gerr == oerr == 0


def test_fused_more_rows_than_one_launch():
    # 1100 rows run as a 1024-row launch and a 76-row launch on the stream
    rng = np.random.default_rng(92)
    L = [int(x) for x in rng.integers(300, 3000, size=1100)]
    w = W.build("many", L, seed=93, device=DEV)
    _, _, gerr, oerr = _check(w, rows=[0, 1, 511, 1023, 1024, 1025, 1099])
    assert gerr == 0


def test_fused_maximum_rows_in_one_call():
    # 65535 rows (the most one call takes) of one request at different
    # positions: the selection runs in 64 row chunks, and each stream run of
    # the attention spans some 200 rows; sampled rows against the oracle
    R = 65535
    base = W.build("maxrows", [3000], seed=95, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(96)
    w = W.Workload(**{
        **base.__dict__,
        "R": R,
        "q_sel": torch.randn((R, 4, 128), generator=g, device=DEV).half(),
        "q_attn": torch.randn((R, 3, 256), generator=g, device=DEV).half(),
        "token_to_request": torch.zeros(R, dtype=torch.int32, device=DEV),
        "query_positions": torch.randint(0, 3000, (R,), generator=g, device=DEV,
                                         dtype=torch.int64)})
    _, got_out, gerr, oerr = _check(w, rows=[0, 1, 1023, 1024, 32767, 65533, 65534])
    assert gerr == oerr == 0
    assert np.isfinite(got_out).all()


@pytest.mark.parametrize("cfg", [1, 2])
def test_fused_repeat_calls_on_dirty_workspace(cfg):
    w = W.config(cfg, device=DEV)
    a_idx, a_out, _ = _fused(w)
    need = qsa.qsa_select_attend_workspace_bytes(w.R, w.cmp_page_table.shape[1])
    ws = torch.full((need,), 0xAB, dtype=torch.uint8, device=DEV)   # counters start dirty
    for _ in range(3):
        b_idx, b_out, gerr = _fused(w, workspace=ws)
        assert gerr == 0
        assert np.array_equal(a_idx, b_idx) and np.array_equal(a_out, b_out)


def test_fused_fails_closed():
    w = W.config(0, device=DEV)
    with pytest.raises(qsa.QSAError) as e:      # attention query dtype
        qsa.qsa_select_attend(w.q_sel, w.cmp_cache, w.cmp_page_table, w.token_to_request,
                              w.seq_lens, w.query_positions, w.q_attn.float(), w.k_view,
                              w.v_view, w.kv_page_table)
    assert e.value.status == 2
    with pytest.raises(qsa.QSAError) as e:      # workspace too small
        qsa.qsa_select_attend(w.q_sel, w.cmp_cache, w.cmp_page_table, w.token_to_request,
                              w.seq_lens, w.query_positions, w.q_attn, w.k_view, w.v_view,
                              w.kv_page_table,
                              workspace=torch.empty(256, dtype=torch.uint8, device=DEV))
    assert e.value.status == 7
    idx = torch.empty((1, 2051), dtype=torch.int32, device=DEV)
    with pytest.raises(qsa.QSAError) as e:      # attention output aliases the indices
        qsa.qsa_select_attend(w.q_sel, w.cmp_cache, w.cmp_page_table, w.token_to_request,
                              w.seq_lens, w.query_positions, w.q_attn, w.k_view, w.v_view,
                              w.kv_page_table, indices=idx,
                              out=idx.view(torch.float16).as_strided((1, 3, 256), (768, 256, 1)))
    assert e.value.status == 8


@pytest.mark.parametrize("rows", [1, 8, "over"])
def test_steps_captured_in_a_cuda_graph(rows):
    # serving loops capture the decode step in a CUDA graph: the one-call
    # step (the fused kernel for 1 and 8 rows, the chained kernels above the
    # fused limit) and the two calls replay bit for bit like eager calls,
    # on new inputs copied into the captured buffers
    if rows == "over":
        rows = qsa.qsa_select_attend_fused_rows() + 1
    lens = [9215, 131072, 519, 40000] * (rows // 4 + 1)
    w = W.build("graph", lens[:rows], seed=97, device=DEV)
    gen = torch.Generator(device=DEV).manual_seed(98)
    new_q = (torch.randn(w.q_sel.shape, generator=gen, device=DEV).half(),
             torch.randn(w.q_attn.shape, generator=gen, device=DEV).half())
    R, cols = w.R, w.cmp_page_table.shape[1]
    idx = torch.empty((R, 2051), dtype=torch.int32, device=DEV)
    out = torch.empty((R, 3, 256), dtype=torch.float16, device=DEV)
    ws = torch.empty(qsa.qsa_select_attend_workspace_bytes(R, cols), dtype=torch.uint8,
                     device=DEV)
    idx2 = torch.empty_like(idx)
    out2 = torch.empty_like(out)
    sws = torch.empty(qsa.qsa_select_workspace_bytes(R, cols), dtype=torch.uint8, device=DEV)
    aws = torch.empty(qsa.qsa_attention_workspace_bytes(R, 2051), dtype=torch.uint8, device=DEV)
    q_sel, q_attn = w.q_sel.clone(), w.q_attn.clone()
    side = torch.cuda.Stream()

    def one(s):
        qsa.qsa_select_attend(q_sel, w.cmp_cache, w.cmp_page_table, w.token_to_request,
                              w.seq_lens, w.query_positions, q_attn, w.k_view, w.v_view,
                              w.kv_page_table, indices=idx, out=out, workspace=ws, stream=s)

    def two(s):
        qsa.qsa_select_paged_tokens(q_sel, w.cmp_cache, w.cmp_page_table, w.token_to_request,
                                    w.seq_lens, w.query_positions, out=idx2, workspace=sws,
                                    stream=s)
        qsa.qsa_sparse_attention(q_attn, w.k_view, w.v_view, w.kv_page_table,
                                 w.token_to_request, idx2, out=out2, workspace=aws, stream=s)

    graphs = []
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        one(side)
        two(side)
        side.synchronize()
        for fn in (one, two):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                fn(side)
            graphs.append(g)
    torch.cuda.current_stream().wait_stream(side)
    for q_s, q_a in ((w.q_sel, w.q_attn), new_q):
        q_sel.copy_(q_s)
        q_attn.copy_(q_a)
        for g in graphs:
            g.replay()
        torch.cuda.synchronize()
        got = (idx.clone(), out.clone(), idx2.clone(), out2.clone())
        one(torch.cuda.current_stream())
        two(torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert torch.equal(got[0], idx) and torch.equal(got[1], out)
        assert torch.equal(got[2], idx2) and torch.equal(got[3], out2)
        assert torch.equal(idx, idx2)


def test_concurrent_streams_and_host_threads():
    # two batches (one fused, one chained) on two streams at once, from two
    # host threads (ctypes releases the GIL, so the library's per-device
    # caches and launches race for real): each result equals its batch's
    # result computed alone
    import threading
    n = qsa.qsa_select_attend_fused_rows()
    batches = [W.build("cc_a", [131072, 9215, 519, 40000] * 2, seed=31, device=DEV),
               W.build("cc_b", [70001, 3, 2052, 131072] * ((n + 4) // 4), seed=32, device=DEV)]
    assert qsa.qsa_select_attend_fused_cluster(8, batches[0].cmp_page_table.shape[1]) > 0
    assert batches[1].R > n                                   # the chained kernels

    def run(w, stream):
        ws = torch.empty(qsa.qsa_select_attend_workspace_bytes(w.R, w.cmp_page_table.shape[1]),
                         dtype=torch.uint8, device=DEV)
        res = []
        for _ in range(10):
            res.append(qsa.qsa_select_attend(w.q_sel, w.cmp_cache, w.cmp_page_table,
                                             w.token_to_request, w.seq_lens, w.query_positions,
                                             w.q_attn, w.k_view, w.v_view, w.kv_page_table,
                                             workspace=ws, stream=stream))
        stream.synchronize()
        return res

    alone = []
    for w in batches:
        s = torch.cuda.Stream()
        alone.append(run(w, s)[0])
    out = [None, None]
    errs = []

    def worker(i):
        try:
            out[i] = run(batches[i], torch.cuda.Stream())
        except Exception as e:          # reported below; a thread cannot fail the test
            errs.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errs, errs
    for i in range(2):
        for idx, o in out[i]:
            assert torch.equal(idx, alone[i][0]) and torch.equal(o, alone[i][1])


_CAPTURE_FIRST = r"""
import sys, torch
import sparse_paged_attention_qsa_gb300 as qsa
from sparse_paged_attention_qsa_gb300 import workloads as W
rows = int(sys.argv[1])
w = W.build("cap", ([131072, 9215, 519, 40000] * rows)[:rows], seed=3, device="cuda")
R, cols = w.R, w.cmp_page_table.shape[1]
idx = torch.empty((R, 2051), dtype=torch.int32, device="cuda")
out = torch.empty((R, 3, 256), dtype=torch.float16, device="cuda")
ws = torch.empty(qsa.qsa_select_attend_workspace_bytes(R, cols), dtype=torch.uint8, device="cuda")
s = torch.cuda.Stream()
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g, stream=s):     # the library's first calls in this process
    qsa.qsa_select_attend(w.q_sel, w.cmp_cache, w.cmp_page_table, w.token_to_request, w.seq_lens,
                          w.query_positions, w.q_attn, w.k_view, w.v_view, w.kv_page_table,
                          indices=idx, out=out, workspace=ws, stream=s)
g.replay()
torch.cuda.synchronize()
i2, o2 = qsa.qsa_select_attend(w.q_sel, w.cmp_cache, w.cmp_page_table, w.token_to_request,
                               w.seq_lens, w.query_positions, w.q_attn, w.k_view, w.v_view,
                               w.kv_page_table)
torch.cuda.synchronize()
sys.exit(0 if torch.equal(i2, idx) and torch.equal(o2, out) else 3)
"""


@pytest.mark.parametrize("rows", [8, 200])
def test_first_call_inside_a_graph_capture(rows):
    # a fresh process whose first calls into the library happen while a CUDA
    # graph is being captured (its one-time setup runs during the capture):
    # the fused (8 rows) and chained (200 rows) steps replay like eager calls
    import subprocess
    import sys
    root = __file__.rsplit("/tests/", 1)[0]
    r = subprocess.run([sys.executable, "-c", _CAPTURE_FIRST, str(rows)], cwd=root,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
