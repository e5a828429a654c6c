"""GPU parity for qsa_select_paged_tokens: the CUDA path through the C ABI vs
the oracle, bit-exact on every index ("vLLM: integrate FP16 packed QSA
extension", "Exact contracts"/Selection; the page's selection suite: empty,
short tail, full page, cross-page tail, duplicate physical-page mapping,
exact-score ties, P8192 saturated width 2051, multi-request, fail-closed
dtype/output checks)."""
import numpy as np
import pytest
import torch

import sparse_paged_attention_qsa_gb300 as qsa
from sparse_paged_attention_qsa_gb300 import workloads as W
from tests._util import CORES, oracle_select

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _gpu(w, **kw):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = qsa.qsa_select_paged_tokens(w.q_sel, w.cmp_cache, kw.get("pt", w.cmp_page_table),
                                      kw.get("t2r", w.token_to_request), w.seq_lens,
                                      w.query_positions, error_word=err)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(err.item())


def _check(w, rows=None, **kw):
    got, gerr = _gpu(w, **kw)
    exp, oerr = oracle_select(w, rows=rows, cmp_page_table=kw.get("pt"),
                              token_to_request=kw.get("t2r"))
    rows = list(range(w.R)) if rows is None else list(rows)
    for i, r in enumerate(rows):
        if not np.array_equal(got[r], exp[i]):
            bad = np.nonzero(got[r] != exp[i])[0]
            raise AssertionError(f"row {r}: {len(bad)} mismatches, first at {bad[0]}: "
                                 f"got {got[r][bad[0]:bad[0]+8]} expected {exp[i][bad[0]:bad[0]+8]}")
    return got, gerr, oerr


@pytest.mark.parametrize("cfg", [0, 1, 3])
def test_select_configs_small(cfg):
    w = W.config(cfg, device=DEV)
    _, gerr, oerr = _check(w)
    assert gerr == oerr == 0


def test_select_config2_decode_batch():
    w = W.config(2, device=DEV)
    _, gerr, oerr = _check(w)
    assert gerr == oerr == 0


def test_select_config4_full_size_all_rows():
    # the long-context workload (256 rows x 131072 tokens), every row bit for
    # bit against the oracle (all 65536 compressed pages go to the host)
    w = W.config(4, device=DEV)
    got, gerr = _gpu(w)
    assert gerr == 0
    exp, oerr = oracle_select(w, threads=CORES)
    assert oerr == 0
    bad = [r for r in range(w.R) if not np.array_equal(got[r], exp[r])]
    assert not bad, f"rows differing from the oracle: {bad[:10]}"
    # 131072 is a multiple of 4, so the query token completes the last group
    # and the tail is empty (columns 2048..2050 stay -1)
    assert (got[:, :2048] >= 0).all() and (got[:, 2048:] == -1).all()


@pytest.mark.parametrize("lens", [[0], [1], [3], [4], [7], [515], [516], [519], [512 + 3, 1027]])
def test_select_short_empty_and_full_page(lens):
    # 0..7 tokens: empty / short tails; 515 = exactly one full compressed page
    # + 3-token tail; 516/519/1027 cross page boundaries
    w = W.build("edge", lens, seed=sum(lens) + 1, device=DEV)
    _check(w)


def test_select_speculative_positions():
    lens = [5000, 5000, 5000, 5000, 700]
    pos = [4999, 4998, 4997, 4996, 1000]      # pos >= L clamps to L//4 blocks
    w = W.build("spec", lens, positions=pos, seed=3, device=DEV)
    _check(w)


def test_select_exact_ties_and_duplicate_pages():
    w = W.build("ties", [6003, 4099, 30001, 515], distinct_keys=4, dup_mapping=True, seed=12,
                device=DEV)
    _check(w)


@pytest.mark.parametrize("distinct", [2, 4])
def test_select_long_rows_heavy_ties(distinct):
    # rows longer than the top-k's 8192-key candidate list: with 2 distinct
    # keys about half of a 32768-block row ties at the largest score (the
    # candidates overflow: select over the whole row); with 4, a quarter
    # (the lower-bound sweep, then the tie rule over the candidates)
    w = W.build("longties", [131072, 40003, 65539], distinct_keys=distinct, seed=13 + distinct,
                device=DEV)
    _check(w)


def test_select_rows_longer_than_the_staged_unit_maxima():
    # 300003 tokens: 75000 blocks, 4688 unit maxima (more than the 4096 the
    # top-k stages in shared memory: it reads them from the workspace)
    w = W.build("verylong", [300003, 262147, 5000], seed=15, device=DEV)
    _check(w)


@pytest.mark.parametrize("cols", [64, 65])
@pytest.mark.parametrize("distinct", [0, 3])
def test_select_short_row_top_k_boundary(cols, distinct):
    # a page table of at most 64 columns (every row <= 8192 blocks) takes the
    # top-k that loads all of a row's keys as candidates; 65 columns the one
    # that goes through the unit maxima -- both bit-exact at the boundary
    # (rows of exactly 8192 blocks, shorter rows, ties)
    lens = [32768, 32768 + 3, 32767, 8195, 2051]
    w = W.build("cols", lens, cmp_cols=cols, distinct_keys=distinct, seed=40 + cols + distinct,
                device=DEV)
    assert w.cmp_page_table.shape[1] == cols
    _, gerr, oerr = _check(w)
    assert gerr == oerr == 0


def test_select_all_zero_scores_long_row():
    # every key equals bits(+0)+1: 32768 ties, kept in block order
    w = W.build("zeros_long", [131072], seed=14, device=DEV)
    w.q_sel.zero_()
    got, _, _ = _check(w)
    assert got[0, :2048].tolist() == list(range(2048))


def test_select_all_zero_scores():
    w = W.build("zeros", [9215, 2051], seed=4, device=DEV)
    w.q_sel.zero_()
    got, _, _ = _check(w)
    assert got[0, :8].tolist() == [0, 1, 2, 3, 4, 5, 6, 7]


def test_select_multi_request_rows():
    w = W.build("multi", [12000, 600, 20000], seed=5, device=DEV)
    t2r = torch.tensor([2, 0, 1], dtype=torch.int32, device=DEV)
    w2 = W.Workload(**{**w.__dict__, "token_to_request": t2r,
                       "query_positions": w.query_positions[[2, 0, 1]].contiguous()})
    _check(w2)


def test_select_bad_ids_set_error_bits():
    w = W.build("bad", [3000, 3000, 3000], seed=6, device=DEV)
    pt = w.cmp_page_table.clone()
    pt[1, 2] = w.cmp_cache.shape[0] + 5        # page beyond the pool
    pt[2, 0] = -1                               # unmapped page
    t2r = torch.tensor([0, 1, 9], dtype=torch.int32, device=DEV)   # row 2: no such request
    got, gerr, oerr = _check(w, pt=pt, t2r=t2r)
    assert gerr == oerr == (qsa.DERR_REQUEST | qsa.DERR_CMP_PAGE)
    assert (got[2] == -1).all()


def test_select_padded_page_table_and_output_stride():
    w = W.build("stride", [4000, 9000], seed=7, device=DEV)
    wide = torch.full((2, w.cmp_page_table.shape[1] + 13), -7, dtype=torch.int32, device=DEV)
    wide[:, :w.cmp_page_table.shape[1]] = w.cmp_page_table
    pt = wide[:, :w.cmp_page_table.shape[1]]           # row stride > columns
    out_buf = torch.full((2, 2051 + 5), 123, dtype=torch.int32, device=DEV)
    out = out_buf[:, :2051]
    qsa.qsa_select_paged_tokens(w.q_sel, w.cmp_cache, pt, w.token_to_request, w.seq_lens,
                                w.query_positions, out=out)
    torch.cuda.synchronize()
    exp, _ = oracle_select(w)
    assert np.array_equal(out.cpu().numpy(), exp)
    assert (out_buf[:, 2051:] == 123).all()


def test_select_repeat_calls_deterministic():
    w = W.config(1, device=DEV)
    a, _ = _gpu(w)
    ws = torch.full((qsa.qsa_select_workspace_bytes(1, w.cmp_page_table.shape[1]),), 0xAB,
                    dtype=torch.uint8, device=DEV)   # dirty workspace must not matter
    b = qsa.qsa_select_paged_tokens(w.q_sel, w.cmp_cache, w.cmp_page_table, w.token_to_request,
                                    w.seq_lens, w.query_positions, workspace=ws).cpu().numpy()
    assert np.array_equal(a, b)


def test_select_fail_closed_dtypes_and_output():
    w = W.config(0, device=DEV)
    args = [w.q_sel, w.cmp_cache, w.cmp_page_table, w.token_to_request, w.seq_lens,
            w.query_positions]
    bad = [
        (0, w.q_sel.float(), 2), (0, w.q_sel.bfloat16(), 2), (1, w.cmp_cache.float(), 2),
        (2, w.cmp_page_table.long(), 2), (3, w.token_to_request.long(), 2),
        (4, w.seq_lens.long(), 2), (5, w.query_positions.int(), 2),
    ]
    for pos, t, status in bad:
        a = list(args)
        a[pos] = t
        with pytest.raises(qsa.QSAError) as e:
            qsa.qsa_select_paged_tokens(*a)
        assert e.value.status == status
    with pytest.raises(qsa.QSAError) as e:           # output dtype
        qsa.qsa_select_paged_tokens(*args, out=torch.empty((1, 2051), dtype=torch.int64, device=DEV))
    assert e.value.status == 2
    with pytest.raises(qsa.QSAError) as e:           # output width
        qsa.qsa_select_paged_tokens(*args, out=torch.empty((1, 2048), dtype=torch.int32, device=DEV))
    assert e.value.status == 6
    with pytest.raises(qsa.QSAError) as e:           # contract constants
        qsa.qsa_select_paged_tokens(*args, token_topk=1024)
    assert e.value.status == 6
    with pytest.raises(qsa.QSAError) as e:           # non-contiguous query
        qsa.qsa_select_paged_tokens(w.q_sel.transpose(1, 2).contiguous().transpose(1, 2), *args[1:])
    assert e.value.status == 4


# --- FP8-E4M3 compressed keys (qsa_cache.py: the optional e4m3 compressed
# indexer cache); same score rule and order, bit-exact indices ---------------

@pytest.mark.parametrize("cfg", [0, 1, 2, 3])
def test_select_fp8_configs(cfg):
    w = W.config(cfg, device=DEV, cmp_dtype="fp8")
    assert w.cmp_cache.dtype == torch.float8_e4m3fn
    _, gerr, oerr = _check(w)
    assert gerr == oerr == 0


def test_select_fp8_config4_all_rows():
    w = W.config(4, device=DEV, cmp_dtype="fp8")
    got, gerr = _gpu(w)
    assert gerr == 0
    exp, oerr = oracle_select(w, threads=CORES)
    assert oerr == 0
    bad = [r for r in range(w.R) if not np.array_equal(got[r], exp[r])]
    assert not bad, f"rows differing from the oracle: {bad[:10]}"
    assert (got[:, :2048] >= 0).all() and (got[:, 2048:] == -1).all()


def test_select_fp8_edges_ties_and_bad_pages():
    w = W.build("fp8edge", [0, 3, 515, 4099, 30001], distinct_keys=4, dup_mapping=True,
                cmp_dtype="fp8", seed=41, device=DEV)
    pt = w.cmp_page_table.clone()
    pt[3, 5] = w.cmp_cache.shape[0] + 1
    got, gerr, oerr = _check(w, pt=pt)
    assert gerr == oerr == qsa.DERR_CMP_PAGE


def test_select_fp8_matches_fp16_on_identical_values():
    # E4M3 keys and the same values stored as fp16 must select identically
    w8 = W.build("same", [20003, 777], cmp_dtype="fp8", seed=42, device=DEV)
    w16 = W.Workload(**{**w8.__dict__, "cmp_cache": w8.cmp_cache.to(torch.float16)})
    a, _ = _gpu(w8)
    b, _ = _gpu(w16)
    assert np.array_equal(a, b)
