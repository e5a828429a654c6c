"""GPU parity for qsa_sparse_attention: the CUDA path through the C ABI vs the
binary64 oracle, max |err| <= 2e-3 ("vLLM: integrate FP16 packed QSA
extension", "Exact contracts"/Attention; the page's attention suite: R in
{1,2} across empty, holes/duplicates/cross-page, valid width 32 and full
width 2051, plus fail-closed dtype/layout checks).

Tolerance: outputs are convex combinations of FP16 V values (|V| < 6 for
N(0,1) draws); FP32 accumulation over <= 2051 terms errs by ~1e-6 relative
and the final FP16 rounding by <= 2^-11 relative (<= 1.5e-3 at |o| < 3),
so 2e-3 absolute -- the bound the path is specified to -- holds with margin.
"""
import numpy as np
import pytest
import torch

import sparse_paged_attention_qsa_gb300 as qsa
from sparse_paged_attention_qsa_gb300 import workloads as W
from tests._util import CORES, oracle_attention, oracle_select, stream_edge_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = 2e-3


def _gpu(w, idx, **kw):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = qsa.qsa_sparse_attention(w.q_attn, w.k_view, w.v_view, kw.get("pt", w.kv_page_table),
                                   kw.get("t2r", w.token_to_request), idx,
                                   scale=kw.get("scale", 1.0 / 16.0), error_word=err)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), int(err.item())


def _check(w, idx, rows=None, **kw):
    got, gerr = _gpu(w, idx, **kw)
    exp, oerr = oracle_attention(w, idx, rows=rows, kv_page_table=kw.get("pt"),
                                 token_to_request=kw.get("t2r"),
                                 scale=kw.get("scale", 1.0 / 16.0))
    rows = list(range(w.R)) if rows is None else list(rows)
    diff = np.abs(got[rows] - exp).max() if rows else 0.0
    assert diff <= TOL, f"max abs error {diff}"
    return got, gerr, oerr, diff


def _lists(R, widths, L, seed, hole=0.1, dup=0.05):
    w = W.build("idx", [L] * R, premade_widths=widths, hole_frac=hole, dup_frac=dup, seed=seed,
                device=DEV)
    return w


@pytest.mark.parametrize("R", [1, 2])
@pytest.mark.parametrize("case", ["empty", "holes_dups_cross_page", "width32", "width2051"])
def test_attention_page_suite(R, case):
    widths = {"empty": [0], "holes_dups_cross_page": [1500], "width32": [32],
              "width2051": [2051]}[case]
    hole = 0.0 if case in ("width32", "width2051") else 0.1
    dup = 0.0 if case in ("width32", "width2051") else 0.05
    w = _lists(R, widths, 3000, seed=R * 10 + len(case), hole=hole, dup=dup)
    got, gerr, _, _ = _check(w, w.indices)
    assert gerr == 0
    if case == "empty":
        assert (got == 0).all()


@pytest.mark.parametrize("cfg", [0, 1, 2])
def test_attention_on_selected_indices(cfg):
    w = W.config(cfg, device=DEV)
    idx = qsa.qsa_select_paged_tokens(w.q_sel, w.cmp_cache, w.cmp_page_table,
                                      w.token_to_request, w.seq_lens, w.query_positions)
    # the oracle attends over the oracle's own selection (bit-exact by the
    # selection tests; checked again here)
    sel, _ = oracle_select(w)
    assert np.array_equal(idx.cpu().numpy(), sel)
    _, gerr, oerr, _ = _check(w, torch.from_numpy(sel).to(DEV))
    assert gerr == oerr == 0


def test_attention_config3_premade_lists():
    w = W.config(3, device=DEV)      # widths {0,1,32,1024,2051}, 10% holes, 5% dups
    _, gerr, oerr, _ = _check(w, w.indices)
    assert gerr == oerr == 0


def config4_attention_rows(R):
    """At least 32 rows of the 256-row batch: every row that starts or ends at
    a boundary of the stream split's runs (and its neighbour), the first and
    last rows, filled up with every 8th row."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rows = set(stream_edge_rows(R, 2051, sms)) | {0, 1, R - 2, R - 1}
    r = 0
    while len(rows) < 32:
        rows.add(r)
        r += 8
    return sorted(rows)


def test_attention_config4_full_size_many_rows():
    w = W.config(4, device=DEV)
    idx = qsa.qsa_select_paged_tokens(w.q_sel, w.cmp_cache, w.cmp_page_table,
                                      w.token_to_request, w.seq_lens, w.query_positions)
    got, gerr = _gpu(w, idx)
    assert gerr == 0
    rows = config4_attention_rows(w.R)
    assert len(rows) >= 32
    exp, oerr = oracle_attention(w, idx, rows=rows, threads=CORES)
    assert oerr == 0
    assert np.abs(got[rows] - exp).max() <= TOL
    assert np.isfinite(got).all()


@pytest.mark.parametrize("R", [16, 32, 33, 40])
def test_attention_batch_sizes_around_the_split_switch(R):
    # batches of up to 32 rows take 64-entry splits, larger ones the stream
    # split: premade lists with holes and duplicates, every width, bad ids
    w = _lists(R, [0, 1, 32, 1024, 2051, 1500, 77], 3000, seed=60 + R)
    pt = w.kv_page_table.clone()
    pt[1, 0] = -1                                   # an unmapped K/V page
    t2r = torch.arange(R, dtype=torch.int32, device=DEV)
    t2r[R - 1] = R + 5                              # the last row has no request
    got, gerr, oerr, _ = _check(w, w.indices, pt=pt, t2r=t2r)
    assert gerr == oerr
    assert (got[R - 1] == 0).all()


@pytest.mark.parametrize("R,L,width", [(33, 3000, 0), (33, 3000, 1), (40, 3000, 33),
                                        (97, 3000, 300), (300, 2100, 2051), (1100, 700, 2051),
                                        (1100, 700, 77)])
def test_attention_stream_runs_across_rows(R, L, width):
    # batches of more than 32 rows: the index lists cut into 32-entry chunks
    # laid end to end and split into equal runs, one per CTA of one wave; a
    # run spans two rows (or three at 1100 rows), a row several runs
    valid = [min(v, L) for v in (2051, 1500, 77, 0, 32, 513)]
    w = _lists(R, valid, L, seed=70 + R + width)
    idx = w.indices[:, :width].contiguous()
    rows = sorted({0, 1, R // 3, R // 2, R - 2, R - 1})
    got, gerr, oerr, _ = _check(w, idx, rows=rows)
    assert gerr == oerr == 0
    assert np.isfinite(got).all()
    if width == 0:
        assert (got == 0).all()


def test_attention_single_index_exact():
    w = W.build("one", [5000, 5000], seed=3, device=DEV)
    idx = torch.full((2, 2051), -1, dtype=torch.int32, device=DEV)
    idx[0, 2050] = 4999
    idx[1, 0] = 512
    got, _ = _gpu(w, idx)
    kv = w.kv_cache.float().cpu().numpy()
    pt = w.kv_page_table.cpu().numpy()
    for r, t in ((0, 4999), (1, 512)):
        v = kv[pt[r, t // 512], t % 512, 1]
        assert np.array_equal(got[r], np.stack([v] * 3))


def test_attention_short_width_and_other_scale():
    w = _lists(3, [5, 40, 300], 700, seed=9)
    idx = w.indices[:, :300].contiguous()       # width 300 (< 2051)
    _check(w, idx)
    _check(w, idx, scale=0.3)


def test_attention_bad_ids_are_holes():
    w = _lists(3, [2051], 2000, seed=4)
    pt = w.kv_page_table.clone()
    pt[0, 1] = -1
    pt[1, 0] = w.kv_cache.shape[0] + 3
    t2r = torch.tensor([0, 1, 17], dtype=torch.int32, device=DEV)
    got, gerr, oerr, _ = _check(w, w.indices, pt=pt, t2r=t2r)
    assert gerr == oerr == (qsa.DERR_REQUEST | qsa.DERR_KV_PAGE)
    assert (got[2] == 0).all()


def test_attention_index_beyond_table_is_hole():
    w = _lists(1, [100], 1000, seed=5, hole=0, dup=0)
    idx = w.indices.clone()
    idx[0, 7] = 10 ** 7                              # column beyond the table
    _, gerr, oerr, _ = _check(w, idx)
    assert gerr == oerr == qsa.DERR_KV_PAGE


def test_attention_fail_closed_dtypes_and_layout():
    w = _lists(1, [64], 1000, seed=6)
    ok = [w.q_attn, w.k_view, w.v_view, w.kv_page_table, w.token_to_request, w.indices]

    def expect(status, *a, **kw):
        with pytest.raises(qsa.QSAError) as e:
            qsa.qsa_sparse_attention(*a, **kw)
        assert e.value.status == status

    expect(2, w.q_attn.float(), *ok[1:])
    expect(2, w.q_attn.bfloat16(), *ok[1:])
    kvb = w.kv_cache.bfloat16()
    expect(2, ok[0], kvb[:, :, 0:1], kvb[:, :, 1:2], *ok[3:])
    expect(2, *ok[:3], w.kv_page_table.long(), *ok[4:])
    expect(2, *ok[:5], w.indices.long())
    expect(2, *ok, out=torch.empty((1, 3, 256), dtype=torch.float32, device=DEV))
    # V not at storage offset 256 of K's buffer
    expect(4, ok[0], w.k_view, w.k_view, *ok[3:])
    # K/V with a non-contract layout (separate contiguous tensors)
    kc = w.k_view.contiguous()
    vc = w.v_view.contiguous()
    expect(4, ok[0], kc, vc, *ok[3:])
    # wrong head dim / scale / width
    expect(3, ok[0], w.kv_cache[:, :, 0:1, :128], w.kv_cache[:, :, 1:2, :128], *ok[3:])
    expect(6, *ok, scale=float("nan"))
    expect(6, *ok[:5], torch.full((1, 2052), -1, dtype=torch.int32, device=DEV))
