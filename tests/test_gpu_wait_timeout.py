"""Failure detection on the GPU: a device wait that runs out.

The score kernel's consumers wait on an mbarrier for each page the producer
streams in; every such wait is bounded, and when one gives up the kernel
stops, lets the copies it issued land, sets QSA_DERR_TIMEOUT in the error
word and returns, so the context stays usable.  Nothing in a healthy run
makes such a wait run out, so this test loads libqsa_waittest.so, a build of
the same sources compiled with QSA_WAIT_TEST: its stage waits give up after
2 ms, and one extra symbol makes the first CTA of the score kernel (or of
the fused small-batch kernel) leave one stage fill without a copy (no
arrive ever comes for it).  No trap, no bad address and no endless loop is
involved: the wait ends by its own limit.

Checks: the call that withholds a fill returns quickly with the timeout bit
set; the next call on the same stream and workspace is bit-exact again
(against the product library); the same holds for the one-call step
qsa_select_attend -- through the fused small-batch kernel and through the
chained kernels -- whose top-k and attention run over the partial scores of
the aborted scoring without leaving their buffers.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

import sparse_paged_attention_qsa_gb300 as qsa
from sparse_paged_attention_qsa_gb300 import build as qbuild
from sparse_paged_attention_qsa_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
WITHHELD_FILL = 2        # the third page the first CTA streams


def _wait_test_lib():
    lib = ctypes.CDLL(qbuild.build_wait_test())
    qsa.declare_signatures(lib)
    lib.qsa_test_withhold_score_fill.restype = None
    lib.qsa_test_withhold_score_fill.argtypes = [ctypes.c_int64]
    return lib


def _workload(rows=16):
    # rows x 65536 tokens: at 16 rows 2048 compressed pages over the score
    # kernel's CTAs (one per SM), at 40 rows 5120; either way CTA 0 streams
    # more than WITHHELD_FILL + 1 pages, as does the first CTA of the fused
    # small-batch kernel's first cluster (128 pages over 4 to 16 CTAs)
    return W.build("waits", [65536] * rows, seed=51, device=DEV)


def _select(w, lib, ws, err):
    out = qsa.qsa_select_paged_tokens(w.q_sel, w.cmp_cache, w.cmp_page_table,
                                      w.token_to_request, w.seq_lens, w.query_positions,
                                      workspace=ws, error_word=err, library=lib)
    torch.cuda.synchronize()
    return out


def test_selection_wait_runs_out_then_next_call_is_exact():
    lib = _wait_test_lib()
    w = _workload()
    ref = qsa.qsa_select_paged_tokens(w.q_sel, w.cmp_cache, w.cmp_page_table,
                                      w.token_to_request, w.seq_lens, w.query_positions)
    ws = torch.empty(qsa.qsa_select_workspace_bytes(w.R, w.cmp_page_table.shape[1]),
                     dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.qsa_test_withhold_score_fill(-1)
    assert torch.equal(_select(w, lib, ws, err), ref)        # the test build, healthy
    assert int(err.item()) == 0
    try:
        lib.qsa_test_withhold_score_fill(WITHHELD_FILL)
        t0 = time.perf_counter()
        _select(w, lib, ws, err)
        dt = time.perf_counter() - t0
    finally:
        lib.qsa_test_withhold_score_fill(-1)
    assert int(err.item()) & qsa.DERR_TIMEOUT, int(err.item())
    assert dt < 5.0, dt                   # 2 ms waits; the drain only waits for issued copies
    err.zero_()
    again = _select(w, lib, ws, err)      # same stream, same (now stale) workspace
    assert int(err.item()) == 0
    assert torch.equal(again, ref)
    # the product library on the same context is unaffected
    assert torch.equal(qsa.qsa_select_paged_tokens(w.q_sel, w.cmp_cache, w.cmp_page_table,
                                                   w.token_to_request, w.seq_lens,
                                                   w.query_positions), ref)


@pytest.mark.parametrize("rows", [16, "over"])
def test_one_call_step_wait_runs_out_then_next_call_is_exact(rows):
    # 16 rows: the fused small-batch kernel (one cluster per row); one row
    # above its limit: the chained score, top-k and attention kernels
    lib = _wait_test_lib()
    if rows == "over":
        rows = qsa.qsa_select_attend_fused_rows() + 1
    assert (qsa.qsa_select_attend_fused_cluster(rows, 128) > 0) == (rows == 16)
    w = _workload(rows)
    ref_idx, ref_out = qsa.qsa_select_attend(w.q_sel, w.cmp_cache, w.cmp_page_table,
                                             w.token_to_request, w.seq_lens, w.query_positions,
                                             w.q_attn, w.k_view, w.v_view, w.kv_page_table)
    ws = torch.empty(qsa.qsa_select_attend_workspace_bytes(w.R, w.cmp_page_table.shape[1]),
                     dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)

    def step():
        idx, out = qsa.qsa_select_attend(w.q_sel, w.cmp_cache, w.cmp_page_table,
                                         w.token_to_request, w.seq_lens, w.query_positions,
                                         w.q_attn, w.k_view, w.v_view, w.kv_page_table,
                                         workspace=ws, error_word=err, library=lib)
        torch.cuda.synchronize()
        return idx, out

    try:
        lib.qsa_test_withhold_score_fill(WITHHELD_FILL)
        _, out = step()
    finally:
        lib.qsa_test_withhold_score_fill(-1)
    assert int(err.item()) & qsa.DERR_TIMEOUT, int(err.item())
    err.zero_()
    idx, out = step()
    assert int(err.item()) == 0
    assert torch.equal(idx, ref_idx)
    assert np.array_equal(out.cpu().numpy(), ref_out.cpu().numpy())   # the same kernels
