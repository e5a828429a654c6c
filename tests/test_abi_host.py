"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/*.h declares, answers workspace queries, and fails
closed on bad arguments -- each rejected before any CUDA call, so fake
(aligned, never dereferenced) device addresses are enough here.  Mirrors the
fail-closed dtype/layout/output checks of "vLLM: integrate FP16 packed QSA
extension" (Validation)."""
import ctypes
import glob
import os
import re
import subprocess

import pytest
import torch

import sparse_paged_attention_qsa_gb300 as qsa
from sparse_paged_attention_qsa_gb300 import build as qbuild

INC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
HDR = os.path.join(INC, "qsa.h")


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return qsa.load_library()


def _declared():
    src = "".join(open(h).read() for h in sorted(glob.glob(os.path.join(INC, "*.h"))))
    return re.findall(r"QSA_API\s+[\w\s\*]+?\b(qsa_\w+)\s*\(", src)


def test_header_declares_and_library_exports_every_symbol(lib):
    names = _declared()
    assert set(names) == set(qsa.EXPORTED), names
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", qbuild.LIB], capture_output=True,
                         text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(names) <= exported
    # nothing but the ABI leaks out of the library
    assert {e for e in exported if e.startswith("qsa")} == set(names)


def test_package_exports_every_binding_function():
    from sparse_paged_attention_qsa_gb300 import binding
    public = {n for n in dir(binding) if n.startswith("qsa_") and callable(getattr(binding, n))}
    assert public and all(getattr(qsa, n, None) is getattr(binding, n) for n in public), \
        sorted(n for n in public if not hasattr(qsa, n))


def test_header_constants_match_binding():
    src = open(HDR).read()
    consts = dict(re.findall(r"#define\s+(QSA_\w+)\s+(\d+)u?\b", src))
    assert int(consts["QSA_TOKEN_TOPK"]) == qsa.TOKEN_TOPK == 2048
    assert int(consts["QSA_COMPRESS_RATIO"]) == qsa.COMPRESS_RATIO == 4
    assert int(consts["QSA_OUT_WIDTH"]) == qsa.OUT_WIDTH == 2051
    assert int(consts["QSA_TOPK_BLOCKS"]) == qsa.TOPK_BLOCKS == 512
    assert int(consts["QSA_KV_PAGE_STRIDE"]) == 262144
    assert int(consts["QSA_V_OFFSET"]) == 256
    assert int(consts["QSA_DERR_REQUEST"]) == qsa.DERR_REQUEST
    assert int(consts["QSA_DERR_CMP_PAGE"]) == qsa.DERR_CMP_PAGE
    assert int(consts["QSA_DERR_KV_PAGE"]) == qsa.DERR_KV_PAGE


def test_status_strings_and_version(lib):
    for s in range(10):
        assert lib.qsa_status_string(s)
    assert lib.qsa_status_string(99) == b"unknown status"
    assert lib.qsa_version() >= 100


def test_workspace_queries(lib):
    assert lib.qsa_select_workspace_bytes(0, 10) == 0
    # per row: a 32-bit key per block (128 per page-table column) and the
    # largest key of each run of 16 blocks
    assert lib.qsa_select_workspace_bytes(256, 256) == 256 * 256 * (128 + 8) * 4
    assert lib.qsa_select_workspace_bytes(1, 1) % 256 == 0
    assert lib.qsa_attention_workspace_bytes(0, 2051) == 0
    a = lib.qsa_attention_workspace_bytes(256, 2051)
    assert a >= 256 * 3 * 256 * 4 and a % 256 == 0
    assert lib.qsa_attention_workspace_bytes(1, 0) > 0


# --- fail-closed selection --------------------------------------------------

A = 1 << 20          # fake device addresses: distinct, 256-byte aligned
def _addr(k):
    return A * (k + 1)


def _arr(v):
    return (ctypes.c_int64 * len(v))(*v)


def _sel(lib, **over):
    R = over.pop("R", 4)
    cols = over.pop("cols", 8)
    a = dict(q=_addr(1), qdt=1, R=R, qs=_arr([512, 128, 1]),
             cmp=_addr(2), cdt=1, cshape=_arr([64, 128, 1, 128]), cstr=_arr([16384, 128, 128, 1]),
             pt=_addr(40), ptdt=4, nreq=R, cols=cols, pts0=cols,
             t2r=_addr(50), t2rdt=4, sl=_addr(60), sldt=4, qp=_addr(70), qpdt=5,
             topk=2048, ratio=4, out=_addr(80), odt=4, ow=2051, os0=2051,
             ws=_addr(100), wsb=lib.qsa_select_workspace_bytes(R, cols), err=None, stream=None)
    a.update(over)
    return lib.qsa_select_paged_tokens(*a.values())


@pytest.mark.parametrize("over,status", [
    (dict(topk=1024), 6), (dict(ratio=8), 6), (dict(ow=2048), 6),
    (dict(qdt=3), 2), (dict(qdt=2), 2), (dict(cdt=2), 2), (dict(cdt=5), 2), (dict(ptdt=5), 2),
    (dict(cdt=6, ws=None), 7),   # E4M3 keys pass the dtype check (then: no workspace)
    (dict(t2rdt=5), 2), (dict(sldt=5), 2), (dict(qpdt=4), 2), (dict(odt=5), 2),
    (dict(R=70000), 3), (dict(R=-1), 3),
    (dict(cshape=_arr([64, 64, 1, 128])), 3), (dict(cshape=_arr([64, 128, 2, 128])), 3),
    (dict(cshape=_arr([64, 128, 1, 64])), 3),
    (dict(qs=_arr([1024, 128, 1])), 4), (dict(qs=_arr([512, 1, 4])), 4),
    (dict(cstr=_arr([16384 * 2, 128, 128, 1])), 4), (dict(cstr=_arr([16384, 256, 128, 1])), 4),
    (dict(pts0=4), 4), (dict(os0=2050), 4),
    (dict(q=None), 1), (dict(cmp=None), 1), (dict(pt=None), 1), (dict(t2r=None), 1),
    (dict(sl=None), 1), (dict(qp=None), 1), (dict(out=None), 1), (dict(qs=None), 1),
    (dict(q=_addr(1) + 8), 5), (dict(cmp=_addr(2) + 2), 5), (dict(qp=_addr(70) + 4), 5),
    (dict(out=_addr(80) + 2), 5), (dict(err=_addr(120) + 1), 5),
    (dict(ws=None), 7), (dict(wsb=100), 7), (dict(ws=_addr(100) + 16), 5),
    (dict(out=_addr(1)), 8), (dict(out=_addr(40)), 8), (dict(out=_addr(100)), 8),
    (dict(err=_addr(80) + 64), 8), (dict(err=_addr(1)), 8),
])
def test_select_fails_closed(lib, over, status):
    assert _sel(lib, **over) == status


def test_select_zero_rows_is_noop(lib):
    assert _sel(lib, R=0, ws=None, wsb=0) == 0


def _static_sel(lib, **over):
    """qsa_select_paged_tokens_static_scratch with _sel's arguments (no workspace pair)."""
    R = over.pop("R", 4)
    cols = over.pop("cols", 8)
    a = dict(q=_addr(1), qdt=1, R=R, qs=_arr([512, 128, 1]),
             cmp=_addr(2), cdt=1, cshape=_arr([64, 128, 1, 128]), cstr=_arr([16384, 128, 128, 1]),
             pt=_addr(40), ptdt=4, nreq=R, cols=cols, pts0=cols,
             t2r=_addr(50), t2rdt=4, sl=_addr(60), sldt=4, qp=_addr(70), qpdt=5,
             topk=2048, ratio=4, out=_addr(80), odt=4, ow=2051, os0=2051, err=None, stream=None)
    a.update(over)
    return lib.qsa_select_paged_tokens_static_scratch(*a.values())


@pytest.mark.parametrize("over,status", [
    # malformed calls get the workspace entry point's status, whatever their size
    (dict(R=70000), 3), (dict(cols=(1 << 20) + 1), 3), (dict(topk=1024, cols=4096), 6),
    (dict(qdt=3, cols=4096), 2), (dict(q=None, cols=4096), 1), (dict(out=_addr(1), cols=4096), 8),
    # a well-formed request beyond the array: the scratch limit, nothing launched
    (dict(cols=4096), 10), (dict(R=1024, cols=64), 10),
    (dict(R=0), 0),            # empty batch: a no-op
])
def test_static_scratch_validates_before_the_size_check(lib, over, status):
    assert lib.qsa_static_scratch_bytes() == 4 << 20
    assert _static_sel(lib, **over) == status


# --- fail-closed one-call step ---------------------------------------------

def _sa(lib, **over):
    """qsa_select_attend: the selection's and the attention's arguments."""
    R = over.pop("R", 4)
    cols = over.pop("cols", 8)
    k = over.pop("k", _addr(10))
    a = dict(q=_addr(1), qdt=1, R=R, qs=_arr([512, 128, 1]),
             cmp=_addr(2), cdt=1, cshape=_arr([64, 128, 1, 128]), cstr=_arr([16384, 128, 128, 1]),
             pt=_addr(40), ptdt=4, nreq=R, cols=cols, pts0=cols,
             t2r=_addr(50), t2rdt=4, sl=_addr(60), sldt=4, qp=_addr(70), qpdt=5,
             topk=2048, ratio=4, idx=_addr(80), idt=4, ow=2051, os0=2051,
             qa=_addr(90), qadt=1, qas=_arr([768, 256, 1]),
             k=k, v=over.pop("v", None if k is None else k + 512), kvdt=1,
             kvshape=_arr([64, 512, 1, 256]), ks=_arr([262144, 512, 256, 1]),
             vs=_arr([262144, 512, 256, 1]),
             kvpt=_addr(500), kvptdt=4, kvcols=16, kvpts0=16, scale=1.0 / 16.0,
             out=_addr(600), odt=1, os=_arr([768, 256, 1]),
             ws=_addr(700), wsb=lib.qsa_select_attend_workspace_bytes(R, cols), err=None,
             stream=None)
    a.update(over)
    return lib.qsa_select_attend(*a.values())


@pytest.mark.parametrize("over,status", [
    (dict(qdt=3), 2), (dict(cdt=2), 2), (dict(qadt=3), 2), (dict(kvdt=2), 2), (dict(odt=3), 2),
    (dict(kvptdt=5), 2), (dict(idt=5), 2),
    (dict(topk=1024), 6), (dict(scale=float("nan")), 6), (dict(scale=0.0), 6),
    (dict(R=70000), 3), (dict(kvshape=_arr([64, 256, 1, 256])), 3),
    (dict(cshape=_arr([64, 64, 1, 128])), 3),
    (dict(qas=_arr([768, 1, 3])), 4), (dict(kvpts0=8), 4), (dict(pts0=4), 4),
    (dict(qa=None), 1), (dict(k=None, v=None), 1), (dict(kvpt=None), 1), (dict(out=None), 1),
    (dict(idx=None), 1),
    (dict(qa=_addr(90) + 2), 5), (dict(out=_addr(600) + 8), 5), (dict(ws=_addr(700) + 16), 5),
    (dict(ws=None), 7), (dict(wsb=16), 7),
    (dict(out=_addr(80)), 8), (dict(out=_addr(700)), 8), (dict(idx=_addr(1)), 8),
    (dict(idx=_addr(700)), 8), (dict(err=_addr(600)), 8), (dict(err=_addr(80)), 8),
])
def test_select_attend_fails_closed(lib, over, status):
    # every rejection comes from the host checks, before any launch
    assert _sa(lib, **over) == status


def test_fused_path_queries_without_a_device_answer(lib):
    # the answers that need no device: other key types, empty batches, more
    # rows than the kernel takes, tables wider than 128 columns per row
    assert lib.qsa_select_attend_fused_rows(4) == 0          # int32 tag
    assert lib.qsa_select_attend_fused_cluster(1, 2, 4) == 0
    assert lib.qsa_select_attend_fused_cluster(0, 2, 1) == 0
    assert lib.qsa_select_attend_fused_cluster(-3, 2, 1) == 0
    assert lib.qsa_select_attend_fused_cluster(257, 2, 1) == 0
    assert lib.qsa_select_attend_fused_cluster(2, 257, 1) == 0
    assert lib.qsa_select_attend_fused_cluster(1 << 40, 2, 1) == 0


def test_select_attend_zero_rows_is_noop(lib):
    assert lib.qsa_select_attend_workspace_bytes(0, 8) == 0
    assert _sa(lib, R=0, ws=None, wsb=0) == 0


# --- fail-closed attention --------------------------------------------------

def _att(lib, **over):
    R = over.pop("R", 2)
    W = over.pop("W", 2051)
    k = over.pop("k", _addr(10))
    a = dict(q=_addr(1), qdt=1, R=R, qs=_arr([768, 256, 1]),
             k=k, v=over.pop("v", None if k is None else k + 512), kvdt=1, kvshape=_arr([64, 512, 1, 256]),
             ks=_arr([262144, 512, 256, 1]), vs=_arr([262144, 512, 256, 1]),
             pt=_addr(500), ptdt=4, nreq=R, cols=16, pts0=16, t2r=_addr(510), t2rdt=4,
             idx=_addr(520), idxdt=4, W=W, is0=W, scale=1.0 / 16.0,
             out=_addr(600), odt=1, os=_arr([768, 256, 1]),
             ws=_addr(700), wsb=lib.qsa_attention_workspace_bytes(R, W), err=None, stream=None)
    a.update(over)
    return lib.qsa_sparse_attention(*a.values())


@pytest.mark.parametrize("over,status", [
    (dict(qdt=3), 2), (dict(kvdt=2), 2), (dict(odt=3), 2), (dict(ptdt=5), 2),
    (dict(t2rdt=5), 2), (dict(idxdt=5), 2),
    (dict(scale=float("nan")), 6), (dict(scale=0.0), 6), (dict(scale=-1.0), 6),
    (dict(scale=float("inf")), 6), (dict(W=2052, is0=2052), 6),
    (dict(R=70000), 3), (dict(kvshape=_arr([64, 256, 1, 256])), 3),
    (dict(kvshape=_arr([64, 512, 2, 256])), 3), (dict(kvshape=_arr([64, 512, 1, 512])), 3),
    (dict(qs=_arr([768, 1, 3])), 4), (dict(os=_arr([1024, 256, 1])), 4),
    (dict(ks=_arr([131072, 256, 256, 1])), 4), (dict(vs=_arr([262144, 256, 256, 1])), 4),
    (dict(ks=_arr([262144, 512, 256, 2])), 4), (dict(v=_addr(10)), 4), (dict(v=_addr(10) + 1024), 4),
    (dict(pts0=8), 4), (dict(is0=100), 4),
    (dict(q=None), 1), (dict(k=None, v=None), 1), (dict(pt=None), 1), (dict(t2r=None), 1),
    (dict(idx=None), 1), (dict(out=None), 1), (dict(ks=None), 1),
    (dict(q=_addr(1) + 2), 5), (dict(k=_addr(10) + 8), 5), (dict(out=_addr(600) + 8), 5),
    (dict(idx=_addr(520) + 2), 5),
    (dict(ws=None), 7), (dict(wsb=16), 7),
    (dict(out=_addr(1)), 8), (dict(out=_addr(10) + 4096), 8), (dict(out=_addr(520)), 8),
    (dict(out=_addr(700)), 8), (dict(err=_addr(600)), 8),
])
def test_attention_fails_closed(lib, over, status):
    assert _att(lib, **over) == status


def test_attention_zero_rows_and_zero_width(lib):
    assert _att(lib, R=0, ws=None, wsb=0) == 0


def test_binding_raises_without_library(tmp_path):
    import importlib
    import sparse_paged_attention_qsa_gb300.binding as b
    saved = b._lib
    try:
        b._lib = None
        with pytest.raises(RuntimeError, match="not found"):
            b.load_library(str(tmp_path / "missing.so"))
    finally:
        b._lib = saved


# --- fail-closed metadata builder -------------------------------------------

def _meta(lib, **over):
    T = over.pop("T", 300)
    a = dict(qsl=_addr(1), qsldt=4, sl=_addr(2), sldt=4, common=_addr(3), cdt=5,
             bt=_addr(4), btdt=4, rows=8, cols=16, s0=16, s1=1,
             nreq=8, nmapped=T, T=T, sbs=128, cr=4, cbs=0,
             t2r=_addr(10), lpos=_addr(11), vis=_addr(12), slot=_addr(13),
             work=_addr(14), maxw=64, stream=None)
    a.update(over)
    return lib.qsa_build_metadata(*a.values())


@pytest.mark.parametrize("over,status", [
    (dict(qsldt=5), 2), (dict(sldt=5), 2), (dict(btdt=5), 2), (dict(cdt=4), 2),
    (dict(nreq=0), 3), (dict(T=-1), 3), (dict(T=1 << 31), 3), (dict(nmapped=-1), 3),
    (dict(maxw=-1), 3), (dict(rows=7), 3), (dict(cols=-1), 3),
    (dict(sbs=0), 6), (dict(cr=0), 6), (dict(cbs=-1), 6), (dict(cr=1 << 31), 6),
    (dict(s0=0), 4), (dict(s1=0), 4),
    (dict(qsl=None), 1), (dict(sl=None), 1), (dict(t2r=None), 1), (dict(lpos=None), 1),
    (dict(vis=None), 1), (dict(slot=None), 1), (dict(bt=None), 1), (dict(common=None), 1),
    (dict(work=None), 1),
    (dict(qsl=_addr(1) + 2), 5), (dict(lpos=_addr(11) + 4), 5), (dict(slot=_addr(13) + 4), 5),
    (dict(common=_addr(3) + 4), 5), (dict(work=_addr(14) + 2), 5),
    (dict(t2r=_addr(11)), 8), (dict(slot=_addr(3)), 8), (dict(vis=_addr(10) + 1024), 8),
    (dict(work=_addr(4)), 8), (dict(lpos=_addr(1)), 8),
])
def test_metadata_fails_closed(lib, over, status):
    assert _meta(lib, **over) == status


def test_metadata_nothing_to_do_and_optional_inputs(lib):
    assert _meta(lib, T=0, maxw=0, work=None) == 0
    # circular mode ignores common_slot_mapping (and its dtype tag)
    assert _meta(lib, T=0, maxw=0, work=None, cbs=8, common=None, cdt=0) == 0
    # a table without columns needs no pointer; no tokens need no outputs
    assert _meta(lib, T=0, maxw=0, work=None, cols=0, bt=None) == 0
    assert _meta(lib, T=0, maxw=0, work=None, t2r=None, lpos=None, vis=None, slot=None,
                 common=None) == 0


# --- fail-closed indexer ------------------------------------------------------

def _logits(lib, **over):
    a = dict(q=_addr(1), qdt=6, rows=8, heads=64, kv=_addr(2), kvdt=6, nblocks=100, bs=64,
             w=_addr(3), wdt=3, ctx=_addr(4), ctxdt=4, batch=4, bt=_addr(5), btdt=4, cols=16,
             bts0=16, next_n=2, out=_addr(10), odt=3, mml=4096, ld=4096, err=None, stream=None)
    a.update(over)
    return lib.qsa_paged_mqa_logits(*a.values())


@pytest.mark.parametrize("over,status", [
    (dict(qdt=1), 2), (dict(kvdt=1), 2), (dict(wdt=1), 2), (dict(odt=1), 2), (dict(ctxdt=5), 2),
    (dict(btdt=5), 2),
    (dict(heads=48), 3), (dict(heads=8), 3), (dict(next_n=0), 3), (dict(next_n=5), 3),
    (dict(heads=128, next_n=4, rows=16), 3), (dict(bs=48), 3), (dict(bs=4), 3),
    (dict(rows=9), 3), (dict(batch=-1), 3), (dict(nblocks=-1), 3), (dict(mml=-1), 3),
    (dict(bts0=8), 4), (dict(ld=100), 4),
    (dict(q=None), 1), (dict(w=None), 1), (dict(ctx=None), 1), (dict(out=None), 1),
    (dict(kv=None), 1), (dict(bt=None), 1),
    (dict(q=_addr(1) + 8), 5), (dict(kv=_addr(2) + 4), 5), (dict(w=_addr(3) + 4), 5),
    (dict(ctx=_addr(4) + 2), 5), (dict(out=_addr(10) + 2), 5),
    (dict(out=_addr(1)), 8), (dict(out=_addr(2) + 4096), 8), (dict(out=_addr(5)), 8),
    (dict(err=_addr(10) + 64), 8),
])
def test_paged_mqa_logits_fails_closed(lib, over, status):
    assert _logits(lib, **over) == status


def test_paged_mqa_logits_nothing_to_do(lib):
    assert _logits(lib, rows=0, batch=0) == 0
    assert _logits(lib, mml=0, ld=0) == 0


def _topk(lib, **over):
    a = dict(lg=_addr(1), lgdt=3, rows=8, cols=4096, s0=4096, s1=1, next_n=2, sl=_addr(2),
             sldt=4, batch=4, topk=2048, out=_addr(10), odt=4, os0=2048, stream=None)
    a.update(over)
    return lib.qsa_top_k_per_row_decode(*a.values())


@pytest.mark.parametrize("over,status", [
    (dict(lgdt=1), 2), (dict(sldt=5), 2), (dict(odt=5), 2),
    (dict(rows=9), 3), (dict(next_n=0), 3), (dict(cols=-1), 3),
    (dict(topk=0), 6), (dict(topk=2049), 6),
    (dict(s1=0), 4), (dict(os0=100), 4), (dict(s0=0), 4),
    (dict(lg=None), 1), (dict(sl=None), 1), (dict(out=None), 1),
    (dict(lg=_addr(1) + 2), 5), (dict(out=_addr(10) + 2), 5),
    (dict(out=_addr(1)), 8), (dict(out=_addr(2)), 8),
])
def test_top_k_per_row_fails_closed(lib, over, status):
    assert _topk(lib, **over) == status


def test_top_k_per_row_nothing_to_do(lib):
    assert _topk(lib, rows=0, batch=0) == 0


def test_fused_cost_fit_constants_agree():
    # the fused-or-chained rule in csrc/qsa_fused.h, the figures include/qsa.h
    # states for it, and the copy of the rule the GPU tests check the
    # library's choice against must stay one rule
    from tests import test_gpu_fused as tf
    src = open(os.path.join(os.path.dirname(INC), "sparse_paged_attention_qsa_gb300", "csrc",
                            "qsa_fused.h")).read()
    c = {k: int(v) for k, v in re.findall(r"(k(?:Fused|Chain)\w+Cost) = (\d+)", src)}
    assert c == {"kFusedBaseCost": 40000, "kFusedPageCost": 1440, "kChainBaseCost": 80000,
                 "kChainPageCost": 10}
    # in microseconds: 25 + 0.9 per page of a CTA against 50 + 0.00625 per page of the batch
    assert (c["kFusedBaseCost"] / 1600, c["kFusedPageCost"] / 1600) == (25.0, 0.9)
    assert (c["kChainBaseCost"] / 1600, c["kChainPageCost"] / 1600) == (50.0, 0.00625)
    hdr = open(HDR).read()
    assert "25 us + 0.9 us per page" in hdr and "50 us + 6.25 ns per page" in hdr
    for R, cols, cs in ((1, 2, 16), (32, 256, 4), (48, 256, 2), (64, 256, 2), (100, 256, 1),
                        (152, 256, 1)):
        fused = c["kFusedBaseCost"] + c["kFusedPageCost"] * -(-cols // cs)
        chain = c["kChainBaseCost"] + c["kChainPageCost"] * R * cols
        assert tf._fused_wins(R, cols, cs) == (fused <= chain)


def test_binding_rejects_host_tensors(lib):
    # host (CPU) tensors would reach the kernels as invalid device addresses:
    # the binding refuses them before calling the library
    from sparse_paged_attention_qsa_gb300 import workloads as W
    w = W.config(0, device="cpu")
    calls = [
        lambda: qsa.qsa_select_paged_tokens(w.q_sel, w.cmp_cache, w.cmp_page_table,
                                            w.token_to_request, w.seq_lens, w.query_positions),
        lambda: qsa.qsa_sparse_attention(w.q_attn, w.k_view, w.v_view, w.kv_page_table,
                                         w.token_to_request,
                                         torch.zeros((1, 2051), dtype=torch.int32)),
        lambda: qsa.qsa_select_attend(w.q_sel, w.cmp_cache, w.cmp_page_table,
                                      w.token_to_request, w.seq_lens, w.query_positions,
                                      w.q_attn, w.k_view, w.v_view, w.kv_page_table),
    ]
    for call in calls:
        with pytest.raises(qsa.QSAError) as e:
            call()
        assert e.value.status == 1 and "device memory" in str(e.value)
