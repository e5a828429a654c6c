"""GPU test of qsa_select_paged_tokens_static_scratch, the selection entry
point for callers that cannot allocate device memory where they call the
library (a plugin handed only its input and output buffers, or a serving loop
that bans cudaMalloc after start-up).  It takes its scratch from an array
inside the library instead of a caller workspace.

Checks, through the C ABI: two calls in a row on each of several workloads
give exactly the indices of qsa_select_paged_tokens (the workspace entry
point); switching workloads between calls leaves no stale scratch behind;
the calls allocate no device memory (the driver's free-memory figure and
torch's allocator are unchanged across them); an empty batch returns OK and
writes nothing; a request larger than the array is refused without
launching, and a malformed one gets the workspace entry point's status, not
the scratch-limit one.

This file is collected last so a run that stops at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import pytest
import torch

import sparse_paged_attention_qsa_gb300 as qsa
from sparse_paged_attention_qsa_gb300 import build as qbuild
from sparse_paged_attention_qsa_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCRATCH_LIMIT = 10   # QSA_ERR_SCRATCH_LIMIT
SHAPE = 3            # QSA_ERR_SHAPE


def _lib():
    qbuild.build()
    lib = qsa.load_library()
    i32, i64, vp, ci = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    p64 = ctypes.POINTER(ctypes.c_int64)
    f = lib.qsa_select_paged_tokens_static_scratch
    f.restype = ci
    f.argtypes = [vp, ci, i64, p64, vp, ci, p64, p64, vp, ci, i64, i64, i64,
                  vp, ci, vp, ci, vp, ci, i32, i32, vp, ci, i64, i64, vp, vp]
    lib.qsa_static_scratch_bytes.restype = ctypes.c_size_t
    lib.qsa_static_scratch_bytes.argtypes = []
    return lib


def _a(v):
    v = list(v)
    return (ctypes.c_int64 * len(v))(*v)


def _static_select(lib, w, out, err, pt=None, rows=None):
    pt = w.cmp_page_table if pt is None else pt
    return lib.qsa_select_paged_tokens_static_scratch(
        w.q_sel.data_ptr(), 1, w.R if rows is None else rows, _a(w.q_sel.stride()),
        w.cmp_cache.data_ptr(), 1, _a(w.cmp_cache.shape), _a(w.cmp_cache.stride()),
        pt.data_ptr(), 4, pt.shape[0], pt.shape[1], pt.stride(0),
        w.token_to_request.data_ptr(), 4, w.seq_lens.data_ptr(), 4,
        w.query_positions.data_ptr(), 5, 2048, 4,
        out.data_ptr(), 4, out.shape[1], out.stride(0),
        err.data_ptr(), torch.cuda.current_stream().cuda_stream)


def test_static_scratch_matches_workspace_entry_point():
    lib = _lib()
    assert lib.qsa_static_scratch_bytes() == 4 << 20
    loads = [W.config(1, device=DEV),
             W.build("mixed", [60001, 519, 33333, 9215, 2, 48000, 1027, 20000],
                     distinct_keys=0, seed=21, device=DEV),
             W.build("ties", [30000, 12000, 515], distinct_keys=4, dup_mapping=True, seed=22,
                     device=DEV),
             W.config(0, device=DEV)]
    for w in loads:
        need = qsa.qsa_select_workspace_bytes(w.R, w.cmp_page_table.shape[1])
        assert need <= lib.qsa_static_scratch_bytes()
        ref = qsa.qsa_select_paged_tokens(w.q_sel, w.cmp_cache, w.cmp_page_table,
                                          w.token_to_request, w.seq_lens, w.query_positions)
        for _ in range(2):                       # two calls in a row
            out = torch.full((w.R, 2051), -7, dtype=torch.int32, device=DEV)
            err = torch.zeros(1, dtype=torch.int32, device=DEV)
            assert _static_select(lib, w, out, err) == 0
            torch.cuda.synchronize()
            assert torch.equal(out, ref), w.name
            assert int(err.item()) == 0


def test_static_scratch_refuses_oversized_request():
    lib = _lib()
    w = W.build("small", [515] * 8, seed=23, device=DEV)
    wide = torch.full((8, 4096), -1, dtype=torch.int32, device=DEV)   # 16 MiB of scratch
    wide[:, :w.cmp_page_table.shape[1]] = w.cmp_page_table
    out = torch.full((8, 2051), -7, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert _static_select(lib, w, out, err, pt=wide) == SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert (out == -7).all()                  # nothing was launched
    assert b"static scratch" in lib.qsa_status_string(SCRATCH_LIMIT)


def test_static_scratch_allocates_nothing():
    lib = _lib()
    w = W.build("mixed", [60001, 519, 33333, 9215], seed=24, device=DEV)
    out = torch.full((w.R, 2051), -7, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert _static_select(lib, w, out, err) == 0       # first call: any one-time set-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(5):
        assert _static_select(lib, w, out, err) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    assert torch.cuda.memory_allocated() == alloc0
    assert int(err.item()) == 0


def test_static_scratch_empty_batch_writes_nothing():
    lib = _lib()
    w = W.build("small", [515] * 2, seed=25, device=DEV)
    out = torch.full((2, 2051), -7, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert _static_select(lib, w, out, err, rows=0) == 0
    torch.cuda.synchronize()
    assert (out == -7).all()
    assert int(err.item()) == 0


def test_static_scratch_malformed_call_gets_the_argument_status():
    # 70000 rows is beyond the per-call row limit: the argument check answers
    # (QSA_ERR_SHAPE) before the scratch size is looked at
    lib = _lib()
    w = W.build("small", [515] * 2, seed=26, device=DEV)
    out = torch.full((2, 2051), -7, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert _static_select(lib, w, out, err, rows=70000) == SHAPE
    torch.cuda.synchronize()
    assert (out == -7).all()
