"""Plain CPU oracle for the QSA sparse decode path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (``cpu_baseline`` / ``--impl reference``) may import this package.  The
product library never imports, links or calls it, and it shares no code with
the CUDA path: the C source next to this file is compiled on its own with gcc.

What it computes is restated from the pages in ``qsa_oracle.c``:
selection follows "vLLM: integrate FP16 packed QSA extension" (Summary,
"Exact contracts"/Selection) with the visible-block rule of qsa_cache.py
(_build_qsa_metadata_kernel); attention follows the same page's
"Exact contracts"/Attention, evaluated in binary64.

Every function here is pinned by ``tests/test_oracle_*.py`` against brute
force, closed forms and invariants.  Parity status per function:
  - ``score``            pinned (exact-sum cases, hand-derived rounding cases,
                          error bound against the exact dot product)
  - ``select``           pinned (brute-force rank, special cases, invariants)
  - ``attention``        pinned (dense-softmax brute force via scipy, single
                          index, equal keys, hole/permutation invariance)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qsa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libqsa_oracle.so")

TOKEN_TOPK = 2048
COMPRESS_RATIO = 4
TOPK_BLOCKS = 512
OUT_WIDTH = 2051
ERR_REQUEST = 1
ERR_CMP_PAGE = 2
ERR_KV_PAGE = 4

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, no fast-math, no contraction)."""
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC),
                                               os.path.getmtime(os.path.join(_HERE, "qsa_oracle.h"))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        i64, u32, vp = ctypes.c_int64, ctypes.c_uint32, ctypes.c_void_p
        lib.qsa_oracle_half_to_double.restype = ctypes.c_double
        lib.qsa_oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.qsa_oracle_e4m3_to_double.restype = ctypes.c_double
        lib.qsa_oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.qsa_oracle_score_e4m3.restype = ctypes.c_float
        lib.qsa_oracle_score_e4m3.argtypes = [vp, vp]
        lib.qsa_oracle_select_keys.restype = u32
        lib.qsa_oracle_select_keys.argtypes = [i64, vp, ctypes.c_int, vp, i64, vp, i64, i64, i64,
                                               vp, vp, vp, vp, i64]
        lib.qsa_oracle_score.restype = ctypes.c_float
        lib.qsa_oracle_score.argtypes = [vp, vp]
        lib.qsa_oracle_visible_blocks.restype = i64
        lib.qsa_oracle_visible_blocks.argtypes = [i64, i64]
        lib.qsa_oracle_tail_end.restype = i64
        lib.qsa_oracle_tail_end.argtypes = [i64, i64]
        sel_args = [i64, vp, vp, i64, vp, i64, i64, i64, vp, vp, vp, vp, i64]
        lib.qsa_oracle_select.restype = u32
        lib.qsa_oracle_select.argtypes = sel_args
        lib.qsa_oracle_select_scored.restype = u32
        lib.qsa_oracle_select_scored.argtypes = sel_args + [vp]
        lib.qsa_oracle_attention.restype = u32
        lib.qsa_oracle_attention.argtypes = [i64, vp, vp, i64, vp, i64, i64, i64, vp,
                                             vp, i64, ctypes.c_double, vp]
        _lib = lib
        return lib


def _u16(a) -> np.ndarray:
    """fp16 array (or its uint16 bits) -> C-contiguous uint16 bits."""
    a = np.asarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected float16/uint16, got {a.dtype}")
    return np.ascontiguousarray(a)


def _u8(a) -> np.ndarray:
    """E4M3 bytes (uint8, or any 1-byte dtype) -> C-contiguous uint8."""
    a = np.asarray(a)
    if a.dtype.itemsize != 1:
        raise TypeError(f"expected 1-byte elements, got {a.dtype}")
    return np.ascontiguousarray(a.view(np.uint8))


KEY_F16, KEY_E4M3 = 0, 1


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


class PagePool:
    """Physical page pool given to the oracle as one pointer per page id.

    ``pages`` is either a contiguous array whose first axis is the page id, or
    a dict {page_id: page array} for a pool of ``num_pages`` where only some
    pages are present (the rest read as absent).  ``kind`` is KEY_F16 (fp16
    elements, also used for K/V pages) or KEY_E4M3 (one byte per element).
    Pages are kept alive here.
    """

    def __init__(self, pages, num_pages: int | None = None, page_halves: int = 0,
                 kind: int = KEY_F16):
        self._keep = []
        self.kind = kind
        conv = _u8 if kind == KEY_E4M3 else _u16
        esize = 1 if kind == KEY_E4M3 else 2
        if isinstance(pages, dict):
            if num_pages is None:
                raise ValueError("num_pages is required for a sparse pool")
            self.num_pages = int(num_pages)
            arr = (ctypes.c_void_p * max(self.num_pages, 1))()
            for pid, pg in pages.items():
                pg = conv(pg)
                if page_halves and pg.size != page_halves:
                    raise ValueError("page of wrong size")
                self._keep.append(pg)
                arr[int(pid)] = _ptr(pg)
        else:
            pool = conv(pages)
            self.num_pages = int(pool.shape[0]) if num_pages is None else int(num_pages)
            self._keep.append(pool)
            arr = (ctypes.c_void_p * max(self.num_pages, 1))()
            if pool.shape[0]:
                per = pool[0].size
                if page_halves and per != page_halves:
                    raise ValueError("page of wrong size")
                base = _ptr(pool)
                for p in range(min(self.num_pages, pool.shape[0])):
                    arr[p] = base + esize * per * p
        self.array = arr


def half_to_double(bits: int) -> float:
    return _load().qsa_oracle_half_to_double(int(bits) & 0xFFFF)


def e4m3_to_double(bits: int) -> float:
    return _load().qsa_oracle_e4m3_to_double(int(bits) & 0xFF)


def score_e4m3(q_sel_row, key_bytes) -> np.float32:
    """Canonical binary32 score of one E4M3 key [128 bytes] against q [4,128]."""
    q = _u16(q_sel_row).reshape(4, 128)
    k = _u8(key_bytes).reshape(128)
    return np.float32(_load().qsa_oracle_score_e4m3(_ptr(q), _ptr(k)))


def score(q_sel_row, key) -> np.float32:
    """Canonical binary32 score of one key [128] against q [4,128]."""
    q = _u16(q_sel_row).reshape(4, 128)
    k = _u16(key).reshape(128)
    return np.float32(_load().qsa_oracle_score(_ptr(q), _ptr(k)))


def visible_blocks(seq_len: int, pos: int) -> int:
    return int(_load().qsa_oracle_visible_blocks(int(seq_len), int(pos)))


def tail_end(seq_len: int, pos: int) -> int:
    return int(_load().qsa_oracle_tail_end(int(seq_len), int(pos)))


def _row_chunks(R: int, threads: int):
    threads = max(1, min(threads, R))
    step = (R + threads - 1) // threads
    return [(s, min(R, s + step)) for s in range(0, R, step)]


def select(q_sel, cmp_pool, cmp_page_table, token_to_request, seq_lens,
           query_positions, out_width: int = OUT_WIDTH, return_scores: bool = False,
           threads: int = 1):
    """Selection for all rows; returns (indices [R,out_width] int32, err bits
    [, scores [R,512] float32]).  ``cmp_pool`` is a PagePool or an array
    [P,128,1,128] of fp16 keys or of E4M3 key bytes (any 1-byte dtype).  Rows are independent; ``threads`` splits them over
    OS threads (the C code itself is single-threaded)."""
    lib = _load()
    q = _u16(q_sel).reshape(-1, 4, 128)
    R = q.shape[0]
    if isinstance(cmp_pool, PagePool):
        pool = cmp_pool
    else:
        kind = KEY_E4M3 if np.asarray(cmp_pool).dtype.itemsize == 1 else KEY_F16
        pool = PagePool(cmp_pool, page_halves=128 * 128, kind=kind)
    if pool.kind == KEY_E4M3 and return_scores:
        raise ValueError("return_scores is only implemented for fp16 keys")
    pt = np.ascontiguousarray(np.asarray(cmp_page_table, dtype=np.int32))
    if pt.ndim != 2:
        raise ValueError("page table must be 2-D")
    t2r = np.ascontiguousarray(np.asarray(token_to_request, dtype=np.int32).reshape(R))
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32).reshape(-1))
    qp = np.ascontiguousarray(np.asarray(query_positions, dtype=np.int64).reshape(R))
    if pt.shape[0] < sl.shape[0]:
        raise ValueError("page table needs one row per request")
    out = np.empty((R, out_width), dtype=np.int32)
    scores = np.empty((R, TOPK_BLOCKS), dtype=np.float32) if return_scores else None
    errs = []

    def run(lo, hi):
        n = hi - lo
        if n <= 0:
            return 0
        args = [n, _ptr(q) + lo * 4 * 128 * 2, pool.array, pool.num_pages, _ptr(pt),
                sl.shape[0], pt.shape[1], pt.shape[1], _ptr(t2r) + lo * 4, _ptr(sl),
                _ptr(qp) + lo * 8, _ptr(out) + lo * out_width * 4, out_width]
        if return_scores:
            return lib.qsa_oracle_select_scored(*args, _ptr(scores) + lo * TOPK_BLOCKS * 4)
        if pool.kind == KEY_E4M3:
            return lib.qsa_oracle_select_keys(args[0], args[1], KEY_E4M3, *args[2:])
        return lib.qsa_oracle_select(*args)

    chunks = _row_chunks(R, threads)
    if len(chunks) <= 1:
        errs = [run(0, R)]
    else:
        with ThreadPoolExecutor(len(chunks)) as ex:
            errs = list(ex.map(lambda c: run(*c), chunks))
    err = 0
    for e in errs:
        err |= int(e)
    if return_scores:
        return out, err, scores
    return out, err


def attention(q_attn, kv_pool, kv_page_table, token_to_request, indices,
              scale: float = 1.0 / 16.0, threads: int = 1):
    """Sparse attention for all rows in binary64; returns (out [R,3,256]
    float64, err bits).  ``kv_pool`` is a PagePool or an array
    [P,512,1,512] fp16 (token t of a page: K = halves 0..255, V = 256..511)."""
    lib = _load()
    q = _u16(q_attn).reshape(-1, 3, 256)
    R = q.shape[0]
    pool = kv_pool if isinstance(kv_pool, PagePool) else PagePool(kv_pool, page_halves=512 * 512)
    pt = np.ascontiguousarray(np.asarray(kv_page_table, dtype=np.int32))
    t2r = np.ascontiguousarray(np.asarray(token_to_request, dtype=np.int32).reshape(R))
    idx = np.ascontiguousarray(np.asarray(indices, dtype=np.int32).reshape(R, -1))
    width = idx.shape[1]
    num_reqs = int(pt.shape[0])
    out = np.empty((R, 3, 256), dtype=np.float64)

    def run(lo, hi):
        n = hi - lo
        if n <= 0:
            return 0
        return lib.qsa_oracle_attention(
            n, _ptr(q) + lo * 3 * 256 * 2, pool.array, pool.num_pages, _ptr(pt), num_reqs,
            pt.shape[1], pt.shape[1], _ptr(t2r) + lo * 4, _ptr(idx) + lo * width * 4, width,
            float(scale), _ptr(out) + lo * 3 * 256 * 8)

    chunks = _row_chunks(R, threads)
    if len(chunks) <= 1:
        errs = [run(0, R)]
    else:
        with ThreadPoolExecutor(len(chunks)) as ex:
            errs = list(ex.map(lambda c: run(*c), chunks))
    err = 0
    for e in errs:
        err |= int(e)
    return out, err
