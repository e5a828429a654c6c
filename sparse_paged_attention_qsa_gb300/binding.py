"""Thin ctypes binding over libqsa (include/qsa.h).

Argument marshalling only: tensors become (data pointer, dtype tag, shape,
strides); the stream is torch's current CUDA stream unless given.  Every step
of the computation runs in libqsa's CUDA kernels.  PyTorch is used here for
device memory (outputs and workspaces the caller did not pass) and streams.

If libqsa.so has not been built the first call raises -- there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqsa.so")

TOKEN_TOPK = 2048
COMPRESS_RATIO = 4
TOPK_BLOCKS = 512
OUT_WIDTH = 2051
DERR_REQUEST, DERR_CMP_PAGE, DERR_KV_PAGE, DERR_TIMEOUT = 1, 2, 4, 8
DERR_IDX_BLOCK = 16
IDX_HEAD_DIM, IDX_MAX_TOPK = 128, 2048

DT_F16, DT_BF16, DT_F32, DT_I32, DT_I64, DT_F8E4M3 = 1, 2, 3, 4, 5, 6
_DTYPE_TAG = {torch.float16: DT_F16, torch.bfloat16: DT_BF16, torch.float32: DT_F32,
              torch.int32: DT_I32, torch.int64: DT_I64, torch.float8_e4m3fn: DT_F8E4M3}

STATUS = {0: "QSA_OK", 1: "QSA_ERR_NULL", 2: "QSA_ERR_DTYPE", 3: "QSA_ERR_SHAPE",
          4: "QSA_ERR_STRIDE", 5: "QSA_ERR_ALIGN", 6: "QSA_ERR_CONTRACT",
          7: "QSA_ERR_WORKSPACE", 8: "QSA_ERR_ALIAS", 9: "QSA_ERR_CUDA",
          10: "QSA_ERR_SCRATCH_LIMIT"}

EXPORTED = ("qsa_status_string", "qsa_version", "qsa_select_workspace_bytes",
            "qsa_select_paged_tokens", "qsa_attention_workspace_bytes",
            "qsa_sparse_attention", "qsa_select_attend_workspace_bytes", "qsa_select_attend",
            "qsa_select_attend_fused_rows",
            "qsa_select_attend_fused_cluster",
            "qsa_static_scratch_bytes",
            "qsa_select_paged_tokens_static_scratch", "qsa_build_metadata",
            "qsa_paged_mqa_logits", "qsa_top_k_per_row_decode")


class QSAError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


_lock = threading.Lock()
_lib = None


def load_library(path: str | None = None):
    """Load libqsa.so (once) and declare the C signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(
                f"libqsa.so not found at {path}; build it with "
                "`python -m sparse_paged_attention_qsa_gb300.build` (nvcc, sm_103a)")
        lib = ctypes.CDLL(path)
        declare_signatures(lib)
        _lib = lib
        return lib


class _Only:
    """Attribute access on a library that may lack some entry points (a
    test build carries a subset): missing ones are skipped."""

    def __init__(self, lib):
        self._lib = lib

    def __getattr__(self, name):
        try:
            return getattr(self._lib, name)
        except AttributeError:
            return _Sink()


class _Sink:
    def __setattr__(self, name, value):
        pass


def declare_signatures(lib):
    """Declare the C signatures of include/*.h on a loaded library handle."""
    full = lib
    lib = _Only(full)
    i32, i64, u64, vp, sz = (ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64,
                             ctypes.c_void_p, ctypes.c_size_t)
    p64 = ctypes.POINTER(ctypes.c_int64)
    lib.qsa_status_string.restype = ctypes.c_char_p
    lib.qsa_status_string.argtypes = [ctypes.c_int]
    lib.qsa_version.restype = ctypes.c_int
    lib.qsa_version.argtypes = []
    lib.qsa_select_workspace_bytes.restype = sz
    lib.qsa_select_workspace_bytes.argtypes = [i64, i64]
    lib.qsa_attention_workspace_bytes.restype = sz
    lib.qsa_attention_workspace_bytes.argtypes = [i64, i64]
    lib.qsa_select_paged_tokens.restype = ctypes.c_int
    lib.qsa_select_paged_tokens.argtypes = [
        vp, ctypes.c_int, i64, p64,
        vp, ctypes.c_int, p64, p64,
        vp, ctypes.c_int, i64, i64, i64,
        vp, ctypes.c_int, vp, ctypes.c_int, vp, ctypes.c_int,
        i32, i32,
        vp, ctypes.c_int, i64, i64,
        vp, sz, vp, vp]
    lib.qsa_static_scratch_bytes.restype = sz
    lib.qsa_static_scratch_bytes.argtypes = []
    lib.qsa_select_paged_tokens_static_scratch.restype = ctypes.c_int
    lib.qsa_select_paged_tokens_static_scratch.argtypes = [
        vp, ctypes.c_int, i64, p64,
        vp, ctypes.c_int, p64, p64,
        vp, ctypes.c_int, i64, i64, i64,
        vp, ctypes.c_int, vp, ctypes.c_int, vp, ctypes.c_int,
        i32, i32,
        vp, ctypes.c_int, i64, i64,
        vp, vp]
    lib.qsa_sparse_attention.restype = ctypes.c_int
    lib.qsa_sparse_attention.argtypes = [
        vp, ctypes.c_int, i64, p64,
        vp, vp, ctypes.c_int, p64, p64, p64,
        vp, ctypes.c_int, i64, i64, i64,
        vp, ctypes.c_int,
        vp, ctypes.c_int, i64, i64,
        ctypes.c_float,
        vp, ctypes.c_int, p64,
        vp, sz, vp, vp]
    lib.qsa_select_attend_fused_rows.restype = i64
    lib.qsa_select_attend_fused_rows.argtypes = [ctypes.c_int]
    lib.qsa_select_attend_fused_cluster.restype = i64
    lib.qsa_select_attend_fused_cluster.argtypes = [i64, i64, ctypes.c_int]
    lib.qsa_select_attend_workspace_bytes.restype = sz
    lib.qsa_select_attend_workspace_bytes.argtypes = [i64, i64]
    lib.qsa_select_attend.restype = ctypes.c_int
    lib.qsa_select_attend.argtypes = [
        vp, ctypes.c_int, i64, p64,
        vp, ctypes.c_int, p64, p64,
        vp, ctypes.c_int, i64, i64, i64,
        vp, ctypes.c_int, vp, ctypes.c_int, vp, ctypes.c_int,
        i32, i32,
        vp, ctypes.c_int, i64, i64,
        vp, ctypes.c_int, p64,
        vp, vp, ctypes.c_int, p64, p64, p64,
        vp, ctypes.c_int, i64, i64,
        ctypes.c_float,
        vp, ctypes.c_int, p64,
        vp, sz, vp, vp]
    lib.qsa_build_metadata.restype = ctypes.c_int
    lib.qsa_build_metadata.argtypes = [
        vp, ctypes.c_int, vp, ctypes.c_int, vp, ctypes.c_int,
        vp, ctypes.c_int, i64, i64, i64, i64,
        i64, i64, i64, i64, i64, i64,
        vp, vp, vp, vp, vp, i64, vp]
    lib.qsa_paged_mqa_logits.restype = ctypes.c_int
    lib.qsa_paged_mqa_logits.argtypes = [
        vp, ctypes.c_int, i64, i64,
        vp, ctypes.c_int, i64, i64,
        vp, ctypes.c_int,
        vp, ctypes.c_int, i64,
        vp, ctypes.c_int, i64, i64,
        i64,
        vp, ctypes.c_int, i64, i64,
        vp, vp]
    lib.qsa_top_k_per_row_decode.restype = ctypes.c_int
    lib.qsa_top_k_per_row_decode.argtypes = [
        vp, ctypes.c_int, i64, i64, i64, i64, i64,
        vp, ctypes.c_int, i64,
        i64, vp, ctypes.c_int, i64, vp]
    return full


def _arr(vals):
    vals = list(vals)
    return (ctypes.c_int64 * len(vals))(*vals)


def _tag(t: torch.Tensor) -> int:
    return _DTYPE_TAG.get(t.dtype, 0)


def _ptr(t: torch.Tensor | None) -> int | None:
    # the library reads and writes device memory only: a host tensor's address
    # would reach a kernel as an invalid device address
    if t is None:
        return None
    if t.device.type != "cuda":
        raise QSAError(1, f"every tensor must be in CUDA device memory (got a {t.device} tensor)")
    return t.data_ptr() or None


def _on_current_device(*tensors):
    """Every tensor given must be in the memory of the current CUDA device,
    which the library runs on: a host tensor, or one on another GPU, would
    reach a kernel as an invalid address."""
    cur = None
    for t in tensors:
        if t is None:
            continue
        d = t.get_device()                  # -1: host memory
        if d < 0:
            raise QSAError(1, f"every tensor must be in CUDA device memory (got a {t.device} "
                              "tensor)")
        if cur is None:
            cur = torch.cuda.current_device()
        if d != cur:
            raise QSAError(1, f"a tensor is on cuda:{d} but the current device is cuda:{cur} "
                              "(select it with torch.cuda.device)")


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int):
    if status != 0:
        raise QSAError(status, load_library().qsa_status_string(status).decode())


def qsa_select_workspace_bytes(num_rows: int, cmp_pt_cols: int) -> int:
    return int(load_library().qsa_select_workspace_bytes(num_rows, cmp_pt_cols))


def qsa_attention_workspace_bytes(num_rows: int, index_width: int) -> int:
    return int(load_library().qsa_attention_workspace_bytes(num_rows, index_width))


def _workspace(nbytes: int, device) -> torch.Tensor:
    # torch's CUDA allocator returns 512-byte aligned blocks
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def qsa_select_paged_tokens(q_sel, cmp_cache, cmp_page_table, token_to_request, seq_lens,
                            query_positions, token_topk: int = TOKEN_TOPK,
                            compress_ratio: int = COMPRESS_RATIO, out=None, workspace=None,
                            error_word=None, stream=None, library=None):
    """Selection: returns out [R,2051] int32 (see include/qsa.h).  `library`:
    another loaded build of the C ABI (declare_signatures) instead of libqsa."""
    lib = library or load_library()
    _on_current_device(q_sel, cmp_cache, cmp_page_table, token_to_request, seq_lens,
                       query_positions, out, workspace, error_word)
    R = q_sel.shape[0] if q_sel.dim() == 3 else -1
    if q_sel.dim() != 3 or cmp_cache.dim() != 4 or cmp_page_table.dim() != 2:
        raise QSAError(3, "q_sel must be [R,4,128], cmp_cache [P,128,1,128], page table 2-D")
    if tuple(q_sel.shape[1:]) != (4, 128):
        raise QSAError(3, "q_sel must be [R,4,128]")
    if out is None:
        out = torch.empty((R, OUT_WIDTH), dtype=torch.int32, device=q_sel.device)
    if cmp_page_table.stride(1) != 1 and cmp_page_table.shape[1] > 1:
        raise QSAError(4, "page table columns must be contiguous")
    if out.dim() != 2 or (out.stride(1) != 1 and out.shape[1] > 1):
        raise QSAError(4, "out must be [R,2051] with contiguous columns")
    cols = cmp_page_table.shape[1]
    need = qsa_select_workspace_bytes(R, cols)
    if workspace is None:
        workspace = _workspace(need, q_sel.device)
    st = lib.qsa_select_paged_tokens(
        _ptr(q_sel), _tag(q_sel), R, _arr(q_sel.stride()),
        _ptr(cmp_cache), _tag(cmp_cache), _arr(cmp_cache.shape), _arr(cmp_cache.stride()),
        _ptr(cmp_page_table), _tag(cmp_page_table), cmp_page_table.shape[0], cols,
        cmp_page_table.stride(0),
        _ptr(token_to_request), _tag(token_to_request), _ptr(seq_lens), _tag(seq_lens),
        _ptr(query_positions), _tag(query_positions),
        int(token_topk), int(compress_ratio),
        _ptr(out), _tag(out), out.shape[1], out.stride(0),
        _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(error_word), _stream(stream))
    _check(st)
    return out


def qsa_sparse_attention(q, k_cache, v_cache, kv_page_table, token_to_request, indices,
                         scale: float = 1.0 / 16.0, out=None, workspace=None, error_word=None,
                         stream=None):
    """Sparse attention: returns out [R,3,256] FP16 (see include/qsa.h).
    k_cache / v_cache are the exact-packed views (strides [262144,512,256,1],
    V at storage offset 256 of the same buffer)."""
    lib = load_library()
    _on_current_device(q, k_cache, v_cache, kv_page_table, token_to_request, indices, out,
                       workspace, error_word)
    if q.dim() != 3 or k_cache.dim() != 4 or v_cache.dim() != 4 or indices.dim() != 2:
        raise QSAError(3, "q [R,3,256], k/v [P,512,1,256], indices [R,W] expected")
    if k_cache.shape != v_cache.shape:
        raise QSAError(3, "k_cache and v_cache shapes differ")
    R = q.shape[0]
    if out is None:
        out = torch.empty((R, 3, 256), dtype=torch.float16, device=q.device)
    if kv_page_table.dim() != 2 or (kv_page_table.stride(1) != 1 and kv_page_table.shape[1] > 1):
        raise QSAError(4, "page table must be 2-D with contiguous columns")
    if indices.stride(1) != 1 and indices.shape[1] > 1:
        raise QSAError(4, "index columns must be contiguous")
    width = indices.shape[1]
    need = qsa_attention_workspace_bytes(R, width)
    if workspace is None:
        workspace = _workspace(need, q.device)
    st = lib.qsa_sparse_attention(
        _ptr(q), _tag(q), R, _arr(q.stride()),
        _ptr(k_cache), _ptr(v_cache), _tag(k_cache) if k_cache.dtype == v_cache.dtype else 0,
        _arr(k_cache.shape), _arr(k_cache.stride()), _arr(v_cache.stride()),
        _ptr(kv_page_table), _tag(kv_page_table), kv_page_table.shape[0], kv_page_table.shape[1],
        kv_page_table.stride(0),
        _ptr(token_to_request), _tag(token_to_request),
        _ptr(indices), _tag(indices), width, indices.stride(0),
        float(scale),
        _ptr(out), _tag(out), _arr(out.stride()),
        _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(error_word), _stream(stream))
    _check(st)
    return out


def qsa_decode(q_sel, cmp_cache, cmp_page_table, token_to_request, seq_lens, query_positions,
               q_attn, k_cache, v_cache, kv_page_table, scale: float = 1.0 / 16.0,
               indices=None, out=None, sel_workspace=None, att_workspace=None,
               error_word=None, stream=None):
    """One decode step of the whole path: selection then sparse attention on
    the same stream (the index list stays on the device)."""
    indices = qsa_select_paged_tokens(q_sel, cmp_cache, cmp_page_table, token_to_request,
                                      seq_lens, query_positions, out=indices,
                                      workspace=sel_workspace, error_word=error_word,
                                      stream=stream)
    out = qsa_sparse_attention(q_attn, k_cache, v_cache, kv_page_table, token_to_request,
                               indices, scale=scale, out=out, workspace=att_workspace,
                               error_word=error_word, stream=stream)
    return indices, out


def qsa_select_attend_workspace_bytes(num_rows: int, cmp_pt_cols: int) -> int:
    return int(load_library().qsa_select_attend_workspace_bytes(num_rows, cmp_pt_cols))


def qsa_select_attend_fused_rows(cmp_dtype=torch.float16) -> int:
    """The largest batch qsa_select_attend runs as one fused kernel on the
    current device (include/qsa.h)."""
    return int(load_library().qsa_select_attend_fused_rows(_DTYPE_TAG.get(cmp_dtype, 0)))


def qsa_select_attend_fused_cluster(num_rows: int, cmp_pt_cols: int,
                                    cmp_dtype=torch.float16) -> int:
    """CTAs per row's cluster with which qsa_select_attend runs this batch
    as one fused kernel on the current device, 0 = the chained kernels
    (include/qsa.h)."""
    return int(load_library().qsa_select_attend_fused_cluster(
        num_rows, cmp_pt_cols, _DTYPE_TAG.get(cmp_dtype, 0)))


def qsa_select_attend(q_sel, cmp_cache, cmp_page_table, token_to_request, seq_lens,
                      query_positions, q_attn, k_cache, v_cache, kv_page_table,
                      scale: float = 1.0 / 16.0, indices=None, out=None, workspace=None,
                      error_word=None, stream=None, library=None):
    """One decode step in one call (include/qsa.h, qsa_select_attend): the
    selection's indices [R,2051] int32 and the attention output [R,3,256]
    FP16.  Both page tables are indexed by token_to_request.  `library` as in
    qsa_select_paged_tokens."""
    lib = library or load_library()
    _on_current_device(q_sel, cmp_cache, cmp_page_table, token_to_request, seq_lens,
                       query_positions, q_attn, k_cache, v_cache, kv_page_table, indices, out,
                       workspace, error_word)
    if q_sel.dim() != 3 or cmp_cache.dim() != 4 or cmp_page_table.dim() != 2:
        raise QSAError(3, "q_sel must be [R,4,128], cmp_cache [P,128,1,128], page table 2-D")
    if q_attn.dim() != 3 or k_cache.dim() != 4 or v_cache.dim() != 4 or kv_page_table.dim() != 2:
        raise QSAError(3, "q_attn [R,3,256], k/v [P,512,1,256], K/V page table 2-D expected")
    if k_cache.shape != v_cache.shape:
        raise QSAError(3, "k_cache and v_cache shapes differ")
    if kv_page_table.shape[0] != cmp_page_table.shape[0]:
        raise QSAError(3, "both page tables need one row per request")
    for t in (cmp_page_table, kv_page_table):
        if t.stride(1) != 1 and t.shape[1] > 1:
            raise QSAError(4, "page table columns must be contiguous")
    R = q_sel.shape[0]
    if indices is None:
        indices = torch.empty((R, OUT_WIDTH), dtype=torch.int32, device=q_sel.device)
    if indices.dim() != 2 or (indices.stride(1) != 1 and indices.shape[1] > 1):
        raise QSAError(4, "indices must be [R,2051] with contiguous columns")
    if out is None:
        out = torch.empty((R, 3, 256), dtype=torch.float16, device=q_sel.device)
    cols = cmp_page_table.shape[1]
    need = qsa_select_attend_workspace_bytes(R, cols)
    if workspace is None:
        workspace = _workspace(need, q_sel.device)
    st = lib.qsa_select_attend(
        _ptr(q_sel), _tag(q_sel), R, _arr(q_sel.stride()),
        _ptr(cmp_cache), _tag(cmp_cache), _arr(cmp_cache.shape), _arr(cmp_cache.stride()),
        _ptr(cmp_page_table), _tag(cmp_page_table), cmp_page_table.shape[0], cols,
        cmp_page_table.stride(0),
        _ptr(token_to_request), _tag(token_to_request), _ptr(seq_lens), _tag(seq_lens),
        _ptr(query_positions), _tag(query_positions),
        TOKEN_TOPK, COMPRESS_RATIO,
        _ptr(indices), _tag(indices), indices.shape[1], indices.stride(0),
        _ptr(q_attn), _tag(q_attn), _arr(q_attn.stride()),
        _ptr(k_cache), _ptr(v_cache), _tag(k_cache) if k_cache.dtype == v_cache.dtype else 0,
        _arr(k_cache.shape), _arr(k_cache.stride()), _arr(v_cache.stride()),
        _ptr(kv_page_table), _tag(kv_page_table), kv_page_table.shape[1],
        kv_page_table.stride(0),
        float(scale),
        _ptr(out), _tag(out), _arr(out.stride()),
        _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(error_word), _stream(stream))
    _check(st)
    return indices, out


def qsa_build_metadata(query_start_loc, seq_lens, block_table, num_tokens: int, *,
                       storage_block_size: int, compress_ratio: int,
                       circular_buffer_size: int = 0, common_slot_mapping=None,
                       num_mapped_tokens: int | None = None, max_num_work: int = 0,
                       out=None, stream=None):
    """Side-cache metadata (include/qsa_metadata.h).  Returns a dict of
    device tensors: token_to_req int32, logical_positions int64,
    visible_blocks int32, slot_mapping int64 (each [num_tokens]) and, when
    max_num_work > 0, work_metadata int32 [max_num_work, 2].

    ``num_mapped_tokens`` is the host's copy of query_start_loc[-1]; when it
    is not given it is read from the device (one synchronising read).
    ``out`` may hold preallocated tensors under the same keys."""
    lib = load_library()
    _on_current_device(query_start_loc, seq_lens, block_table, common_slot_mapping,
                       *(out or {}).values())
    dev = query_start_loc.device
    num_reqs = query_start_loc.numel() - 1
    if query_start_loc.dim() != 1 or seq_lens.dim() != 1 or block_table.dim() != 2:
        raise QSAError(3, "query_start_loc and seq_lens 1-D, block_table 2-D expected")
    if not query_start_loc.is_contiguous() or not seq_lens.is_contiguous():
        raise QSAError(4, "query_start_loc and seq_lens must be contiguous")
    if seq_lens.numel() < num_reqs:
        raise QSAError(3, "seq_lens shorter than the request count")
    if num_mapped_tokens is None:
        num_mapped_tokens = int(query_start_loc[-1].item())
    out = dict(out or {})
    T = int(num_tokens)
    for key, dt in (("token_to_req", torch.int32), ("logical_positions", torch.int64),
                    ("visible_blocks", torch.int32), ("slot_mapping", torch.int64)):
        if key not in out:
            out[key] = torch.empty(T, dtype=dt, device=dev)
    if max_num_work and "work_metadata" not in out:
        out["work_metadata"] = torch.empty((max_num_work, 2), dtype=torch.int32, device=dev)
    work = out.get("work_metadata")
    for key in ("token_to_req", "logical_positions", "visible_blocks", "slot_mapping"):
        if out[key].numel() < T or not out[key].is_contiguous():
            raise QSAError(3, f"{key} must be a contiguous tensor of >= num_tokens entries")
    if work is not None and (not work.is_contiguous() or work.numel() < 2 * max_num_work):
        raise QSAError(3, "work_metadata must be contiguous [max_num_work, 2]")
    common = common_slot_mapping
    st = lib.qsa_build_metadata(
        _ptr(query_start_loc), _tag(query_start_loc), _ptr(seq_lens), _tag(seq_lens),
        _ptr(common), _tag(common) if common is not None else 0,
        _ptr(block_table), _tag(block_table), block_table.shape[0], block_table.shape[1],
        block_table.stride(0), block_table.stride(1),
        num_reqs, int(num_mapped_tokens), T,
        int(storage_block_size), int(compress_ratio), int(circular_buffer_size),
        _ptr(out["token_to_req"]), _ptr(out["logical_positions"]),
        _ptr(out["visible_blocks"]), _ptr(out["slot_mapping"]),
        _ptr(work) if max_num_work else None, int(max_num_work), _stream(stream))
    _check(st)
    return out


def qsa_paged_mqa_logits(q, kv_cache, weights, context_lens, block_tables, next_n: int,
                         max_model_len: int, *, block_size: int, out=None, error_word=None,
                         stream=None, library=None):
    """Weighted paged MQA indexer logits (include/qsa_indexer.h): returns fp32
    [rows, max_model_len].  q is E4M3 [rows, heads, 128]; kv_cache holds
    [num_blocks, block_size*132] bytes (uint8 or float8_e4m3fn storage).
    `library` as in qsa_select_paged_tokens."""
    lib = library or load_library()
    _on_current_device(q, kv_cache, weights, context_lens, block_tables, out, error_word)
    if q.dim() != 3 or kv_cache.dim() != 2 or weights.dim() != 2 or block_tables.dim() != 2:
        raise QSAError(3, "q [rows,H,128], kv_cache [blocks, bs*132], weights [rows,H], "
                          "block_tables 2-D expected")
    if not (q.is_contiguous() and kv_cache.is_contiguous() and weights.is_contiguous()
            and context_lens.is_contiguous()):
        raise QSAError(4, "q, kv_cache, weights and context_lens must be contiguous")
    if kv_cache.shape[1] != block_size * (IDX_HEAD_DIM + 4):
        raise QSAError(3, "kv_cache rows must hold block_size * 132 bytes")
    if block_tables.shape[1] > 1 and block_tables.stride(1) != 1:
        raise QSAError(4, "block-table columns must be contiguous")
    rows, heads = q.shape[0], q.shape[1]
    if out is None:
        out = torch.empty((rows, max_model_len), dtype=torch.float32, device=q.device)
    if out.dim() != 2 or (out.shape[1] > 1 and out.stride(1) != 1):
        raise QSAError(4, "logits must be 2-D with contiguous columns")
    kv_tag = DT_F8E4M3 if kv_cache.dtype in (torch.uint8, torch.float8_e4m3fn) else 0
    st = lib.qsa_paged_mqa_logits(
        _ptr(q), _tag(q), rows, heads,
        _ptr(kv_cache), kv_tag, kv_cache.shape[0], int(block_size),
        _ptr(weights), _tag(weights),
        _ptr(context_lens), _tag(context_lens), context_lens.numel(),
        _ptr(block_tables), _tag(block_tables), block_tables.shape[1], block_tables.stride(0),
        int(next_n),
        _ptr(out), _tag(out), int(max_model_len), out.stride(0),
        _ptr(error_word), _stream(stream))
    _check(st)
    return out


def qsa_top_k_per_row_decode(logits, next_n: int, seq_lens, topk_tokens: int, out=None,
                             stream=None):
    """Per-row top-k of the indexer logits (include/qsa_indexer.h): returns
    int32 [rows, topk_tokens], -1 padded."""
    lib = load_library()
    _on_current_device(logits, seq_lens, out)
    if logits.dim() != 2:
        raise QSAError(3, "logits must be 2-D")
    rows, cols = logits.shape
    if out is None:
        out = torch.empty((rows, topk_tokens), dtype=torch.int32, device=logits.device)
    if out.dim() != 2 or (out.shape[1] > 1 and out.stride(1) != 1):
        raise QSAError(4, "indices must be 2-D with contiguous columns")
    st = lib.qsa_top_k_per_row_decode(
        _ptr(logits), _tag(logits), rows, cols, logits.stride(0), logits.stride(1),
        int(next_n), _ptr(seq_lens), _tag(seq_lens), seq_lens.numel(),
        int(topk_tokens), _ptr(out), _tag(out), out.stride(0), _stream(stream))
    _check(st)
    return out
