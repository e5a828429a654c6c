"""Plain CPU oracle for the QSA side-cache metadata builder -- TEST
INFRASTRUCTURE (same rules as the rest of ``oracle/``: only the tests, the
smoke check and the benchmark's CPU legs call it; the product library never
does, and this file shares nothing with the CUDA path).

What it restates: qsa_cache.py (vLLM fork, Qwen4Exp QSA side caches), the
per-forward metadata of one QSA side cache:
  * _build_qsa_metadata_kernel / _build_qsa_metadata_torch -- for every
    scheduled token: its request (the last request whose query starts at or
    before it), its logical position, its visible compressed blocks, and the
    slot it writes in the side cache; optionally the per-request work list of
    the pre-indexer (one item per completed compression group, at least one
    for a request with queries);
  * _logical_positions -- position = seq_len - query_len + offset in query;
  * circular_qsa_slot_mapping -- a request's single ring block, only the
    last ``circular_buffer_size`` tokens of its query write;
  * compressed_qsa_slot_mapping / _logical_to_physical_qsa_slots -- only
    the token that closes a compression group writes, at the group's paged
    slot; a missing page (negative id, or a column past the table) pads.

Steps are written one token (and one work item) at a time with plain Python
integers, in the order the page takes them.  Pinned by
``tests/test_oracle_metadata.py`` (brute-force counting definitions, closed
forms of plain decode, invariants that tie the slot map to the selection's
page lookup).

Readings (where the page's two versions, the Triton kernel and the torch
fallback, could differ, the Triton kernel -- the path that runs -- is taken):
  * a token at or past ``num_mapped_tokens`` is padding: request 0, position
    -1, no visible blocks, slot -1;
  * the compressed slot map also pads a token whose common slot is negative
    (both versions do this); the circular map does not look at it;
  * with ``compress_ratio == 1`` and no circular buffer the slot map is the
    common slot map itself (copied);
  * ``query_start_loc`` is non-decreasing from 0 (vLLM's invariant); the
    search then returns the last of several requests that start at the same
    token, i.e. never an empty one.
"""
from __future__ import annotations

from bisect import bisect_right

import numpy as np

PAD_SLOT_ID = -1


def _floordiv(a: int, b: int) -> int:
    return a // b      # Python floor division; every use has a >= 0 or b > 0


def token_request(qsl, num_reqs: int, t: int) -> int:
    """The last request i < num_reqs whose query starts at or before token t
    (0 when none does); qsl is a non-decreasing list, searched with the
    standard library's bisection."""
    return max(bisect_right(qsl, t, 0, num_reqs) - 1, 0)


def build_metadata(query_start_loc, seq_lens, block_table, num_tokens: int, *,
                   storage_block_size: int, compress_ratio: int,
                   circular_buffer_size: int = 0, common_slot_mapping=None,
                   num_mapped_tokens: int | None = None,
                   max_num_work: int | None = None) -> dict:
    """Metadata for ``num_tokens`` scheduled tokens of ``len(qsl) - 1``
    requests.  Returns numpy arrays: token_to_req int32, logical_positions
    int64, visible_blocks int32, slot_mapping int64 and, when max_num_work
    is given, work_metadata int32 [max_num_work, 2]."""
    qsl = [int(x) for x in np.asarray(query_start_loc).ravel()]
    sl = [int(x) for x in np.asarray(seq_lens).ravel()]
    bt = np.asarray(block_table)
    num_reqs = len(qsl) - 1
    if num_reqs < 1:
        raise ValueError("need at least one request")
    if storage_block_size <= 0 or compress_ratio <= 0 or circular_buffer_size < 0:
        raise ValueError("block size and compression ratio must be positive")
    n_mapped = qsl[-1] if num_mapped_tokens is None else int(num_mapped_tokens)
    cols = bt.shape[1] if bt.ndim == 2 else 0
    common = None if common_slot_mapping is None else \
        [int(x) for x in np.asarray(common_slot_mapping).ravel()]
    cr = compress_ratio

    t2r = np.zeros(num_tokens, np.int32)
    lpos = np.full(num_tokens, -1, np.int64)
    vis = np.zeros(num_tokens, np.int32)
    slots = np.full(num_tokens, PAD_SLOT_ID, np.int64)
    for t in range(num_tokens):
        mapped = t < n_mapped
        if mapped:
            req = token_request(qsl, num_reqs, t)
            q0, q1, L = qsl[req], qsl[req + 1], sl[req]
            lp = L - (q1 - q0) + (t - q0)
        else:
            req, q1, L, lp = 0, 0, 0, -1
        t2r[t] = req
        lpos[t] = lp
        vis[t] = max(0, min(_floordiv(lp + 1, cr), _floordiv(L, cr)))

        if circular_buffer_size > 0:
            # the request's one ring block, column 0; only the query's last
            # circular_buffer_size tokens write
            ok = mapped and lp >= 0 and t + circular_buffer_size >= q1 and cols > 0
            if ok:
                pb = int(bt[req, 0])
                if pb >= 0:
                    slots[t] = pb * circular_buffer_size + lp % circular_buffer_size
        elif cr != 1:
            # boundary token of a compression group writes the group's key
            g = _floordiv(max(lp, 0), cr)
            col = _floordiv(g, storage_block_size)
            ok = mapped and lp >= 0 and (lp + 1) % cr == 0 and col < cols
            if ok:
                pb = int(bt[req, col])
                c = common[t] if common is not None else -1
                if pb >= 0 and c >= 0:
                    slots[t] = pb * storage_block_size + g % storage_block_size
        else:
            if common is not None:
                slots[t] = common[t]

    out = {"token_to_req": t2r, "logical_positions": lpos,
           "visible_blocks": vis, "slot_mapping": slots}

    if max_num_work is not None:
        counts = []
        for i in range(num_reqs):
            ql = qsl[i + 1] - qsl[i]
            chunk_start = sl[i] - ql
            groups = _floordiv(sl[i], cr) - _floordiv(chunk_start, cr)
            counts.append(max(groups, 1) if ql > 0 else 0)
        work = np.full((max_num_work, 2), -1, np.int32)
        w = 0
        for i, n in enumerate(counts):
            for j in range(n):
                if w < max_num_work:
                    work[w] = (i, j)
                w += 1
        out["work_metadata"] = work
        out["work_total"] = w
    return out
