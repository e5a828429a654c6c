"""Shared test helpers: run the oracle on a workload's tensors (copied to the
host) and run the CUDA path through the binding.  The oracle receives only the
pages the checked rows reference, so full-size pools never leave the GPU."""
import os

import numpy as np
import torch

import oracle

# oracle threads for full-size checks: one per usable host core
CORES = max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
            else (os.cpu_count() or 1))


def stream_edge_rows(R: int, width: int, sms: int, ctas_per_sm: int = 2):
    """Rows of a batch of more than 32 rows whose index list starts or ends
    exactly at a boundary between two CTA runs of the attention's stream
    split (32-entry chunks laid end to end, cut into G equal runs, G = the
    CTAs of one wave: ctas_per_sm per SM), plus the rows on either side."""
    C = max(1, -(-width // 32))
    T = R * C
    lmin = max(-(-(C - 1) // 8), 8)
    G = max(1, min(sms * ctas_per_sm, T // lmin))
    rows = set()
    for b in range(G + 1):
        x = T * b // G
        if x % C == 0:
            r = x // C
            rows.update(v for v in (r - 1, r) if 0 <= v < R)
    return sorted(rows)


def _pool(cache: torch.Tensor, page_ids, page_halves: int) -> "oracle.PagePool":
    P = cache.shape[0]
    kind = oracle.KEY_E4M3 if cache.dtype == torch.float8_e4m3fn else oracle.KEY_F16
    ids = sorted({int(p) for p in page_ids if 0 <= int(p) < P})
    if not ids:
        return oracle.PagePool({}, num_pages=P, kind=kind)
    sel = torch.tensor(ids, dtype=torch.long, device=cache.device)
    pages = cache.index_select(0, sel)
    if kind == oracle.KEY_E4M3:
        pages = pages.view(torch.uint8)
    host = pages.cpu().numpy().reshape(len(ids), -1)
    return oracle.PagePool({p: host[i] for i, p in enumerate(ids)}, num_pages=P,
                           page_halves=page_halves, kind=kind)


def _req_pages(pt: np.ndarray, t2r: np.ndarray, rows):
    reqs = sorted({int(t2r[r]) for r in rows if 0 <= int(t2r[r]) < pt.shape[0]})
    return pt[reqs].ravel() if reqs else np.zeros(0, np.int32)


def oracle_select(w, rows=None, threads=8, cmp_page_table=None, token_to_request=None):
    rows = list(range(w.R)) if rows is None else list(rows)
    pt = (cmp_page_table if cmp_page_table is not None else w.cmp_page_table).cpu().numpy()
    t2r = (token_to_request if token_to_request is not None else w.token_to_request).cpu().numpy()
    pool = _pool(w.cmp_cache, _req_pages(pt, t2r, rows), 128 * 128)
    q = w.q_sel.cpu().numpy()[rows]
    return oracle.select(q, pool, pt, t2r[rows], w.seq_lens.cpu().numpy(),
                         w.query_positions.cpu().numpy()[rows], threads=threads)


def oracle_attention(w, indices, rows=None, threads=8, kv_page_table=None,
                     token_to_request=None, scale=1.0 / 16.0):
    rows = list(range(w.R)) if rows is None else list(rows)
    pt = (kv_page_table if kv_page_table is not None else w.kv_page_table).cpu().numpy()
    t2r = (token_to_request if token_to_request is not None else w.token_to_request).cpu().numpy()
    idx = indices.cpu().numpy() if isinstance(indices, torch.Tensor) else np.asarray(indices)
    idx = idx[rows]
    # only pages holding a listed token are needed
    need = set()
    for i, r in enumerate(rows):
        req = int(t2r[r])
        if not (0 <= req < pt.shape[0]):
            continue
        cols = np.unique(idx[i][idx[i] >= 0] // 512)
        cols = cols[cols < pt.shape[1]]
        need.update(int(x) for x in pt[req, cols])
    pool = _pool(w.kv_cache, need, 512 * 512)
    return oracle.attention(w.q_attn.cpu().numpy()[rows], pool, pt, t2r[rows], idx,
                            scale=scale, threads=threads)
