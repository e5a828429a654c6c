"""Plain CPU oracle for the weighted paged MQA indexer and its per-row top-k
-- TEST INFRASTRUCTURE (same rules as the rest of ``oracle/``: only the
tests, the smoke check and the benchmark's CPU legs call it; it shares
nothing with the CUDA path).

What it restates.  "[XPU] Enable multiple key kernels for sparse attention"
(vllm-project/vllm PR 37888 report), "Implementation" and "Key source
snippets": the DeepSeek-V3.2 sparse-attention indexer's decode step is
``fp8_paged_mqa_logits(q, kv_cache, weights, context_lens, block_tables,
schedule_metadata, max_model_len)`` followed by ``top_k_per_row_decode(
logits, next_n, seq_lens, raw_topk_indices, num_rows, stride0, stride1,
topk_tokens)``; the removed Python fallback quantised the indexer keys per
group (``group_quant_torch``) into the cache.  The page prints signatures
only; what they compute is taken in the plainest way the rest supports
(each reading is listed with the design notes):

  * rows: r = b * next_n + j is query token j of request b; q is FP8 E4M3
    [rows, H, D]; weights fp32 [rows, H];
  * a cached key is D E4M3 values times one fp32 scale per token (the group
    quantisation, one group per key); a cache block of ``block_size`` tokens
    holds the tokens' D-byte value rows, then their 4-byte scales;
    token t of request b lives in block ``block_tables[b, t // block_size]``,
    slot ``t % block_size``;
  * logit(r, t) = scale_t * sum_h weights[r, h] * ReLU(q[r, h, :] . k_t)
    (the QSA selection score, sum_h ReLU(q_h . k), with per-head weights and
    the key's scale), for the tokens row r may see: t < L_r with
    L_r = context_lens[b] - next_n + j + 1 (speculative token j sees the
    context up to itself); -inf for every other column up to max_model_len;
  * top_k_per_row_decode keeps, per row, the topk_tokens largest logits among
    t < L_r (L_r from seq_lens the same way), largest first, equal logits by
    ascending token index, then -1 up to topk_tokens.

Arithmetic: E4M3 values are decoded exactly; each q_h . k_t is formed in
binary64, which is exact (products of two E4M3 values carry at most 8
significant bits between 2^-18 and 2^18, so a 128-term sum fits in 53 bits);
the head sum and scaling are binary64.  Pinned by tests/test_oracle_indexer.py.
"""
from __future__ import annotations

import numpy as np

import oracle

ERR_BLOCK = 2          # a block id negative / past the cache: its tokens get -inf


def _e4m3_table() -> np.ndarray:
    return np.array([oracle.e4m3_to_double(i) for i in range(256)], dtype=np.float64)


_TABLE = None


def e4m3_decode(codes) -> np.ndarray:
    """E4M3 codes (uint8 array) -> binary64 values, exactly."""
    global _TABLE
    if _TABLE is None:
        _TABLE = _e4m3_table()
    return _TABLE[np.asarray(codes, dtype=np.uint8)]


def split_block(block_bytes: np.ndarray, block_size: int, head_dim: int):
    """One cache block's bytes -> (values [block_size, D] uint8, scales
    [block_size] float32): the D-byte value rows of the block's tokens,
    then their 4-byte scales."""
    b = np.asarray(block_bytes, dtype=np.uint8).reshape(-1)
    vals = b[:block_size * head_dim].reshape(block_size, head_dim)
    scales = b[block_size * head_dim:block_size * (head_dim + 4)].view(np.float32)
    return vals, scales


def row_length(lens, r: int, next_n: int) -> int:
    """Columns row r = b*next_n + j may see: lens[b] - next_n + j + 1 (>= 0)."""
    b, j = divmod(r, next_n)
    return max(0, int(lens[b]) - next_n + j + 1)


def paged_mqa_logits(q, kv_cache, weights, context_lens, block_tables, next_n: int,
                     max_model_len: int, block_size: int, rows=None):
    """Logits [len(rows), max_model_len] binary64 and the OR of error bits.

    q        uint8 [R, H, D] E4M3 codes
    kv_cache uint8 [num_blocks, block_size * (D + 4)]
    weights  float32 [R, H]
    context_lens int [B], block_tables int [B, max_blocks]
    """
    q = np.asarray(q, dtype=np.uint8)
    R, H, D = q.shape
    kv = np.asarray(kv_cache, dtype=np.uint8)
    nblk = kv.shape[0]
    bt = np.asarray(block_tables)
    w = np.asarray(weights, dtype=np.float32).astype(np.float64)
    rows = list(range(R)) if rows is None else list(rows)
    out = np.full((len(rows), max_model_len), -np.inf, dtype=np.float64)
    err = 0
    for i, r in enumerate(rows):
        b = r // next_n
        L = min(row_length(context_lens, r, next_n), max_model_len)
        if L == 0:
            continue
        qv = e4m3_decode(q[r])                                  # [H, D]
        for c in range((L + block_size - 1) // block_size):
            t0 = c * block_size
            t1 = min(L, t0 + block_size)
            blk = int(bt[b, c]) if c < bt.shape[1] else -1
            if not (0 <= blk < nblk):
                err |= ERR_BLOCK
                continue
            vals, scales = split_block(kv[blk], block_size, D)
            k = e4m3_decode(vals[:t1 - t0])                      # [n, D]
            dots = k @ qv.T                                      # [n, H], exact
            relu = np.where(dots > 0, dots, 0.0)
            out[i, t0:t1] = scales[:t1 - t0].astype(np.float64) * (relu @ w[r])
    return out, err


def top_k_per_row(logits, next_n: int, seq_lens, topk: int, rows=None):
    """int32 [len(rows), topk]: per row the topk largest logits among the row's
    first L_r columns, largest first, ties by ascending column, then -1."""
    lg = np.asarray(logits)
    rows = list(range(lg.shape[0])) if rows is None else list(rows)
    out = np.full((len(rows), topk), -1, dtype=np.int32)
    for i, r in enumerate(rows):
        L = min(row_length(seq_lens, r, next_n), lg.shape[1])
        if L == 0:
            continue
        v = lg[r, :L]
        order = np.lexsort((np.arange(L), -v))                  # value desc, index asc
        keep = order[:topk]
        out[i, :len(keep)] = keep
    return out
