"""The algorithmic byte counts behind the roofline's numerator (bench.py):
what one decode row must move, counted by hand for the pages' shapes --
selection: 256 B per visible key, the query, the page-table entries, the
2051-entry index write and the row metadata; attention: 1 KiB per distinct
valid token, the query and output, the index read, the K/V page-table
entries touched and the request id ("vLLM: integrate FP16 packed QSA
extension", Exact contracts)."""
import numpy as np

import bench


def test_select_bytes_long_context_row():
    # 131072 tokens, decode position 131071: 32768 visible blocks on 256 pages
    assert bench.select_bytes_per_row(131072, 131071) == (
        256 * 32768 + 4 * 128 * 2 + 4 * 256 + 4 * 2051 + 16)
    assert bench.select_bytes_per_row(131072, 131071) == 8_398_876


def test_select_bytes_short_rows():
    # 519 tokens: 129 visible blocks on 2 pages (the pages' first worked case)
    assert bench.select_bytes_per_row(519, 518) == 256 * 129 + 1024 + 4 * 2 + 8204 + 16
    # fewer than 4 tokens: no visible block, only the fixed traffic
    assert bench.select_bytes_per_row(3, 2) == 1024 + 8204 + 16
    # a position before the end of the sequence sees only its own blocks
    assert bench.select_bytes_per_row(10_000, 1023) == 256 * 256 + 1024 + 4 * 2 + 8204 + 16


def test_select_bytes_e4m3_keys_half_the_key_bytes():
    for L in (519, 9215, 131072):
        full = bench.select_bytes_per_row(L, L - 1)
        fp8 = bench.select_bytes_per_row_fp8(L, L - 1)
        V = L // 4
        assert full - fp8 == 128 * V


def test_attend_bytes_count_distinct_valid_tokens_once():
    row = np.array([5, 5, -1, 600, 1023, -1], dtype=np.int32)   # a duplicate and two holes
    # tokens {5, 600, 1023} on pages {0, 1}
    assert bench.attend_bytes_per_row(row) == 1024 * 3 + 3072 + 4 * 6 + 4 * 2 + 4


def test_attend_bytes_saturated_row():
    # 512 blocks x 4 tokens spread over 256 pages, then 3 holes: 2048 tokens
    rng = np.random.default_rng(0)
    pages = rng.permutation(256)
    slots = np.stack([rng.choice(128, size=2, replace=False) for _ in range(256)])
    blocks = (pages[:, None] * 128 + slots).ravel()           # two blocks on every page
    toks = (blocks[:, None] * 4 + np.arange(4)).ravel()
    row = np.concatenate([toks, [-1, -1, -1]]).astype(np.int32)
    assert row.size == 2051
    assert bench.attend_bytes_per_row(row) == 1024 * 2048 + 3072 + 8204 + 4 * 256 + 4
    assert bench.attend_bytes_per_row(row) == 2_109_456
