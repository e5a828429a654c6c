"""Pins for the oracle's FP8-E4M3 compressed-key selection.

qsa_cache.py's QSAStateBackend lists "fp8"/"fp8_e4m3" cache dtypes for "the
optional e4m3 compressed indexer cache".  The keys are then E4M3 values; the
score keeps the canonical binary32 definition and order over the decoded key
values (every E4M3 value is exact in fp16 and binary32, so q*k stays exact).

Independent checks:
  * decoding: all 256 codes against torch.float8_e4m3fn -> float64 (a library
    routine);
  * exact-sum inputs (small integers / dyadics representable in E4M3) against
    rational arithmetic;
  * the E4M3 path equals the fp16 path on the same key values (both decode
    to the same numbers before the fixed-order sum);
  * brute-force ranking on small rows with E4M3 pools, including heavy ties.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from sparse_paged_attention_qsa_gb300 import workloads as W


def _bytes(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.uint8).numpy()


def test_e4m3_decode_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert nan.sum() == 2                         # S.1111.111 only
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.nanmax(got) == 448.0 and oracle.e4m3_to_double(0x01) == 2.0 ** -9


@pytest.mark.parametrize("seed", range(12))
def test_e4m3_score_exact_on_exactly_summable_inputs(seed):
    rng = np.random.default_rng(200 + seed)
    q = rng.integers(-3, 4, size=(4, 128)).astype(np.float16)
    kv = rng.integers(-8, 9, size=128).astype(np.float32) / (1 if seed % 2 == 0 else 8)
    k8 = torch.from_numpy(kv).to(torch.float8_e4m3fn)
    assert torch.equal(k8.to(torch.float32), torch.from_numpy(kv))   # exactly representable
    exact = sum(max(Fraction(0), sum(Fraction(float(q[h, i])) * Fraction(float(kv[i]))
                                     for i in range(128))) for h in range(4))
    assert Fraction(float(oracle.score_e4m3(q, _bytes(k8)))) == exact


def test_e4m3_score_equals_fp16_score_on_same_values():
    rng = np.random.default_rng(7)
    for _ in range(200):
        q = rng.standard_normal((4, 128)).astype(np.float16)
        k8 = torch.from_numpy((rng.standard_normal(128) * 0.1).astype(np.float32)).to(
            torch.float8_e4m3fn)
        k16 = k8.to(torch.float16).numpy()
        a = oracle.score_e4m3(q, _bytes(k8))
        b = oracle.score(q, k16)
        assert np.float32(a).view(np.uint32) == np.float32(b).view(np.uint32)


def _brute_e4m3(w, r):
    q = w.q_sel[r].numpy()
    req = int(w.token_to_request[r])
    L, pos = int(w.seq_lens[req]), int(w.query_positions[r])
    last = min(pos, L - 1)
    V = sum(1 for g in range(L // 4 + 1) if 4 * g + 3 <= last)
    pt = w.cmp_page_table.numpy()
    pool = _bytes(w.cmp_cache)
    sc = {b: float(oracle.score_e4m3(q, pool[int(pt[req, b // 128]), b % 128, 0]))
          for b in range(V)}
    rank = {b: sum(1 for c in sc if sc[c] > sc[b] or (sc[c] == sc[b] and c < b)) for b in sc}
    order = sorted((rk, b) for b, rk in rank.items() if rk < 512)
    toks = [4 * b + i for _, b in order for i in range(4)] + list(range(4 * V, last + 1))
    return toks + [-1] * (2051 - len(toks))


@pytest.mark.parametrize("distinct", [0, 3])
def test_e4m3_select_matches_brute_force(distinct):
    w = W.build("fp8", [2803, 519, 130, 7], cmp_dtype="fp8", distinct_keys=distinct,
                seed=30 + distinct)
    out, err = oracle.select(w.q_sel.numpy(), _bytes(w.cmp_cache), w.cmp_page_table.numpy(),
                             w.token_to_request.numpy(), w.seq_lens.numpy(),
                             w.query_positions.numpy())
    assert err == 0
    for r in range(w.R):
        assert out[r].tolist() == _brute_e4m3(w, r), r
