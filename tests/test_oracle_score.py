"""Pins for the oracle's fp16 decoding and canonical selection score.

The score is "four-head ReLU(Q*K) scores" ("vLLM: integrate FP16 packed QSA
extension", Summary bullet 3).  The pages fix no precision or order; the
oracle evaluates binary32 in one stated order.  Pinned here by:
  * fp16 decoding: every one of the 65536 bit patterns against numpy's
    float16 -> float64 conversion (a library routine);
  * exact-sum inputs (small integers and dyadic fractions whose every partial
    sum is exact): any order gives the exact value, so the score must equal
    sum_h max(0, exact dot) computed with Python integers/fractions -- a
    dropped term, a wrong dim or head index, a wrong sign or a missing ReLU
    fails;
  * hand-derived rounding cases (tests/golden/score_rounding_cases.json) that
    make the stated summation order observable;
  * the error bound of the stated summation tree against the exact dot
    products on random inputs of the workloads' distributions.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle


def test_half_decode_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits], dtype=np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros decode with their sign
    assert math.copysign(1.0, oracle.half_to_double(0x8000)) == -1.0


def _exact_score(q, k):
    """sum over heads of max(0, exact dot) with exact rational arithmetic."""
    tot = Fraction(0)
    for h in range(4):
        d = sum(Fraction(float(q[h, i])) * Fraction(float(k[i])) for i in range(128))
        tot += max(d, Fraction(0))
    return tot


@pytest.mark.parametrize("seed", range(40))
def test_score_exact_on_exactly_summable_inputs(seed):
    rng = np.random.default_rng(seed)
    if seed % 2 == 0:
        q = rng.integers(-3, 4, size=(4, 128)).astype(np.float16)
        k = rng.integers(-4, 5, size=128).astype(np.float16)
    else:   # dyadic fractions: multiples of 1/8 and 1/16, still exact in binary32
        q = (rng.integers(-24, 25, size=(4, 128)) / 8.0).astype(np.float16)
        k = (rng.integers(-40, 41, size=128) / 16.0).astype(np.float16)
    # sparsify some heads so ReLU clipping and zero heads both occur
    q[rng.integers(0, 4)] *= -1
    if seed % 5 == 0:
        q[rng.integers(0, 4)] = 0
    s = oracle.score(q, k)
    assert Fraction(float(s)) == _exact_score(q, k)


def test_score_single_term_each_dim_and_head():
    # one nonzero product at every (head, dim): catches any index mix-up
    for h in range(4):
        for i in range(128):
            q = np.zeros((4, 128), np.float16)
            k = np.zeros(128, np.float16)
            q[h, i] = 3.0
            k[i] = 5.0
            k[(i + 1) % 128] = 7.0       # a term no head should pick up here
            assert float(oracle.score(q, k)) == 15.0, (h, i)
            q[h, i] = -3.0
            s = oracle.score(q, k)
            assert float(s) == 0.0 and not math.copysign(1.0, float(s)) < 0, (h, i)


def test_score_golden_rounding_cases(golden_dir):
    d = json.load(open(os.path.join(golden_dir, "score_rounding_cases.json")))
    for case in d["cases"]:
        q = np.zeros((4, 128), np.float16)
        k = np.zeros(128, np.float16)
        seen = {}
        for h, dim, qv, kv in case["terms"]:
            assert seen.get(dim, kv) == kv, "fixture reuses a dim with another key value"
            seen[dim] = kv
            q[h, dim] = qv
            k[dim] = kv
        s = oracle.score(q, k)
        assert float(s) == case["expected"], case["name"]
        assert np.float32(s).view(np.uint32) == np.float32(case["expected"]).view(np.uint32)


def _gamma(n):
    u = 2.0 ** -24
    return n * u / (1 - n * u)


@pytest.mark.parametrize("seed", range(6))
def test_score_error_bound_vs_exact(seed):
    """|s - sum_h max(0, exact_h)| <= gamma_21 * sum_h sum_d |q k|: a term is
    rounded at most 16 (chain) + 1 (E+O) + 2 (slice tree) + 2 (head sum)
    times.  ReLU is 1-Lipschitz, so the bound carries through it."""
    rng = np.random.default_rng(100 + seed)
    g = _gamma(21)
    for _ in range(50):
        q = rng.standard_normal((4, 128)).astype(np.float16)
        k = (rng.standard_normal(128) * 0.1).astype(np.float16)
        s = float(oracle.score(q, k))
        prods = q.astype(np.float64) * k.astype(np.float64)[None, :]   # exact
        exact = sum(max(0.0, math.fsum(prods[h])) for h in range(4))
        bound = g * float(np.abs(prods).sum()) + 1e-300
        assert abs(s - exact) <= bound, (s, exact, bound)
    assert s >= 0.0
