"""Pins for the oracle's Q1_0 . Q8_0 dot product (browseml-gpu.js: header comment, Q1_DOT_WGSL,
Q1_MM_WGSL, Q1_MM4_WGSL).

* hand-derived worked cases (tests/golden/q1_q8_cases.json) that isolate the wrapping negate,
  the LSB-first bit order, the sequential ab chain, the single rounding of the scale fma and the
  fixed final reduction;
* brute force: the exact rational value of the dot product (integer lane sums from the
  definition, f16 scales decoded by numpy) bounds the oracle's error on random inputs;
* an exact special case (power-of-two scales, where no step rounds) must agree bit for bit;
* the matrix form equals the per-column dot product.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads as wl
from tests.exact import f16_value, gamma

GOLD = os.path.join(os.path.dirname(__file__), "golden", "q1_q8_cases.json")


def build_case(case):
    n = case["n"]
    nb, na = n // 128, n // 32
    w = np.zeros((nb, 18), dtype=np.uint8)
    a = np.zeros((na, 34), dtype=np.uint8)
    for i, h in enumerate(case["d0"]):
        v = int(h, 16)
        w[i, 0], w[i, 1] = v & 0xFF, v >> 8
    for j, h in enumerate(case["d1"]):
        v = int(h, 16)
        a[j, 0], a[j, 1] = v & 0xFF, v >> 8
    for blk, e, val in case["q"]:
        a[blk, 2 + e] = np.uint8(val & 0xFF)
    for blk, off, val in case["bits"]:
        w[blk, 2 + off] = val
    return w.reshape(-1), a.reshape(-1), n


CASES = json.load(open(GOLD))["cases"]


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_golden_cases(case):
    w, a, n = build_case(case)
    y = oracle.q1_q8_gemv(w, a, 1, n)
    assert hex(int(y.view(np.uint32)[0])) == case["expected_f32"], case["derivation"]


def exact_lane_terms(w_row: np.ndarray, act: np.ndarray, n: int):
    """All terms d0_i * d1_{4i+k} * s_{i,k,l} as exact rationals, s from the definition:
    bit 1 -> +q, bit 0 -> the int8 wrapping negate of q."""
    terms = []
    for i in range(n // 128):
        blk = w_row[i * 18:(i + 1) * 18]
        d0 = f16_value(int(blk[0]) | (int(blk[1]) << 8))
        bits = np.unpackbits(blk[2:], bitorder="little")           # 128 bits, k-major
        for k in range(4):
            ab = act[(4 * i + k) * 34:(4 * i + k + 1) * 34]
            d1 = f16_value(int(ab[0]) | (int(ab[1]) << 8))
            q = ab[2:].view(np.int8).astype(np.int64)
            for l in range(8):
                s = 0
                for e in range(4 * l, 4 * l + 4):
                    qe = int(q[e])
                    neg = -128 if qe == -128 else -qe
                    s += qe if bits[32 * k + e] else neg
                terms.append(d0 * d1 * s)
    return terms


@pytest.mark.parametrize("dist", ["uniform", "page"])
def test_exact_bound_random(dist):
    rows, n = 12, 1024
    rng = wl.Rng(101 if dist == "uniform" else 202)
    w = wl.q1_0_weights(rng, rows, n, scales=dist)
    a = wl.q8_0_acts(rng, 1, n, scales=dist, quants=dist)
    y = oracle.q1_q8_gemv(w, a, rows, n)
    rb = (n // 128) * 18
    g = gamma(n // 128 + 3 + 3)
    for r in range(rows):
        terms = exact_lane_terms(w[r * rb:(r + 1) * rb], a, n)
        exact = sum(terms, Fraction(0))
        bound = g * float(sum(abs(t) for t in terms))
        assert abs(float(Fraction(float(y[r])) - exact)) <= bound, (r, float(exact), y[r], bound)
        # the bound is tight enough to catch one dropped or sign-flipped term
        assert bound < 0.05 * float(max(abs(t) for t in terms))


def pow2_case(rows, n, seed, lo=-2, hi=1):
    """Scales +-2^e with e in [lo, hi]: every product, ab sum, fma and reduction is exact."""
    rng = np.random.default_rng(seed)
    nb, na = n // 128, n // 32

    def f16_pow2(count):
        e = rng.integers(lo, hi + 1, count)
        s = np.where(rng.uniform(0, 1, count) < 0.5, -1.0, 1.0)
        return (s * 2.0 ** e).astype(np.float16).view(np.uint16)

    w = np.zeros((rows * nb, 18), dtype=np.uint8)
    w[:, 0:2] = f16_pow2(rows * nb).view(np.uint8).reshape(-1, 2)
    w[:, 2:] = rng.integers(0, 256, (rows * nb, 16))
    a = np.zeros((na, 34), dtype=np.uint8)
    a[:, 0:2] = f16_pow2(na).view(np.uint8).reshape(-1, 2)
    q = rng.integers(-128, 128, (na, 32)).astype(np.int8)
    a[:, 2:] = q.view(np.uint8)
    return w.reshape(-1), a.reshape(-1)


def test_exact_special_case_bit_for_bit():
    rows, n = 24, 1024
    w, a = pow2_case(rows, n, 5)
    y = oracle.q1_q8_gemv(w, a, rows, n)
    rb = (n // 128) * 18
    for r in range(rows):
        exact = sum(exact_lane_terms(w[r * rb:(r + 1) * rb], a, n), Fraction(0))
        assert Fraction(float(y[r])) == exact, r


def test_lanes_match_exact_per_lane():
    """The eight lane accumulators, before the final reduction, each equal their exact lane sum
    in the exact special case (pins lane = elements 4l..4l+3)."""
    n = 512
    w, a = pow2_case(1, n, 9)
    _, lanes = oracle.q1_q8_row(w, a, n)
    terms = exact_lane_terms(w, a, n)          # ordered (i, k, l)
    for l in range(8):
        lane_exact = sum((terms[j] for j in range(len(terms)) if j % 8 == l), Fraction(0))
        assert Fraction(float(lanes[l])) == lane_exact, l


def test_gemm_columns_equal_gemv():
    rows, n, cols = 40, 768, 5
    rng = wl.Rng(33)
    w = wl.q1_0_weights(rng, rows, n)
    a = wl.q8_0_acts(rng, cols, n, quants="page")
    Y = oracle.q1_q8_gemm(w, a, rows, n, cols)
    ab = (n // 32) * 34
    for c in range(cols):
        yc = oracle.q1_q8_gemv(w, a[c * ab:(c + 1) * ab], rows, n)
        assert np.array_equal(Y[c].view(np.uint32), yc.view(np.uint32))
