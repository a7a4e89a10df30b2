"""Pins for the oracle's block_q8_matmul_nt (kopitiam-gpu block_q8_matmul_nt.wgsl), ternary
bitplane GEMV (BonsaiのWebGPUカーネルを読み解く, the P/N popcount identity), Q8_0 activation
quantizer (reading) and Bonsai-format prefill (reading)."""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads as wl
from tests.exact import f16_value, gamma, round_f32

GOLD = os.path.join(os.path.dirname(__file__), "golden", "block_q8_cases.json")
BQ_CASES = json.load(open(GOLD))["cases"]


def pack_quants(q_int8: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(q_int8.astype(np.int8)).view(np.uint8).reshape(-1, 4).copy().view(np.uint32).reshape(-1)


# ----------------------------------------------------------------------------- block_q8

@pytest.mark.parametrize("case", BQ_CASES, ids=[c["name"] for c in BQ_CASES])
def test_block_q8_golden(case):
    k = case["k"]
    x = np.zeros(k, dtype=np.float32)
    q = np.zeros(k, dtype=np.int8)
    for e, v in case["x"]:
        x[e] = v
    for e, v in case["q"]:
        q[e] = v
    scales = np.array(case["scales"], dtype=np.float32)
    y = oracle.block_q8_matmul_nt(x, pack_quants(q), scales, 1, k, 1)
    assert hex(int(y.view(np.uint32)[0, 0])) == case["expected_f32"], case["derivation"]


def test_block_q8_sign_extension_all_bytes():
    """Every byte value as quant element t (all four byte positions): y = sign-extended byte."""
    k, n = 32, 256
    for t in range(4):
        q = np.zeros((n, k), dtype=np.uint8)
        q[:, t] = np.arange(256, dtype=np.uint8)
        x = np.zeros(k, dtype=np.float32)
        x[t] = 1.0
        y = oracle.block_q8_matmul_nt(x, pack_quants(q.view(np.int8)), np.ones((n, 1), np.float32), 1, k, n)
        want = np.arange(256)
        want = np.where(want >= 128, want - 256, want).astype(np.float32)
        assert np.array_equal(y[0], want)


def test_block_q8_exact_special_case():
    """Integer x in [-8, 8] and power-of-two scales: every product and sum is exact, so the
    oracle equals the integer dot product scaled, bit for bit (pins indexing and layout)."""
    rng = np.random.default_rng(4)
    m, k, n = 3, 160, 17
    x = rng.integers(-8, 9, (m, k)).astype(np.float32)
    q = rng.integers(-128, 128, (n, k)).astype(np.int8)
    sc = (2.0 ** rng.integers(-3, 2, (n, k // 32))).astype(np.float32)
    y = oracle.block_q8_matmul_nt(x, pack_quants(q), sc, m, k, n)
    blocks = (x.astype(np.int64)[:, None, :] * q.astype(np.int64)[None, :, :]).reshape(m, n, k // 32, 32).sum(-1)
    want = (blocks * sc.astype(np.float64)[None]).sum(-1)
    assert np.array_equal(y.astype(np.float64), want)


def test_block_q8_f64_bound():
    rng = wl.Rng(55)
    m, k, n = 4, 960, 24
    x, quants, scales = wl.block_q8_inputs(rng, m, k, n)
    y = oracle.block_q8_matmul_nt(x, quants, scales, m, k, n).astype(np.float64)
    q = quants.view(np.int8).reshape(n, k).astype(np.float64)
    x64 = x.astype(np.float64)
    terms = x64[:, None, :] * q[None, :, :] * np.repeat(scales.astype(np.float64), 32, axis=1)[None]
    ref = terms.sum(-1)
    bound = gamma(32 + k // 32 + 2) * np.abs(terms).sum(-1)
    assert np.all(np.abs(y - ref) <= bound)


# ----------------------------------------------------------------------------- ternary

def brute_ternary(P, N, X, rows, k, batch):
    p = np.unpackbits(P.view(np.uint8), bitorder="little").reshape(rows, k).astype(np.int64)
    nn = np.unpackbits(N.view(np.uint8), bitorder="little").reshape(rows, k).astype(np.int64)
    x = np.unpackbits(X.view(np.uint8), bitorder="little").reshape(batch, k).astype(np.int64) * 2 - 1
    return (x @ (p - nn).T).astype(np.int32)


@pytest.mark.parametrize("p_zero", [0.4, 0.0, 1.0])
def test_ternary_identity_equals_direct_and_brute_force(p_zero):
    rows, k, batch = 37, 4096, 5
    P, N, X = wl.ternary_inputs(wl.Rng(7), rows, k, batch, p_zero=p_zero)
    a = oracle.ternary_direct(P, N, X, rows, k, batch)
    b = oracle.ternary_identity(P, N, X, rows, k, batch)
    c = brute_ternary(P, N, X, rows, k, batch)
    assert np.array_equal(a, c) and np.array_equal(b, c)


def test_ternary_overlapping_planes_are_zero():
    """P and N both set: w = P - N = 0, and the identity agrees."""
    rows, k = 3, 64
    P = np.full((rows, 2), 0xFFFFFFFF, dtype=np.uint32)
    X = np.array([[0x12345678, 0x9ABCDEF0]], dtype=np.uint32)
    assert np.all(oracle.ternary_identity(P, P, X, rows, k, 1) == 0)
    assert np.all(oracle.ternary_direct(P, P, X, rows, k, 1) == 0)


def test_ternary_all_plus_is_activation_sum():
    rows, k = 2, 96
    P = np.full((rows, 3), 0xFFFFFFFF, dtype=np.uint32)
    N = np.zeros_like(P)
    X = np.array([[0xF0F0F0F0, 0, 0xFFFFFFFF]], dtype=np.uint32)
    # 16 + 0 + 32 ones, 48 minus-ones: sum = 48 - 48 = 0; flip the middle word to all ones
    assert oracle.ternary_identity(P, N, X, rows, k, 1)[0, 0] == 0
    X[0, 1] = 0xFFFFFFFF
    assert oracle.ternary_identity(P, N, X, rows, k, 1)[0, 0] == 80 - 16


# ----------------------------------------------------------------------------- quantizer

def test_quantize_hand_cases():
    """amax = 127 makes d = 1 exactly: q is x rounded half up, stored d is f16 1.0."""
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, :8] = [127.0, 2.5, -2.5, 0.49999997, 126.5, -126.5, -0.5, 0.5]
    d, q = oracle.quantize_q8_0(x, 1, 32)
    assert d[0, 0] == 0x3C00
    assert q[0, :8].tolist() == [127, 3, -2, 0, 127, -126, 0, 1]
    assert np.all(q[0, 8:] == 0)


def test_quantize_zero_block():
    d, q = oracle.quantize_q8_0(np.zeros((2, 64), np.float32), 2, 64)
    assert np.all(d == 0) and np.all(q == 0)


def test_quantize_invariants():
    rng = wl.Rng(8)
    m, k = 16, 4096
    x = wl.f32_normal(rng, m * k).reshape(m, k)
    x[3, 64:96] *= 1e-30                     # tiny block (d rounds to an f16 subnormal or zero)
    d, q = oracle.quantize_q8_0(x, m, k)
    xb = x.reshape(m, k // 32, 32).astype(np.float64)
    amax = np.abs(xb).max(-1)
    d32 = (amax.astype(np.float32) / np.float32(127.0)).astype(np.float32)
    assert np.array_equal(d, d32.astype(np.float16).view(np.uint16))       # numpy RN-even
    qb = q.reshape(m, k // 32, 32).astype(np.int64)
    assert np.all(np.abs(qb) <= 127)
    nz = amax > 0
    assert np.all(np.abs(qb).max(-1)[nz] == 127)
    # reconstruction with the f32 d: |q*d - x| <= d/2 (plus the division's rounding)
    err = np.abs(qb * d32[..., None].astype(np.float64) - xb)
    assert np.all(err <= d32[..., None] * (0.5 + 1e-6) + 1e-45)



def _exact_quantize_block(xb):
    """The stated quantizer, in exact rationals: d = RN_f32(amax / 127); q = round half up of
    RN_f32(x / d), clamped to [-127, 127]; the stored scale is numpy's RN-even f16 of d."""
    amax = max(abs(Fraction(float(v))) for v in xb)
    if amax == 0:
        return 0, [0] * 32
    d = round_f32(amax / 127)
    qs = []
    for v in xb:
        vv = Fraction(round_f32(Fraction(float(v)) / Fraction(d)))
        fl = vv.numerator // vv.denominator
        qi = fl + (1 if vv - fl >= Fraction(1, 2) else 0)
        qs.append(max(-127, min(127, qi)))
    return int(np.array([d], np.float32).astype(np.float16).view(np.uint16)[0]), qs


def test_quantize_general_d_exact_rational():
    """q at a general scale d, against exact rational arithmetic.  Each block holds its amax and
    values a few ulps either side of (n + 1/2) * d, where the IEEE division x / d and the multiply
    by a reciprocal x * (1/d) round to different sides of the tie; at least some of those cases must
    tell the two apart, so a quantizer that multiplied by 1/d (or by 127/amax) fails here."""
    rng = np.random.default_rng(5)
    blocks, alt_differs = [], 0
    for _ in range(24):
        amax = np.float32(rng.uniform(0.3, 900.0))
        d = round_f32(Fraction(float(amax)) / 127)
        inv = round_f32(1 / Fraction(d))
        xb = [float(amax) * (1 if rng.random() < 0.5 else -1)]
        while len(xb) < 32:
            n = int(rng.integers(-126, 126))
            t = np.float32(round_f32((n + Fraction(1, 2)) * Fraction(d)))
            for ul in (-2, -1, 0, 1, 2):
                x = float(np.nextafter(t, np.float32(np.inf * ul), dtype=np.float32)) if ul else float(t)
                if abs(ul) == 2:
                    x = float(np.nextafter(np.float32(x), np.float32(np.inf * ul), dtype=np.float32))
                if len(xb) < 32 and abs(x) <= float(amax):
                    xb.append(x)
                    by_div = Fraction(round_f32(Fraction(x) / Fraction(d)))
                    by_mul = Fraction(round_f32(Fraction(x) * Fraction(inv)))
                    half_up = [v.numerator // v.denominator + (1 if v - v.numerator // v.denominator >= Fraction(1, 2)
                                                               else 0) for v in (by_div, by_mul)]
                    alt_differs += int(half_up[0] != half_up[1])
        blocks.append(xb)
    x = np.array(blocks, dtype=np.float32).reshape(1, -1)
    d, q = oracle.quantize_q8_0(x, 1, x.size)
    for b, xb in enumerate(blocks):
        dw, qw = _exact_quantize_block(np.array(xb, np.float32))
        assert d[0, b] == dw, b
        assert q[0, 32 * b:32 * b + 32].tolist() == qw, b
    assert alt_differs > 0

# ----------------------------------------------------------------------------- prefill (Q1_S32 x Q8_0)

def exact_prefill(signs, ws, xd, xq, M, N, K):
    nb = K // 32
    out = np.empty((M, N), dtype=object)
    bits = np.unpackbits(signs.view(np.uint8), bitorder="little").reshape(N, nb, 32)
    q = xq.astype(np.int64).reshape(M, nb, 32)
    wrapneg = np.where(q == -128, -128, -q)
    for m in range(M):
        S = np.where(bits[None, :, :, :].astype(bool), q[m][None], wrapneg[m][None]).sum(-1)[0]  # [N, nb]
        for n in range(N):
            out[m, n] = [Fraction(float(ws[n, b])) * f16_value(int(xd[m, b])) * int(S[n, b]) for b in range(nb)]
    return out


def test_prefill_exact_special_case():
    """Power-of-two weight and activation scales: p and every fma are exact."""
    rng = np.random.default_rng(12)
    M, N, K = 3, 9, 256
    signs = rng.integers(0, 2 ** 32, (N, K // 32), dtype=np.uint64).astype(np.uint32)
    ws = (2.0 ** rng.integers(-2, 2, (N, K // 32))).astype(np.float32)
    xd = (2.0 ** rng.integers(-2, 2, (M, K // 32))).astype(np.float16).view(np.uint16)
    xq = rng.integers(-128, 128, (M, K)).astype(np.int8)
    y = oracle.prefill_q1s32(signs, ws, xd, xq, M, N, K)
    terms = exact_prefill(signs, ws, xd, xq, M, N, K)
    for m in range(M):
        for n in range(N):
            assert Fraction(float(y[m, n])) == sum(terms[m, n], Fraction(0))


def test_prefill_bound_random():
    rng = wl.Rng(21)
    M, N, K = 4, 6, 1024
    signs, ws, x = wl.prefill_inputs(rng, M, K, N)
    xd, xq = oracle.quantize_q8_0(x, M, K)
    y = oracle.prefill_q1s32(signs, ws, xd, xq, M, N, K)
    terms = exact_prefill(signs, ws, xd, xq, M, N, K)
    g = gamma(K // 32 + 1)
    for m in range(M):
        for n in range(N):
            t = terms[m, n]
            ex = sum(t, Fraction(0))
            assert abs(float(Fraction(float(y[m, n])) - ex)) <= g * float(sum(abs(v) for v in t))


def test_prefill_single_rounding_and_wrap():
    """Hand case: block 0 gives acc = -508.9921875 exactly (w_s = -1, d_x = 1+2^-9, S = 508);
    block 1 has w_s = 1+2^-10, d_x = 1+2^-10, S = 508, so one correctly rounded fma leaves
    508*2^-20 (an unfused multiply would give 2^-11).  Block 2 holds four -128 quants with sign
    bit 0 (wrapping negate keeps -128) against d_x = 0: p = -0 and acc is unchanged."""
    K = 96
    signs = np.array([[0xFFFFFFFF, 0xFFFFFFFF, 0x0]], dtype=np.uint32)
    ws = np.array([[-1.0, 1.0 + 2 ** -10, 1.0]], dtype=np.float32)
    xd = np.array([[0x3C02, 0x3C01, 0x0000]], dtype=np.uint16)
    xq = np.zeros((1, K), dtype=np.int8)
    xq[0, 0:4] = 127
    xq[0, 32:36] = 127
    xq[0, 64:68] = -128
    y = oracle.prefill_q1s32(signs, ws, xd, xq, 1, 1, K)
    assert hex(int(y.view(np.uint32)[0, 0])) == "0x39fe0000"


# ----------------------------------------------------------------------------- Bonsai W1A32 decode
# [P3] decode/prefill figure, llama-decode-q1-proj.wgsl: weight = +1 (bit 1) or -1 (bit 0), one f32
# scale per 32 weights, f32 activations; the oracle is the f64 definition.

def _w1a32_exact(signs, ws, x, M, N, K):
    """Exact rational y[m][n] = sum_b ws * sum_t s * x (every f32 input is an exact rational)."""
    nbk = K // 32
    out = [[Fraction(0)] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for b in range(nbk):
                word = int(signs[n, b])
                d = Fraction(0)
                for t in range(32):
                    xv = Fraction(float(x[m, 32 * b + t]))
                    d += xv if (word >> t) & 1 else -xv
                acc += Fraction(float(ws[n, b])) * d
            out[m][n] = acc
    return out


def test_w1a32_within_f64_bound_of_exact():
    M, N, K = 2, 5, 96
    signs, ws, x = wl.prefill_inputs(wl.Rng(31), M, K, N)
    got = oracle.q1s32_f32_gemv(signs, ws, x, M, N, K)
    exact = _w1a32_exact(signs, ws, x, M, N, K)
    nbk = K // 32
    for m in range(M):
        for n in range(N):
            terms = sum(abs(float(ws[n, b])) * sum(abs(float(x[m, 32 * b + t])) for t in range(32)) for b in range(nbk))
            bound = (K + nbk + 2) * 2.0 ** -53 * terms
            assert abs(Fraction(float(got[m, n])) - exact[m][n]) <= Fraction(bound)


def test_w1a32_exact_special_case():
    """Integer activations in [-8, 8] and power-of-two scales: every partial sum is exact in f64 (and
    in f32), so the oracle equals the exact value bit for bit."""
    M, N, K = 3, 7, 160
    rng = wl.Rng(32)
    signs = rng.u32(N * K // 32).reshape(N, K // 32)
    ws = (2.0 ** -(2 + (rng.u32(N * K // 32) % 5).astype(np.int64))).astype(np.float32).reshape(N, K // 32)
    x = ((rng.u32(M * K) % 17).astype(np.int64) - 8).astype(np.float32).reshape(M, K)
    got = oracle.q1s32_f32_gemv(signs, ws, x, M, N, K)
    exact = _w1a32_exact(signs, ws, x, M, N, K)
    for m in range(M):
        for n in range(N):
            assert Fraction(float(got[m, n])) == exact[m][n]


def test_w1a32_sign_convention():
    """One block: all bits set gives +ws * sum(x), none gives -ws * sum(x), a single set bit t gives
    ws * (2 x_t - sum(x))."""
    K = 32
    x = np.arange(1, 33, dtype=np.float32).reshape(1, K)
    total = float(x.sum())
    ws = np.array([[0.5]], dtype=np.float32)
    for word, want in [(0xFFFFFFFF, 0.5 * total), (0x0, -0.5 * total), (1 << 5, 0.5 * (2 * 6.0 - total))]:
        got = oracle.q1s32_f32_gemv(np.array([[word]], dtype=np.uint32), ws, x, 1, 1, K)
        assert got[0, 0] == want
