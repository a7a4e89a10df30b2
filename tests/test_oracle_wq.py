"""Pins for the oracle's W8A32 and W4A32 group-128 matvec/matmul (web-xpu-ops README: the op
table rows matvecQ8 / matvecQ4G128 / matmulQ8 / matmulQ4G128 and "The q4 format").  Each pin is
chosen so that a plausible mistake fails it: byte or nibble order, sign extension, the -8 nibble,
the group index, per-row versus per-group scaling, a dropped tail."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads as wl


def _identity_x(K):
    return np.eye(K, dtype=np.float32)


def test_w8_byte_order_and_sign():
    """Codes are the word's bytes least-significant first, read as signed bytes."""
    w = np.array([[0x80FF017F]], dtype=np.uint32)
    y = oracle.w8a32(w, np.array([1.0], np.float32), _identity_x(4), 4, 1, 4)
    assert y[:, 0].tolist() == [127.0, 1.0, -1.0, -128.0]


def test_w8_matches_little_endian_byte_view():
    """numpy's int8 view of the little-endian words is the code matrix: the oracle equals
    scale * (codes @ x) in float64 on integer-valued x (exact)."""
    T, N, K = 3, 5, 64
    w, scale, _ = wl.wq_inputs(wl.Rng(1), T, K, N, 8)
    x = ((wl.Rng(2).u32(T * K) % 9).astype(np.int64) - 4).astype(np.float32).reshape(T, K)
    codes = w.view("<u4").view(np.int8).reshape(N, -1)[:, :K].astype(np.float64)
    want = (x.astype(np.float64) @ codes.T) * scale.astype(np.float64)[None, :]
    assert np.array_equal(oracle.w8a32(w, scale, x, T, N, K), want)


def test_w8_padding_is_ignored():
    """K = 5: the second word holds one code; its other bytes must not be read."""
    w = np.array([[0x04030201, 0x7F7F7F05]], dtype=np.uint32)
    y = oracle.w8a32(w, np.array([2.0], np.float32), np.ones((1, 5), np.float32), 1, 1, 5)
    assert y[0, 0] == 2.0 * (1 + 2 + 3 + 4 + 5)


def test_w4_nibble_order_and_twos_complement():
    """Codes are the word's nibbles least-significant first, 4-bit two's complement (0x8 = -8)."""
    for word, codes in [(0x87654321, [1, 2, 3, 4, 5, 6, 7, -8]), (0xFEDCBA98, [-8, -7, -6, -5, -4, -3, -2, -1])]:
        w = np.array([[word]], dtype=np.uint32)
        y = oracle.w4a32g128(w, np.array([[1.0]], np.float32), _identity_x(8), 8, 1, 8)
        assert y[:, 0].tolist() == [float(c) for c in codes]


@pytest.mark.parametrize("K", [256, 160])
def test_w4_group_scales(K):
    """Each scale multiplies its own 128 columns (the last group may be short); x = 1."""
    G = (K + 127) // 128
    w, _, _ = wl.wq_inputs(wl.Rng(K), 1, K, 1, 4)
    nibs = [((int(w[0, k // 8]) >> (4 * (k % 8))) & 0xF) for k in range(K)]
    codes = [v - 16 if v >= 8 else v for v in nibs]
    scale = np.array([[0.5, 0.25, 0.125][:G]], dtype=np.float32)
    want = sum(float(scale[0, g]) * sum(codes[128 * g:min(K, 128 * g + 128)]) for g in range(G))
    y = oracle.w4a32g128(w, scale, np.ones((1, K), np.float32), 1, 1, K)
    assert y[0, 0] == want


def _exact(codes_fn, scale_fn, G, x, T, N, K):
    out = [[Fraction(0)] * N for _ in range(T)]
    for t in range(T):
        for n in range(N):
            acc = Fraction(0)
            for g in range(G):
                lo, hi = (0, K) if G == 1 else (128 * g, min(K, 128 * g + 128))
                dot = sum(Fraction(codes_fn(n, k)) * Fraction(float(x[t, k])) for k in range(lo, hi))
                acc += Fraction(float(scale_fn(n, g))) * dot
            out[t][n] = acc
    return out


@pytest.mark.parametrize("bits", [8, 4])
def test_within_f64_bound_of_exact(bits):
    """Random inputs: the oracle lies within (K + G + 2) * 2^-53 * sum |terms| of the exact
    rational result (every f32 input is an exact rational)."""
    T, N, K = 2, 3, 300
    w, scale, x = wl.wq_inputs(wl.Rng(40 + bits), T, K, N, bits, p_m8=0.05)
    if bits == 8:
        codes = lambda n, k: int(np.int8(np.uint8((int(w[n, k // 4]) >> (8 * (k % 4))) & 0xFF)))
        sc = lambda n, g: scale[n]
        G, got = 1, oracle.w8a32(w, scale, x, T, N, K)
    else:
        codes = lambda n, k: (lambda v: v - 16 if v >= 8 else v)((int(w[n, k // 8]) >> (4 * (k % 8))) & 0xF)
        sc = lambda n, g: scale[n, g]
        G, got = (K + 127) // 128, oracle.w4a32g128(w, scale, x, T, N, K)
    exact = _exact(codes, sc, G, x, T, N, K)
    for t in range(T):
        for n in range(N):
            terms = sum(abs(float(sc(n, 0 if G == 1 else k // 128))) * abs(codes(n, k)) * abs(float(x[t, k]))
                        for k in range(K))
            assert abs(Fraction(float(got[t, n])) - exact[t][n]) <= Fraction((K + G + 2) * 2.0 ** -53 * terms)


@pytest.mark.parametrize("bits", [8, 4])
def test_exact_special_case(bits):
    """Integer x in [-8, 8] and power-of-two scales: every partial sum is exact, so the oracle
    equals the exact value."""
    T, N, K = 2, 4, 384
    rng = wl.Rng(50 + bits)
    w, scale, _ = wl.wq_inputs(rng, T, K, N, bits, p_m8=0.05)
    scale = (2.0 ** -(1 + (rng.u32(scale.size) % 6).astype(np.int64))).astype(np.float32).reshape(scale.shape)
    x = ((rng.u32(T * K) % 17).astype(np.int64) - 8).astype(np.float32).reshape(T, K)
    if bits == 8:
        got = oracle.w8a32(w, scale, x, T, N, K)
        codes = w.view("<u4").view(np.int8).reshape(N, -1)[:, :K].astype(np.int64)
        want = (x.astype(np.int64) @ codes.T) * scale.astype(np.float64)[None, :]
    else:
        got = oracle.w4a32g128(w, scale, x, T, N, K)
        nib = ((w[:, :, None] >> (4 * np.arange(8, dtype=np.uint32))[None, None, :]) & 0xF).reshape(N, -1)[:, :K]
        codes = nib.astype(np.int64) - 16 * (nib >= 8)
        want = np.zeros((T, N))
        for g in range(K // 128):
            sl = slice(128 * g, 128 * g + 128)
            want += (x[:, sl].astype(np.int64) @ codes[:, sl].T) * scale[:, g].astype(np.float64)[None, :]
    assert np.array_equal(got, want)
