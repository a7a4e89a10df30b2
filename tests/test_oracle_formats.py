"""Pins for the oracle's scalar formats: f16 decode, f32->f16 rounding, and the page's emulated
fma (browseml-gpu.js fn f16 and fn fma_exact), each against an independent library or an exact
rational computation."""
import ctypes
import ctypes.util
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests.exact import f32_bits, round_f32


def test_f16_decode_exhaustive_vs_numpy():
    h = np.arange(65536, dtype=np.uint16)
    got = oracle.f16_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    # NaN payload kept by the integer decode (m << 13), quiet or not
    m = (h[nan].astype(np.uint32) & 0x3FF) << 13
    assert np.array_equal(got[nan].view(np.uint32) & 0x7FFFFF, m)


@pytest.mark.parametrize("bits,value", [
    (0x0001, 2.0 ** -24), (0x03FF, 1023 * 2.0 ** -24), (0x8001, -(2.0 ** -24)),
    (0x0400, 2.0 ** -14), (0x3C00, 1.0), (0x7BFF, 65504.0), (0xFBFF, -65504.0),
    (0x0200, 2.0 ** -15), (0x7C00, float("inf")), (0xFC00, float("-inf")),
])
def test_f16_decode_closed_forms(bits, value):
    got = oracle.f16_to_f32(np.array([bits], dtype=np.uint16))[0]
    assert got == np.float32(value)


def test_f16_decode_signed_zero():
    got = oracle.f16_to_f32(np.array([0x0000, 0x8000], dtype=np.uint16))
    assert got.view(np.uint32).tolist() == [0x00000000, 0x80000000]


def _check_f32_to_f16(u: np.ndarray):
    f = u.view(np.float32)
    got = oracle.f32_to_f16(f)
    with np.errstate(over="ignore", invalid="ignore"):
        ref = f.astype(np.float16).view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all((got[nan] & 0x7C00) == 0x7C00) and np.all((got[nan] & 0x3FF) != 0)


@pytest.mark.skipif(not os.environ.get("GQ_SLOW"), reason="full 2^32 sweep (~9 min); set GQ_SLOW=1")
def test_f32_to_f16_exhaustive_vs_numpy():
    """Every one of the 2^32 binary32 patterns against numpy's RN-even conversion."""
    chunk = 1 << 24
    for start in range(0, 1 << 32, chunk):
        _check_f32_to_f16(np.arange(start, start + chunk, dtype=np.uint64).astype(np.uint32))


def test_f32_to_f16_structured_vs_numpy():
    """Every sign/exponent/top-mantissa pattern (upper 16 bits) with the low 16 bits at every
    rounding-relevant value (ties, one above/below, all-ones) plus random ones; and every pattern
    whose exponent lands in f16's subnormal range with random low bits."""
    hi = np.arange(1 << 16, dtype=np.uint32) << np.uint32(16)
    lows = [0x0000, 0x0001, 0x0FFF, 0x1000, 0x1001, 0x1FFF, 0x2000, 0x2001, 0x3000, 0x7FFF,
            0x8000, 0x8001, 0xEFFF, 0xF000, 0xF001, 0xFFFF]
    rng = np.random.default_rng(3)
    lows += rng.integers(0, 1 << 16, 48).tolist()
    u = (hi[:, None] | np.array(lows, dtype=np.uint32)[None, :]).reshape(-1)
    _check_f32_to_f16(u)
    # f32 exponents 100..113 (values near and below 2^-14): all upper bits, random low 16 bits
    e = np.arange(100, 114, dtype=np.uint32)
    man_hi = np.arange(1 << 7, dtype=np.uint32)
    base = (e[:, None] << np.uint32(23)) | (man_hi[None, :] << np.uint32(16))
    base = base.reshape(-1)
    low = rng.integers(0, 1 << 16, (base.size, 256)).astype(np.uint32)
    u = (base[:, None] | low).reshape(-1)
    _check_f32_to_f16(np.concatenate([u, u | np.uint32(0x80000000)]))


def test_f32_to_f16_boundaries():
    cases = {
        65504.0: 0x7BFF, 65519.996: 0x7BFF, 65520.0: 0x7C00, 2.0 ** -24: 0x0001,
        2.0 ** -25: 0x0000, 2.0 ** -25 * 1.0000001: 0x0001, 3 * 2.0 ** -25: 0x0002,
        1.0 + 2.0 ** -11: 0x3C00, 1.0 + 3 * 2.0 ** -11: 0x3C02, -0.0: 0x8000,
        2.0 ** -14 - 2.0 ** -25: 0x0400,
    }
    f = np.array(list(cases), dtype=np.float32)
    got = oracle.f32_to_f16(f)
    assert got.tolist() == list(cases.values())


def _libm_fmaf():
    libm = ctypes.CDLL(ctypes.util.find_library("m"))
    libm.fmaf.restype = ctypes.c_float
    libm.fmaf.argtypes = [ctypes.c_float] * 3
    return libm.fmaf


def _fma_triples(n, seed):
    rng = np.random.default_rng(seed)
    # a: an f16 value (at most 11 significant bits), b: any moderate f32, c: often close to -a*b
    a = (rng.uniform(-2, 2, n) * 2.0 ** rng.integers(-12, 12, n)).astype(np.float16).astype(np.float32)
    b = (rng.uniform(-1, 1, n) * 2.0 ** rng.integers(-20, 20, n)).astype(np.float32)
    c = (-(a.astype(np.float64) * b) * (1 + rng.uniform(-1e-6, 1e-6, n))).astype(np.float32)
    mix = rng.uniform(0, 1, n) < 0.3
    c[mix] = (rng.uniform(-1, 1, mix.sum()) * 2.0 ** rng.integers(-20, 20, mix.sum())).astype(np.float32)
    return a, b, c


def test_fmaf_is_correctly_rounded_exact_rational():
    """libm fmaf == RN(a*b + c) computed exactly, on a sample including cancellations."""
    fmaf = _libm_fmaf()
    a, b, c = _fma_triples(4000, 7)
    for x, y, z in zip(a.tolist(), b.tolist(), c.tolist()):
        exact = Fraction(x) * Fraction(y) + Fraction(z)
        want = round_f32(exact)
        got = fmaf(x, y, z)
        if want == 0.0:
            assert got == 0.0
        else:
            assert f32_bits(got) == f32_bits(want), (x, y, z)


def test_page_fma_emulation_equals_fmaf():
    """browseml-gpu.js fma_exact (TwoSum + round-to-odd) restated in the oracle agrees bit for bit
    with a correctly rounded fma: the page's fma is read as correctly rounded."""
    fmaf = _libm_fmaf()
    a, b, c = _fma_triples(200000, 11)
    emu = oracle.fma_emulated(a, b, c)
    ref = np.array([fmaf(x, y, z) for x, y, z in zip(a.tolist(), b.tolist(), c.tolist())], dtype=np.float32)
    nz = (ref != 0)
    assert np.array_equal(emu[nz].view(np.uint32), ref[nz].view(np.uint32))
    assert np.all(emu[~nz] == 0)
