"""Seeded synthetic inputs for the Q1_0/Q8_0, block-int8 and ternary matvec/matmul workloads.

This module holds no arithmetic of the method itself: it draws random numbers and lays them out
in the input formats that the pages define (byte layouts only).  Both the CPU oracle (``oracle/``)
and the CUDA path (``gemm_q1_q8_gb300``) are fed from here, so neither ever produces the other's
inputs.

Generator: splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
OOPSLA 2014), used counter-style: draw ``i`` of a stream is ``mix(seed + (i + 1) * GOLDEN)``.
Uniform doubles take the top 53 bits.  Each ``Rng`` advances a counter, so a fixed sequence of
calls always yields the same arrays.

Distributions (stated in the workload configs, browseml-gpu.js ``randomCase`` for the extra ones):

* f16 scale: uniform in [lo, hi], random sign, rounded to f16 (numpy's RN-even conversion).
* int8 quant: uniform integer in [-127, 127].
* sign bits: Bernoulli(0.5) (raw generator bits).
* ternary weight: P(0) = 0.4, P(+1) = P(-1) = 0.3, stored as P/N bitplanes.
* N(0, 1): Box-Muller in f64, rounded to f32.
* browseml-gpu.js ``f16bits``: random sign, exponent field in [3, 17), random mantissa.
* browseml-gpu.js ``randomCase``: activation quant byte 0x80 (-128) with probability 0.02.
"""
from __future__ import annotations

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

Q1_0_BYTES, QK1_0 = 18, 128   # per 128 weights: f16 d0 + 128 sign bits
Q8_0_BYTES, QK8_0 = 34, 32    # per 32 activations: f16 d1 + 32 int8


class Rng:
    """Counter-based splitmix64 stream."""

    def __init__(self, seed: int):
        self.seed = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
        self.counter = 0

    def u64(self, n: int) -> np.ndarray:
        i = np.arange(self.counter + 1, self.counter + 1 + n, dtype=np.uint64)
        self.counter += n
        with np.errstate(over="ignore"):
            z = self.seed + i * GOLDEN
            z = (z ^ (z >> np.uint64(30))) * _M1
            z = (z ^ (z >> np.uint64(27))) * _M2
            z = z ^ (z >> np.uint64(31))
        return z

    def u32(self, n: int) -> np.ndarray:
        return self.u64((n + 1) // 2).view(np.uint32)[:n].copy()

    def bytes(self, n: int) -> np.ndarray:
        return self.u64((n + 7) // 8).view(np.uint8)[:n].copy()

    def uniform(self, n: int) -> np.ndarray:
        """Doubles uniform in [0, 1)."""
        return (self.u64(n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)

    def normal(self, n: int) -> np.ndarray:
        """N(0, 1) doubles by Box-Muller."""
        m = (n + 1) // 2
        u1 = 1.0 - self.uniform(m)          # (0, 1]
        u2 = self.uniform(m)
        r = np.sqrt(-2.0 * np.log(u1))
        z = np.concatenate([r * np.cos(2 * np.pi * u2), r * np.sin(2 * np.pi * u2)])
        return z[:n]


# ----------------------------------------------------------------------------- scalar fields

def f16_scales(rng: Rng, n: int, lo: float = 1e-3, hi: float = 1e-1) -> np.ndarray:
    """u16 bit patterns of f16 values uniform in [lo, hi] with a random sign."""
    mag = lo + (hi - lo) * rng.uniform(n)
    sign = np.where(rng.uniform(n) < 0.5, -1.0, 1.0)
    return (sign * mag).astype(np.float16).view(np.uint16)


def f16_page_bits(rng: Rng, n: int, lo: int = 3, hi: int = 17) -> np.ndarray:
    """browseml-gpu.js ``f16bits``: random sign, exponent field in [lo, hi), random mantissa."""
    sign = (rng.uniform(n) < 0.5).astype(np.uint16) << np.uint16(15)
    exp = (lo + np.floor(rng.uniform(n) * (hi - lo))).astype(np.uint16) << np.uint16(10)
    man = np.floor(rng.uniform(n) * 1024).astype(np.uint16)
    return sign | exp | man


def int8_uniform(rng: Rng, n: int) -> np.ndarray:
    """int8 uniform in [-127, 127]."""
    return (np.floor(rng.uniform(n) * 255.0) - 127.0).astype(np.int8)


def int8_page(rng: Rng, n: int, p_min: float = 0.02) -> np.ndarray:
    """browseml-gpu.js ``randomCase`` activation bytes: 0x80 with probability p_min, else any byte."""
    u = rng.uniform(n)
    b = np.floor(rng.uniform(n) * 256.0).astype(np.uint8)
    return np.where(u < p_min, np.uint8(128), b).view(np.int8)


def f32_uniform(rng: Rng, n: int, lo: float, hi: float) -> np.ndarray:
    return (lo + (hi - lo) * rng.uniform(n)).astype(np.float32)


def f32_normal(rng: Rng, n: int) -> np.ndarray:
    return rng.normal(n).astype(np.float32)


# ----------------------------------------------------------------------------- block formats

def q1_0_weights(rng: Rng, rows: int, n: int, scales: str = "uniform") -> np.ndarray:
    """Q1_0 weights as the pages' AoS bytes: rows * (n/128) blocks of 18 bytes
    (f16 d0 little-endian, then 16 bytes of sign bits)."""
    assert n % QK1_0 == 0
    nblk = rows * (n // QK1_0)
    if scales == "uniform":
        d = f16_scales(rng, nblk)
    elif scales == "page":
        d = f16_page_bits(rng, nblk)
    else:
        raise ValueError(scales)
    out = np.empty((nblk, Q1_0_BYTES), dtype=np.uint8)
    out[:, 0:2] = d.view(np.uint8).reshape(nblk, 2)
    out[:, 2:] = rng.bytes(nblk * 16).reshape(nblk, 16)
    return out.reshape(-1)


def q8_0_acts(rng: Rng, cols: int, n: int, scales: str = "uniform", quants: str = "uniform") -> np.ndarray:
    """Q8_0 activations as the pages' AoS bytes: cols vectors of (n/32) blocks of 34 bytes
    (f16 d1 little-endian, then 32 int8)."""
    assert n % QK8_0 == 0
    nblk = cols * (n // QK8_0)
    if scales == "uniform":
        d = f16_scales(rng, nblk)
    elif scales == "page":
        d = f16_page_bits(rng, nblk)
    else:
        raise ValueError(scales)
    if quants == "uniform":
        q = int8_uniform(rng, nblk * 32)
    elif quants == "page":
        q = int8_page(rng, nblk * 32)
    else:
        raise ValueError(quants)
    out = np.empty((nblk, Q8_0_BYTES), dtype=np.uint8)
    out[:, 0:2] = d.view(np.uint8).reshape(nblk, 2)
    out[:, 2:] = q.view(np.uint8).reshape(nblk, 32)
    return out.reshape(-1)


def block_q8_inputs(rng: Rng, m: int, k: int, n: int, scale_lo=1e-3, scale_hi=2e-2):
    """kopitiam block_q8_matmul_nt inputs: x [m,k] f32 N(0,1); quants k*n int8 packed four per
    u32 little-endian (row-major [n, k]); scales [n, k/32] f32 uniform."""
    assert k % 32 == 0
    x = f32_normal(rng, m * k).reshape(m, k)
    q = int8_uniform(rng, n * k)
    quants = q.view(np.uint8).reshape(-1, 4).copy().view(np.uint32).reshape(-1)
    scales = f32_uniform(rng, n * (k // 32), scale_lo, scale_hi).reshape(n, k // 32)
    return x, quants, scales


def ternary_inputs(rng: Rng, rows: int, k: int, batch: int, p_zero: float = 0.4):
    """Ternary weights {-1,0,+1} (P(0)=p_zero, the rest split evenly) as P/N u32 bitplanes
    [rows, k/32] (bit j of word w = element 32w+j), and a Bernoulli(0.5) activation bitplane
    X [batch, k/32]."""
    assert k % 32 == 0
    u = rng.uniform(rows * k).reshape(rows, k)
    half = (1.0 - p_zero) / 2.0
    pos = u < half
    neg = (u >= half) & (u < 2 * half)
    P = np.packbits(pos, axis=1, bitorder="little").view(np.uint32).reshape(rows, k // 32)
    N = np.packbits(neg, axis=1, bitorder="little").view(np.uint32).reshape(rows, k // 32)
    X = rng.u32(batch * (k // 32)).reshape(batch, k // 32)
    return P.copy(), N.copy(), X


def prefill_inputs(rng: Rng, M: int, K: int, N: int, scale_lo=1e-3, scale_hi=5e-2):
    """Bonsai-style 1-bit weights: signs u32 [N, K/32] (bit t of word b = weight 32b+t, 1 -> +1),
    one f32 scale per 32 weights [N, K/32]; f32 activations x [M, K] N(0,1)."""
    assert K % 32 == 0
    signs = rng.u32(N * (K // 32)).reshape(N, K // 32)
    ws = f32_uniform(rng, N * (K // 32), scale_lo, scale_hi).reshape(N, K // 32)
    x = f32_normal(rng, M * K).reshape(M, K)
    return signs, ws, x


def wq_inputs(rng: Rng, T: int, K: int, N: int, bits: int, scale_lo=1e-3, scale_hi=2e-2, p_m8: float = 0.0):
    """Block-quantized weights of the web-xpu-ops formats with f32 activations x [T, K] N(0,1).
    bits = 8: codes uniform in [-127, 127], four per u32 least-significant byte first,
      w [N, ceil(K/4)], one f32 scale per row [N].
    bits = 4: codes uniform in [-7, 7] (with probability p_m8 the raw nibble 0x8 = -8, which the
      quantizer never emits), eight per u32 least-significant nibble first, w [N, ceil(K/8)],
      one f32 scale per 128 columns [N, ceil(K/128)].
    Codes past K (the last word's padding) are zero."""
    per = 32 // bits
    words = (K + per - 1) // per
    if bits == 8:
        codes = (rng.u32(N * K) % 255).astype(np.int64) - 127
    else:
        codes = (rng.u32(N * K) % 15).astype(np.int64) - 7
        if p_m8 > 0:
            codes[rng.uniform(N * K) < p_m8] = -8
    codes = codes.reshape(N, K)
    padded = np.zeros((N, words * per), dtype=np.int64)
    padded[:, :K] = codes
    field = (padded & ((1 << bits) - 1)).astype(np.uint64).reshape(N, words, per)
    shifts = (np.arange(per, dtype=np.uint64) * np.uint64(bits))
    w = (field << shifts).sum(axis=2).astype(np.uint32)
    groups = N if bits == 8 else N * ((K + 127) // 128)
    scale = f32_uniform(rng, groups, scale_lo, scale_hi)
    if bits == 4:
        scale = scale.reshape(N, (K + 127) // 128)
    x = f32_normal(rng, T * K).reshape(T, K)
    return w, scale, x


# ----------------------------------------------------------------------------- named workloads

# BitNet-2B layer shapes for one decode token: four 2560x2560 attention projections, two
# 6912x2560 (gate, up) and one 2560x6912 (down), over a stack of 30 distinct layers.
BITNET_LAYER = [(2560, 2560)] * 4 + [(6912, 2560)] * 2 + [(2560, 6912)]
BITNET_LAYERS = 30

CONFIGS = {
    "gemv_small": dict(rows=256, n=1024, seed=0),
    "gemv_bitnet2b_sweep": dict(shapes=BITNET_LAYER, layers=BITNET_LAYERS, seed=1),
    "block_q8_49152x960": dict(n=49152, k=960, ms=(1, 4, 16), seed=2),
    "ternary_14336x4096": dict(rows=14336, k=4096, batches=(1, 4, 16), seed=3),
    "prefill_512x4096x14336": dict(M=512, K=4096, N=14336, seed=4),
    "wq_14336x4096": dict(N=14336, K=4096, tokens=(1, 512), seed=6),
}


def bitnet_sweep(seed: int = 1, layers: int = BITNET_LAYERS):
    """Yields (rows, n, weights AoS bytes, activation AoS bytes) for every matrix of a decode
    token over ``layers`` distinct layers (each matrix has its own activation vector)."""
    rng = Rng(seed)
    for _ in range(layers):
        for rows, n in BITNET_LAYER:
            w = q1_0_weights(rng, rows, n)
            a = q8_0_acts(rng, 1, n)
            yield rows, n, w, a
