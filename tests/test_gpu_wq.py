"""GPU parity for the W8A32 (per-row scale) and W4A32 group-128 matvec/matmul (web-xpu-ops README:
matvecQ8 / matmulQ8 / matvecQ4G128 / matmulQ4G128) against the f64 oracle.  The page fixes no
float order, so each result must lie within the forward error bound of the kernel's own order,
and within 1e-4 relative / 1e-6 absolute wherever it is not a cancellation."""
import numpy as np
import pytest

import oracle
import workloads as wl
from tests.gpu_util import need_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gq():
    need_gpu()
    import gemm_q1_q8_gb300 as m
    return m


def _terms(bits, w, scale, x, N, K):
    """sum_k |scale| * |code| * |x| per (t, n), from an unpack written here with numpy."""
    if bits == 8:
        codes = w.view("<u4").view(np.int8).reshape(N, -1)[:, :K].astype(np.float64)
        return (np.abs(x.astype(np.float64)) @ np.abs(codes).T) * np.abs(scale.astype(np.float64))[None, :]
    nib = ((w[:, :, None] >> (4 * np.arange(8, dtype=np.uint32))[None, None, :]) & 0xF).reshape(N, -1)[:, :K]
    codes = nib.astype(np.float64) - 16.0 * (nib >= 8)
    sc = np.repeat(np.abs(scale.astype(np.float64)), 128, axis=1)[:, :K]
    return np.abs(x.astype(np.float64)) @ (np.abs(codes) * sc).T


def _depth(bits, T, K, mma=False):
    """Roundings a term passes through in the kernel's order.
    T <= 4 (GEMV): 8 bits -- an fma chain over the lane's 16 columns of each of its warp's 512-column
    chunks, a 5-level lane butterfly, a 3-level warp tree, the row-scale multiply; 4 bits -- a
    16-term chain per chunk, one fma with the group scale per chunk, the butterfly and tree.
    T > 4 (GEMM): one fma per column, plus the scale multiply (8 bits) or the dequantizing product
    code * scale (4 bits).
    Tensor cores (matmul_*_mma): per 128-column round, 24 MMA steps (three planes x 8 K16 steps)
    into a fresh accumulator -- the hardware's accumulation rounding is not published, so each step
    is allowed two units -- then a round-to-nearest f32 add (or fma with the group scale) of each
    round partial in round order (ceil(K/128)), the scale multiply, and 7 units of slack for the
    sums inside a step."""
    if mma:
        return -(-K // 128) + 2 * 24 + 8
    if T <= 4:
        return 16 * -(-K // 4096) + 10 if bits == 8 else 28 + -(-K // 512)
    return K + 2


def _check(bits, y, want, w, scale, x, T, N, K, mma=False):
    terms = _terms(bits, w, scale, x, N, K)
    err = np.abs(y.astype(np.float64) - want)
    bound = _depth(bits, T, K, mma) * 2.0 ** -24 * terms
    assert np.all(err <= bound), f"max err/bound {np.max(err / np.maximum(bound, 1e-300))}"
    big = np.abs(want) > 1e-2 * terms
    assert np.all(err[big] <= 1e-4 * np.abs(want[big]) + 1e-6)


def _run(gq, bits, w, scale, x, mma=False):
    T = x.shape[0]
    args = (to_dev(w.view(np.int32)), to_dev(scale), to_dev(x))
    if mma:
        return (gq.matmul_q8_mma if bits == 8 else gq.matmul_q4g128_mma)(*args).cpu().numpy()
    if bits == 8:
        y = gq.matvec_q8(*args) if T == 1 else gq.matmul_q8(*args)
    else:
        y = gq.matvec_q4g128(*args) if T == 1 else gq.matmul_q4g128(*args)
    return y.cpu().numpy()


def _oracle(bits, w, scale, x, T, N, K):
    return oracle.w8a32(w, scale, x, T, N, K) if bits == 8 else oracle.w4a32g128(w, scale, x, T, N, K)


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("T,N,K", [(1, 1, 32), (1, 77, 96), (1, 1000, 544), (2, 129, 4128), (3, 40, 1024),
                                   (4, 300, 2560), (5, 257, 160), (33, 130, 1056), (130, 300, 512),
                                   (1, 3000, 16384), (1, 97, 5152), (1, 50, 24608)])
def test_within_bound(gq, bits, T, N, K):
    w, scale, x = wl.wq_inputs(wl.Rng(1000 * bits + T + N + K), T, K, N, bits, p_m8=0.02)
    _check(bits, _run(gq, bits, w, scale, x), _oracle(bits, w, scale, x, T, N, K), w, scale, x, T, N, K)


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("T", [1, 3, 9])
def test_exact_special_case(gq, bits, T):
    """Integer x in [-8, 8] and power-of-two scales: every partial sum is exact in f32 at this size,
    so the GPU equals the oracle bit for bit, whatever the order."""
    N, K = 200, 1024
    rng = wl.Rng(60 + bits + T)
    w, scale, _ = wl.wq_inputs(rng, T, K, N, bits, p_m8=0.05)
    scale = (2.0 ** -(1 + (rng.u32(scale.size) % 6).astype(np.int64))).astype(np.float32).reshape(scale.shape)
    x = ((rng.u32(T * K) % 17).astype(np.int64) - 8).astype(np.float32).reshape(T, K)
    assert np.array_equal(_run(gq, bits, w, scale, x).astype(np.float64), _oracle(bits, w, scale, x, T, N, K))


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("T", [1, 2, 64])
def test_deterministic(gq, bits, T):
    N, K = 700, 2048
    w, scale, x = wl.wq_inputs(wl.Rng(5 + T), T, K, N, bits)
    a, b = _run(gq, bits, w, scale, x), _run(gq, bits, w, scale, x)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("bits", [8, 4])
def test_matvec_full_size(gq, bits):
    """14336 x 4096 at one token, every row against the oracle."""
    T, N, K = 1, 14336, 4096
    w, scale, x = wl.wq_inputs(wl.Rng(6), T, K, N, bits)
    _check(bits, _run(gq, bits, w, scale, x), _oracle(bits, w, scale, x, T, N, K), w, scale, x, T, N, K)


@pytest.mark.parametrize("bits", [8, 4])
def test_matmul_full_size_sampled(gq, bits):
    """512 tokens x 14336 rows x 4096: sampled rows and tokens (across tile edges) against the oracle."""
    T, N, K = 512, 14336, 4096
    w, scale, x = wl.wq_inputs(wl.Rng(6), T, K, N, bits)
    y = _run(gq, bits, w, scale, x)
    ns = np.unique(np.concatenate([np.arange(0, N, 911), [127, 128, N - 1]]))
    ts = np.unique(np.concatenate([np.arange(0, T, 41), [63, 64, 127, 128, T - 1]]))
    want = _oracle(bits, w[ns], scale[ns], x[ts], ts.size, ns.size, K)
    _check(bits, y[np.ix_(ts, ns)], want, w[ns], scale[ns], x[ts], T, ns.size, K)


# ---- the tensor-core matmuls -------------------------------------------------------------------

@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("T,N,K", [(1, 1, 64), (5, 257, 96), (33, 130, 1056), (128, 128, 64), (129, 129, 4128),
                                   (130, 300, 512), (300, 1000, 2048), (7, 3000, 16384)])
def test_mma_within_bound(gq, bits, T, N, K):
    """Ragged tokens and rows across the 128 x 128 tile, K % 64 == 32 tails (and, for 4 bits, a
    last group shorter than 128), one to many K stages."""
    w, scale, x = wl.wq_inputs(wl.Rng(7000 + bits + T + N + K), T, K, N, bits, p_m8=0.02)
    _check(bits, _run(gq, bits, w, scale, x, mma=True), _oracle(bits, w, scale, x, T, N, K), w, scale, x, T, N, K,
           mma=True)


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("T", [1, 9, 200])
def test_mma_exact_special_case(gq, bits, T):
    """Integer x in [-8, 8] and power-of-two scales: the bf16 split is x itself and every partial
    sum is exact, so the tensor cores give the oracle's value bit for bit."""
    N, K = 300, 1024
    rng = wl.Rng(80 + bits + T)
    w, scale, _ = wl.wq_inputs(rng, T, K, N, bits, p_m8=0.05)
    scale = (2.0 ** -(1 + (rng.u32(scale.size) % 6).astype(np.int64))).astype(np.float32).reshape(scale.shape)
    x = ((rng.u32(T * K) % 17).astype(np.int64) - 8).astype(np.float32).reshape(T, K)
    assert np.array_equal(_run(gq, bits, w, scale, x, mma=True).astype(np.float64),
                          _oracle(bits, w, scale, x, T, N, K))


def test_mma_split_is_exact(gq):
    """One nonzero code per row selects single activations: y = scale * code * x exactly, so the
    three bf16 planes must sum back to every x (normal range, all exponents of N(0,1) data)."""
    T, N, K = 140, 256, 256
    rng = wl.Rng(91)
    x = rng.normal(T * K).astype(np.float32).reshape(T, K)
    codes = np.zeros((N, K), np.int8)
    codes[np.arange(N), np.arange(N) % K] = 1
    w = codes.view(np.uint32).reshape(N, K // 4)
    scale = np.ones(N, np.float32)
    y = _run(gq, 8, w, scale, x, mma=True)
    assert np.array_equal(y, x[:, np.arange(N) % K])


def test_mma_q4_code_range(gq):
    """Every 4-bit code -8..7 once per row position (a raw 0x8 reads as -8), integer x: exact."""
    T, N, K = 3, 16, 128
    codes = (np.arange(N * K) % 16).reshape(N, K).astype(np.uint32)
    w = np.zeros((N, K // 8), np.uint32)
    for j in range(8):
        w |= codes[:, j::8] << np.uint32(4 * j)
    scale = np.ones((N, 1), np.float32)
    x = np.zeros((T, K), np.float32)
    x[0, :] = 1.0
    x[1, np.arange(K) % 16 == 8] = 1.0
    x[2, :] = np.arange(K) % 5 - 2
    y = _run(gq, 4, w, scale, x, mma=True)
    assert np.array_equal(y.astype(np.float64), _oracle(4, w, scale, x, T, N, K))
    assert np.all(y[1] == -8.0 * (K // 16))


@pytest.mark.parametrize("bits", [8, 4])
def test_mma_deterministic_and_workspace(gq, bits):
    import torch
    T, N, K = 260, 700, 2048
    w, scale, x = wl.wq_inputs(wl.Rng(17), T, K, N, bits)
    dw, ds, dx = to_dev(w.view(np.int32)), to_dev(scale), to_dev(x)
    fn = gq.matmul_q8_mma if bits == 8 else gq.matmul_q4g128_mma
    ws = torch.full((gq.wq_mma_workspace_bytes(T, K) + 64,), 0x7F, dtype=torch.uint8, device="cuda")
    a = fn(dw, ds, dx, workspace=ws).cpu().numpy()
    b = fn(dw, ds, dx).cpu().numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    assert gq.device_error() == 0


@pytest.mark.parametrize("bits", [8, 4])
def test_mma_full_size_sampled(gq, bits):
    """512 tokens x 14336 rows x 4096 on the tensor cores: sampled rows and tokens against the oracle."""
    T, N, K = 512, 14336, 4096
    w, scale, x = wl.wq_inputs(wl.Rng(6), T, K, N, bits)
    y = _run(gq, bits, w, scale, x, mma=True)
    ns = np.unique(np.concatenate([np.arange(0, N, 911), [127, 128, N - 1]]))
    ts = np.unique(np.concatenate([np.arange(0, T, 41), [63, 64, 127, 128, T - 1]]))
    want = _oracle(bits, w[ns], scale[ns], x[ts], ts.size, ns.size, K)
    _check(bits, y[np.ix_(ts, ns)], want, w[ns], scale[ns], x[ts], T, ns.size, K, mma=True)
