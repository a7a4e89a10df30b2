"""GPU parity of block_q8_matmul_nt (kopitiam-gpu block_q8_matmul_nt.wgsl), the ternary bitplane
GEMV (the Bonsai P/N popcount identity), the Q8_0 activation quantizer and the Bonsai-format
prefill GEMM, against the CPU oracle through the C ABI."""
import json
import os

import numpy as np
import pytest

import oracle
import workloads as wl
import gemm_q1_q8_gb300 as gqmod
from tests.gpu_util import assert_same_bits, need_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gq():
    return need_gpu()


# ----------------------------------------------------------------------------- block_q8

@pytest.mark.parametrize("m,k,n", [(1, 32, 1), (1, 960, 1001), (3, 96, 513), (4, 960, 257), (7, 64, 33),
                                   (16, 960, 300), (17, 320, 129), (40, 128, 64), (2, 2048, 700), (1, 2080, 100),
                                   (4, 32, 33), (1, 960, 20000), (5, 2080, 300), (16, 4096, 40), (4, 8192, 33),
                                   (3, 32, 1), (12, 960, 2000), (4, 64, 60000), (2, 32, 60001), (16, 96, 56000)])
def test_block_q8_bit_exact(gq, m, k, n):
    rng = wl.Rng(m * 1000 + k + n)
    x, quants, scales = wl.block_q8_inputs(rng, m, k, n)
    y = gq.block_q8_matmul_nt(to_dev(x), to_dev(quants), to_dev(scales)).cpu().numpy()
    assert_same_bits(y, oracle.block_q8_matmul_nt(x, quants, scales, m, k, n), f"block_q8 {m}x{k}x{n}")


def test_block_q8_golden_on_gpu(gq):
    from tests.test_oracle_others import pack_quants
    cases = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "block_q8_cases.json")))["cases"]
    for case in cases:
        k = case["k"]
        x = np.zeros((1, k), dtype=np.float32)
        q = np.zeros(k, dtype=np.int8)
        for e, v in case["x"]:
            x[0, e] = v
        for e, v in case["q"]:
            q[e] = v
        sc = np.array(case["scales"], dtype=np.float32).reshape(1, -1)
        y = gq.block_q8_matmul_nt(to_dev(x), to_dev(pack_quants(q)), to_dev(sc)).cpu().numpy()
        assert hex(int(y.view(np.uint32)[0, 0])) == case["expected_f32"], case["name"]


@pytest.mark.parametrize("m", [1, 4, 16])
def test_block_q8_full_size_sampled(gq, m):
    """The 49152 x 960 output projection at m = 1, 4, 16 (as benchmarked); 512 sampled output
    features against the oracle, bit for bit."""
    n, k = 49152, 960
    x, quants, scales = wl.block_q8_inputs(wl.Rng(2 + m), m, k, n)
    y = gq.block_q8_matmul_nt(to_dev(x), to_dev(quants), to_dev(scales)).cpu().numpy()
    cols = np.sort(np.random.default_rng(m).choice(n, 512, replace=False))
    qs = quants.reshape(n, k // 4)[cols]
    want = oracle.block_q8_matmul_nt(x, qs, scales[cols], m, k, cols.size)
    assert_same_bits(y[:, cols], want, f"block_q8 full m={m}")


# ----------------------------------------------------------------------------- ternary

@pytest.mark.parametrize("rows,k,batch,pz", [(1, 1024, 1, 0.4), (130, 2048, 3, 0.4), (300, 4096, 16, 0.0),
                                             (129, 1024, 17, 1.0), (64, 8192, 64, 0.4), (1000, 4096, 1, 0.4),
                                             (300, 5120, 1, 0.4)])
def test_ternary_exact(gq, rows, k, batch, pz):
    P, N, X = wl.ternary_inputs(wl.Rng(rows + k + batch), rows, k, batch, p_zero=pz)
    y = gq.ternary_bitplane_gemv(to_dev(P), to_dev(N), to_dev(X)).cpu().numpy()
    assert np.array_equal(y, oracle.ternary_identity(P, N, X, rows, k, batch))


def test_ternary_overlapping_planes(gq):
    rows, k, batch = 128, 1024, 2
    P, _, X = wl.ternary_inputs(wl.Rng(4), rows, k, batch)
    N = P | wl.Rng(5).u32(P.size).reshape(P.shape)
    y = gq.ternary_bitplane_gemv(to_dev(P), to_dev(N), to_dev(X)).cpu().numpy()
    assert np.array_equal(y, oracle.ternary_direct(P, N, X, rows, k, batch))


@pytest.mark.parametrize("pattern", ["p_ones", "n_ones", "both_ones"])
def test_ternary_saturated_words(gq, pattern):
    """Planes of whole one-words: every word's popcount is 32 and every counter of the carry-save
    grouping reaches its largest value.  K = 3072 leaves one of a block's four chunk groups idle.
    Closed forms: P = 1s, N = 0 gives 2 popc(X) - k; N = 1s, P = 0 gives k - 2 popc(X); both set
    gives 0."""
    rows, k, batch = 100, 3072, 5
    ones = np.full((rows, k // 32), 0xFFFFFFFF, np.uint32)
    zeros = np.zeros_like(ones)
    P, N = {"p_ones": (ones, zeros), "n_ones": (zeros, ones), "both_ones": (ones, ones)}[pattern]
    kw = k // 32
    X = np.stack([np.full(kw, 0xFFFFFFFF, np.uint32), np.zeros(kw, np.uint32), np.full(kw, 0xAAAAAAAA, np.uint32),
                  np.full(kw, 0x55555555, np.uint32), wl.Rng(9).u32(kw)])
    y = gq.ternary_bitplane_gemv(to_dev(P), to_dev(N), to_dev(X)).cpu().numpy()
    assert np.array_equal(y, oracle.ternary_direct(P, N, X, rows, k, batch))
    px = np.array([sum(bin(int(v)).count("1") for v in X[b]) for b in range(batch)], np.int64)
    closed = {"p_ones": 2 * px - k, "n_ones": k - 2 * px, "both_ones": 0 * px}[pattern]
    assert np.array_equal(y, np.repeat(closed[:, None], rows, axis=1).astype(np.int32))


@pytest.mark.parametrize("batch", [1, 4, 16])
def test_ternary_full_size(gq, batch):
    rows, k = 14336, 4096
    P, N, X = wl.ternary_inputs(wl.Rng(3), rows, k, batch)
    y = gq.ternary_bitplane_gemv(to_dev(P), to_dev(N), to_dev(X)).cpu().numpy()
    assert np.array_equal(y, oracle.ternary_identity(P, N, X, rows, k, batch))


# ----------------------------------------------------------------------------- quantizer

def _interleave(q: np.ndarray) -> np.ndarray:
    """The MMA operand order within each 32-block: position 2u <- element u, 2u+1 <- u+16."""
    m, k = q.shape
    b = q.reshape(m, k // 32, 2, 16)
    return np.stack([b[:, :, 0, :], b[:, :, 1, :]], axis=-1).reshape(m, k)


def _bf16_rn(x: np.ndarray) -> np.ndarray:
    """Upper 16 bits of f32 values rounded to nearest, ties to even (finite inputs)."""
    b = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def test_quantize_out_buffers(gq):
    """Caller buffers (out=) get the same bits as freshly allocated ones, also when reused for
    another input (185 blocks: not a multiple of the eight a warp takes)."""
    import torch
    m, k = 37, 160
    bufs = (torch.empty((m, k // 32), dtype=torch.int16, device="cuda"),
            torch.empty((m, k), dtype=torch.int8, device="cuda"),
            torch.empty((3, m, k), dtype=torch.int16, device="cuda"))
    for seed in (1, 2):
        x = to_dev(wl.f32_normal(wl.Rng(seed), m * k).reshape(m, k))
        want = gq.quantize_q8_0(x, mma_operand=True)
        got = gq.quantize_q8_0(x, mma_operand=True, out=bufs)
        for a, b in zip(got, want):
            assert torch.equal(a, b)
        d_only, q_only, none = gq.quantize_q8_0(x, out=(bufs[0], bufs[1], None))
        assert none is None and torch.equal(d_only, want[0]) and torch.equal(q_only, want[1])


@pytest.mark.parametrize("m,k", [(1, 32), (5, 96), (512, 4096)])
def test_quantize_bit_exact(gq, m, k):
    x = wl.f32_normal(wl.Rng(m + k), m * k).reshape(m, k)
    x[0, :32] = 0.0                                   # an all-zero block
    if k >= 64:
        x[-1, 32:64] *= 1e-30                         # a block whose scale underflows in f16
    d, q, op = gq.quantize_q8_0(to_dev(x), mma_operand=True)
    dw, qw = oracle.quantize_q8_0(x, m, k)
    assert np.array_equal(d.cpu().numpy().view(np.uint16), dw)
    assert np.array_equal(q.cpu().numpy(), qw)
    # the MMA operand: three bf16 planes whose sum is f16(d) * q exactly, hi the nearest bf16
    planes = op.cpu().numpy().view(np.uint16).reshape(3, m, k)
    pf = (planes.astype(np.uint32) << 16).view(np.float32).astype(np.float64)      # bf16 -> f64, exact
    dx = np.repeat(dw.view(np.float16).astype(np.float64), 32, axis=1)
    want = _interleave(dx * qw.astype(np.float64))
    assert np.array_equal(pf[0] + pf[1] + pf[2], want)
    assert np.array_equal(planes[0], _bf16_rn(want.astype(np.float32)))
    assert np.all(np.abs(pf[1]) <= np.abs(pf[0]) * 2.0 ** -8) and np.all(np.abs(pf[2]) <= np.abs(pf[1]) * 2.0 ** -8)


# ----------------------------------------------------------------------------- prefill

def run_prefill(gq, signs, ws, x, path):
    """Quantizes x on the GPU and runs the prefill; the GPU's d and q must equal the oracle's
    quantization of the same x, and the oracle's d and q are what the expected values are built
    from (no expected value takes an input from the CUDA path)."""
    M, K = x.shape
    d, q, op = gq.quantize_q8_0(to_dev(x), mma_operand=True)
    y = gq.q1s32_q8_gemm(to_dev(signs), to_dev(ws), d, q, op, path=path)
    dw, qw = oracle.quantize_q8_0(x, M, K)
    assert np.array_equal(d.cpu().numpy().view(np.uint16), dw), "quantizer scales differ from the oracle"
    assert np.array_equal(q.cpu().numpy(), qw), "quantizer codes differ from the oracle"
    return y.cpu().numpy(), dw, qw


@pytest.mark.parametrize("M,N,K", [(1, 1, 64), (5, 130, 128), (33, 257, 1024), (64, 128, 4096)])
def test_prefill_lut4_bit_exact(gq, M, N, K):
    signs, ws, x = wl.prefill_inputs(wl.Rng(M + N + K), M, K, N)
    y, d, q = run_prefill(gq, signs, ws, x, gq.PATH_LUT4)
    assert_same_bits(y, oracle.prefill_q1s32(signs, ws, d, q, M, N, K), f"lut4 {M}x{N}x{K}")


def test_prefill_lut4_full_size_sampled(gq):
    """M = 512 tokens, K = 4096, N = 14336: 24 tokens x 96 weight rows sampled against the oracle."""
    M, K, N = 512, 4096, 14336
    signs, ws, x = wl.prefill_inputs(wl.Rng(4), M, K, N)
    y, d, q = run_prefill(gq, signs, ws, x, gq.PATH_LUT4)
    rng = np.random.default_rng(1)
    ms = np.sort(rng.choice(M, 24, replace=False))
    ns = np.sort(rng.choice(N, 96, replace=False))
    want = oracle.prefill_q1s32(signs[ns], ws[ns], d[ms], q[ms], ms.size, ns.size, K)
    assert_same_bits(y[np.ix_(ms, ns)], want, "lut4 full sampled")


@pytest.mark.parametrize("M,N,K", [(1, 1, 64), (7, 130, 256), (40, 257, 1024)])
def test_prefill_lut4_caller_codes_with_minus128(gq, M, N, K):
    """The LUT4 path on caller-supplied Q8_0 codes that include -128 (the page's randomCase draws
    the byte 0x80 with probability 0.02): a -128 term is -128 whichever the sign bit (the int8
    wrapping negate), bit for bit as the oracle.  The quantizer never emits -128, so only a caller's
    own codes reach this rule."""
    rng = wl.Rng(900 + M + N + K)
    signs = rng.u32(N * K // 32).reshape(N, K // 32)
    ws = wl.f32_uniform(rng, N * K // 32, 1e-3, 5e-2).reshape(N, K // 32)
    xd = wl.f16_page_bits(rng, M * K // 32).reshape(M, K // 32)
    xq = wl.int8_page(rng, M * K).reshape(M, K)
    assert np.any(xq == -128)
    y = gq.q1s32_q8_gemm(to_dev(signs), to_dev(ws), to_dev(xd), to_dev(xq), None, path=gq.PATH_LUT4)
    assert_same_bits(y.cpu().numpy(), oracle.prefill_q1s32(signs, ws, xd, xq, M, N, K), f"lut4 -128 {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (1, 1, 64), (130, 257, 128), (64, 128, 1024), (300, 200, 4096)])
def test_prefill_mma_bit_exact(gq, M, N, K):
    """tcgen05 path: the same bits as the oracle's fixed order (exact block sums on the tensor core)."""
    signs, ws, x = wl.prefill_inputs(wl.Rng(7 * M + N + K), M, K, N)
    y, d, q = run_prefill(gq, signs, ws, x, gq.PATH_MMA)
    assert_same_bits(y, oracle.prefill_q1s32(signs, ws, d, q, M, N, K), f"mma {M}x{N}x{K}")
    assert gq.device_error() == 0


def test_prefill_mma_full_size_sampled(gq):
    """M = 512 tokens, K = 4096, N = 14336 (as benchmarked): MMA equals LUT4 everywhere, and 24 tokens
    x 96 weight rows equal the oracle."""
    M, K, N = 512, 4096, 14336
    signs, ws, x = wl.prefill_inputs(wl.Rng(4), M, K, N)
    y, d, q = run_prefill(gq, signs, ws, x, gq.PATH_MMA)
    y2, _, _ = run_prefill(gq, signs, ws, x, gq.PATH_LUT4)
    assert_same_bits(y, y2, "mma vs lut4 full")
    rng = np.random.default_rng(2)
    ms = np.sort(rng.choice(M, 24, replace=False))
    ns = np.sort(rng.choice(N, 96, replace=False))
    want = oracle.prefill_q1s32(signs[ns], ws[ns], d[ms], q[ms], ms.size, ns.size, K)
    assert_same_bits(y[np.ix_(ms, ns)], want, "mma full sampled")
    assert gq.device_error() == 0


# ----------------------------------------------------------------------------- Bonsai W1A32

def _w1a32_terms(ws, x):
    """sum_b |ws[n, b]| * sum_t |x[m, 32 b + t]| for every (m, n)."""
    M, K = x.shape
    N, nbk = ws.shape
    ax = np.abs(x.astype(np.float64)).reshape(M, nbk, 32).sum(axis=2)       # [M, nbk]
    return ax @ np.abs(ws.astype(np.float64)).T                              # [M, N]


def _w1a32_depth(path, M, nbk):
    """Roundings any one term passes through in the kernel's order (the gamma_n forward bound
    |got - exact| <= c * 2^-24 * sum |terms| holds with this c, plus slack):
    FMA: 31 adds of the block sum, one fma per block of the lane, a 5-level lane butterfly.
    LUT4 decode (M <= 4, K % 128 == 0): two adds in a table entry, seven between the eight
    lookups, one fma per block of the warp's share (16 per 32-block stage of its K slice, K cut in
    up to eight slices), one add of the two halves, up to seven adds across the slices.
    LUT4 otherwise: two adds in a table entry, seven between lookups, one fma per block.
    Tensor cores ("mma"): six tensor-core steps per block (three bf16 parts x two K16 steps, two
    units each: their accumulation rounding is not published), one fma per block, and slack."""
    if path == "mma":
        return nbk + 16
    if path == gqmod.PATH_FMA:
        return 40 + -(-nbk // 32)
    if M <= 4 and nbk % 4 == 0:
        return 32 + -(-nbk // 8)
    return 12 + nbk


def _w1a32_check(y, want, ws, x, path, M):
    terms = _w1a32_terms(ws, x)
    err = np.abs(y.astype(np.float64) - want)
    bound = _w1a32_depth(path, M, ws.shape[1]) * 2.0 ** -24 * terms
    assert np.all(err <= bound), f"max err/bound {np.max(err / bound)}"
    # the pages' 1e-4 relative / 1e-6 absolute tolerance wherever the result is not a cancellation
    big = np.abs(want) > 1e-2 * terms
    assert np.all(err[big] <= 1e-4 * np.abs(want[big]) + 1e-6)


W1A32_PATHS = [gqmod.PATH_LUT4, gqmod.PATH_FMA]


@pytest.mark.parametrize("path", W1A32_PATHS)
@pytest.mark.parametrize("M", [1, 2, 3, 7, 40])
def test_w1a32_exact_special_case(gq, path, M):
    """Integer activations and power-of-two scales: every partial sum is exact in f32, so the GPU
    result equals the exact value bit for bit, whatever the order."""
    N, K = 77, 1024
    rng = wl.Rng(33 + M)
    signs = rng.u32(N * K // 32).reshape(N, K // 32)
    ws = (2.0 ** -(2 + (rng.u32(N * K // 32) % 5).astype(np.int64))).astype(np.float32).reshape(N, K // 32)
    x = ((rng.u32(M * K) % 17).astype(np.int64) - 8).astype(np.float32).reshape(M, K)
    y = gq.q1s32_f32_gemm(to_dev(signs.view(np.int32)), to_dev(ws), to_dev(x), path=path).cpu().numpy()
    want = oracle.q1s32_f32_gemv(signs, ws, x, M, N, K)
    assert np.array_equal(y.astype(np.float64), want)


@pytest.mark.parametrize("path", W1A32_PATHS)
@pytest.mark.parametrize("M,N,K", [(1, 1, 32), (1, 33, 96), (2, 130, 1024), (3, 300, 8224), (4, 64, 4096),
                                   (1, 200, 16384), (3, 129, 2560), (1, 14336, 4096), (1, 1000, 1152),
                                   (1, 33, 128), (1, 500, 5120), (1, 70, 5248),
                                   (1, 20000, 1024),   # more than three 32-row tiles per block
                                   (5, 257, 160), (16, 513, 1056), (33, 300, 4128), (70, 1000, 512)])
def test_w1a32_within_bound(gq, path, M, N, K):
    signs, ws, x = wl.prefill_inputs(wl.Rng(M + N + K), M, K, N)
    y = gq.q1s32_f32_gemm(to_dev(signs.view(np.int32)), to_dev(ws), to_dev(x), path=path).cpu().numpy()
    _w1a32_check(y, oracle.q1s32_f32_gemv(signs, ws, x, M, N, K), ws, x, path, M)


@pytest.mark.parametrize("path", W1A32_PATHS)
def test_w1a32_deterministic(gq, path):
    M, N, K = 9, 700, 2048
    signs, ws, x = wl.prefill_inputs(wl.Rng(77), M, K, N)
    args = (to_dev(signs.view(np.int32)), to_dev(ws), to_dev(x))
    a = gq.q1s32_f32_gemm(*args, path=path).cpu().numpy()
    b = gq.q1s32_f32_gemm(*args, path=path).cpu().numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("path", W1A32_PATHS)
def test_w1a32_decode_full_size(gq, path):
    """The 14336 x 4096 Bonsai projection at one token, every row against the f64 oracle."""
    M, N, K = 1, 14336, 4096
    signs, ws, x = wl.prefill_inputs(wl.Rng(5), M, K, N)
    y = gq.q1s32_f32_gemm(to_dev(signs.view(np.int32)), to_dev(ws), to_dev(x), path=path).cpu().numpy()
    _w1a32_check(y, oracle.q1s32_f32_gemv(signs, ws, x, M, N, K), ws, x, path, M)


def test_w1a32_prefill_full_size_sampled(gq):
    """M = 512 tokens x 14336 rows x K = 4096 through the LUT4 prefill kernel, in the launch the
    bench times; sampled rows and tokens (spanning every thread-block tile edge) against the oracle."""
    M, N, K = 512, 14336, 4096
    signs, ws, x = wl.prefill_inputs(wl.Rng(4), M, K, N)
    y = gq.q1s32_f32_gemm(to_dev(signs.view(np.int32)), to_dev(ws), to_dev(x), path=gqmod.PATH_LUT4).cpu().numpy()
    ns = np.unique(np.concatenate([np.arange(0, N, 997), [255, 256, N - 1]]))
    ms = np.unique(np.concatenate([np.arange(0, M, 37), [31, 32, M - 1]]))
    want = oracle.q1s32_f32_gemv(signs[ns], ws[ns], x[ms], ms.size, ns.size, K)
    _w1a32_check(y[np.ix_(ms, ns)], want, ws[ns], x[ms], gqmod.PATH_LUT4, M)


# ---- W1A32 on the tensor cores ---------------------------------------------------------------

def _w1a32_mma(gq, signs, ws, x, **kw):
    return gq.q1s32_f32_gemm_mma(to_dev(signs.view(np.int32)), to_dev(ws), to_dev(x), **kw).cpu().numpy()


@pytest.mark.parametrize("M,N,K", [(1, 1, 64), (5, 130, 128), (33, 257, 1024), (129, 300, 4096), (200, 129, 2560),
                                   (7, 1000, 16384), (130, 128, 64)])
def test_w1a32_mma_within_bound(gq, M, N, K):
    """Ragged tokens and rows across the 128 x 128 tile, one to many stages."""
    signs, ws, x = wl.prefill_inputs(wl.Rng(3000 + M + N + K), M, K, N)
    _w1a32_check(_w1a32_mma(gq, signs, ws, x), oracle.q1s32_f32_gemv(signs, ws, x, M, N, K), ws, x, "mma", M)


@pytest.mark.parametrize("M", [1, 40, 200])
def test_w1a32_mma_exact_special_case(gq, M):
    """Integer activations and power-of-two scales: the bf16 split is x itself and every partial
    sum is exact, so the tensor-core path equals the exact value bit for bit."""
    N, K = 77, 1024
    rng = wl.Rng(44 + M)
    signs = rng.u32(N * K // 32).reshape(N, K // 32)
    ws = (2.0 ** -(2 + (rng.u32(N * K // 32) % 5).astype(np.int64))).astype(np.float32).reshape(N, K // 32)
    x = ((rng.u32(M * K) % 17).astype(np.int64) - 8).astype(np.float32).reshape(M, K)
    assert np.array_equal(_w1a32_mma(gq, signs, ws, x).astype(np.float64), oracle.q1s32_f32_gemv(signs, ws, x, M, N, K))


def test_w1a32_mma_deterministic_and_workspace(gq):
    import torch
    M, N, K = 150, 700, 2048
    signs, ws, x = wl.prefill_inputs(wl.Rng(78), M, K, N)
    dirty = torch.full((gq.q1s32_mma_workspace_bytes(M, K) + 32,), 0x7F, dtype=torch.uint8, device="cuda")
    a = _w1a32_mma(gq, signs, ws, x, workspace=dirty)
    b = _w1a32_mma(gq, signs, ws, x)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    assert gq.device_error() == 0


def test_w1a32_mma_full_size_sampled(gq):
    """M = 512 tokens x 14336 rows x K = 4096 on the tensor cores; sampled rows and tokens."""
    M, N, K = 512, 14336, 4096
    signs, ws, x = wl.prefill_inputs(wl.Rng(4), M, K, N)
    y = _w1a32_mma(gq, signs, ws, x)
    ns = np.unique(np.concatenate([np.arange(0, N, 997), [127, 128, N - 1]]))
    ms = np.unique(np.concatenate([np.arange(0, M, 37), [127, 128, M - 1]]))
    want = oracle.q1s32_f32_gemv(signs[ns], ws[ns], x[ms], ms.size, ns.size, K)
    _w1a32_check(y[np.ix_(ms, ns)], want, ws[ns], x[ms], "mma", M)
