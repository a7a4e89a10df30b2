"""The kernels that are launched as programmatic dependents (weights requested before the
wait for the preceding grids, activations read and outputs written after it) must still see an
activation produced by the operation just before them on the stream, and their output writes
must land after the previous call's.  Each case overwrites the activation buffer on the stream
right before the second call and writes both calls into the same output; the second result must
equal the oracle (bit-exact paths) or a lone call of the same kernel (tolerance paths, which are
deterministic)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import assert_same_bits, need_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gq():
    need_gpu()
    import gemm_q1_q8_gb300 as m
    return m


def _chain(first, second, x_dev, x2):
    """first(x_dev) -> y; then x_dev <- x2 on the stream; second(x_dev, out=y); returns y."""
    y = first(x_dev)
    x_dev.copy_(to_dev(x2))
    second(x_dev, y)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def test_ternary_dependent(gq):
    rows, k = 3000, 4096
    P1, N1, X1 = wl.ternary_inputs(wl.Rng(1), rows, k, 1)
    P2, N2, X2 = wl.ternary_inputs(wl.Rng(2), rows, k, 1)
    p1, n1, p2, n2 = (to_dev(a) for a in (P1, N1, P2, N2))
    x = to_dev(X1)
    y = _chain(lambda xd: gq.ternary_bitplane_gemv(p1, n1, xd),
               lambda xd, out: gq.ternary_bitplane_gemv(p2, n2, xd, out=out), x, X2)
    assert np.array_equal(y.reshape(-1), oracle.ternary_identity(P2, N2, X2, rows, k, 1).reshape(-1))


def test_block_q8_dependent(gq):
    m, k, n = 1, 960, 5000
    x1, q1, s1 = wl.block_q8_inputs(wl.Rng(3), m, k, n)
    x2, q2, s2 = wl.block_q8_inputs(wl.Rng(4), m, k, n)
    qa, sa, qb, sb = to_dev(q1), to_dev(s1), to_dev(q2), to_dev(s2)
    x = to_dev(x1)
    y = _chain(lambda xd: gq.block_q8_matmul_nt(xd, qa, sa),
               lambda xd, out: gq.block_q8_matmul_nt(xd, qb, sb, out=out), x, x2)
    assert_same_bits(y, oracle.block_q8_matmul_nt(x2, q2, s2, m, k, n), "block_q8 dependent")


@pytest.mark.parametrize("bits", [8, 4])
def test_wq_matvec_dependent(gq, bits):
    N, K = 5000, 4096
    w1, c1, xa = wl.wq_inputs(wl.Rng(5), 1, K, N, bits)
    w2, c2, xb = wl.wq_inputs(wl.Rng(6), 1, K, N, bits)
    mv = gq.matvec_q8 if bits == 8 else gq.matvec_q4g128
    wa, ca, wb, cb = to_dev(w1.view(np.int32)), to_dev(c1), to_dev(w2.view(np.int32)), to_dev(c2)
    x = to_dev(xa)
    y = _chain(lambda xd: mv(wa, ca, xd), lambda xd, out: mv(wb, cb, xd, out=out), x, xb)
    lone = mv(wb, cb, to_dev(xb)).cpu().numpy()
    assert np.array_equal(y.view(np.uint32), lone.view(np.uint32))


def test_w1a32_decode_dependent(gq):
    N, K = 5000, 4096
    s1, ws1, xa = wl.prefill_inputs(wl.Rng(7), 1, K, N)
    s2, ws2, xb = wl.prefill_inputs(wl.Rng(8), 1, K, N)
    sa, wa, sb, wb = to_dev(s1.view(np.int32)), to_dev(ws1), to_dev(s2.view(np.int32)), to_dev(ws2)
    x = to_dev(xa)
    y = _chain(lambda xd: gq.q1s32_f32_gemm(sa, wa, xd), lambda xd, out: gq.q1s32_f32_gemm(sb, wb, xd, out=out), x, xb)
    lone = gq.q1s32_f32_gemm(sb, wb, to_dev(xb)).cpu().numpy()
    assert np.array_equal(y.view(np.uint32), lone.view(np.uint32))


@pytest.mark.parametrize("bits", [8, 4])
def test_wq_mma_dependent(gq, bits):
    """The tensor-core matmul starts before its activation split finishes (only its activation
    copies wait): a rewritten activation and a shared workspace must still give the lone result."""
    T, N, K = 300, 2000, 2048
    w1, c1, xa = wl.wq_inputs(wl.Rng(9), T, K, N, bits)
    w2, c2, xb = wl.wq_inputs(wl.Rng(10), T, K, N, bits)
    mm = gq.matmul_q8_mma if bits == 8 else gq.matmul_q4g128_mma
    wa, ca, wb, cb = to_dev(w1.view(np.int32)), to_dev(c1), to_dev(w2.view(np.int32)), to_dev(c2)
    ws = torch.empty(gq.wq_mma_workspace_bytes(T, K), dtype=torch.uint8, device="cuda")
    x = to_dev(xa)
    y = _chain(lambda xd: mm(wa, ca, xd, workspace=ws), lambda xd, out: mm(wb, cb, xd, out=out, workspace=ws), x, xb)
    lone = mm(wb, cb, to_dev(xb)).cpu().numpy()
    assert np.array_equal(y.view(np.uint32), lone.view(np.uint32))
