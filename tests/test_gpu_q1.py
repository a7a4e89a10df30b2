"""GPU parity of the Q1_0 . Q8_0 path (browseml-gpu.js Q1_DOT_WGSL / Q1_MM_WGSL / Q1_MM4_WGSL
semantics) against the CPU oracle, bit for bit, through the C ABI."""
import numpy as np
import pytest

import oracle
import workloads as wl
from tests.gpu_util import assert_same_bits, need_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gq():
    return need_gpu()


def gemv(gq, w, a, rows, n):
    packed = gq.q1_0_pack(to_dev(w), rows, n)
    return gq.q1_q8_gemv(packed, to_dev(a), rows, n).cpu().numpy()


@pytest.mark.parametrize("rows,n,dist,seed", [
    (256, 1024, "uniform", 0),      # the small decode workload: 256 rows, 8 blocks
    (1, 128, "uniform", 1),
    (1, 128, "page", 2),
    (129, 640, "page", 3),          # a ragged second tile
    (300, 2560, "page", 4),
    (1000, 6912, "uniform", 5),
    (77, 16384, "page", 6),         # 128 blocks: four passes of the block-parallel kernel
    (2560, 2560, "uniform", 8),     # a BitNet-2B attention projection
    (19500, 256, "page", 7),        # 153 tiles: more than the GPU's SMs, the persistent kernel
])
def test_gemv_bit_exact(gq, rows, n, dist, seed):
    rng = wl.Rng(1000 + seed)
    w = wl.q1_0_weights(rng, rows, n, scales=dist)
    a = wl.q8_0_acts(rng, 1, n, scales=dist, quants=dist)
    assert_same_bits(gemv(gq, w, a, rows, n), oracle.q1_q8_gemv(w, a, rows, n), f"gemv {rows}x{n} {dist}")


def test_gemv_all_minus128_and_zero_scales(gq):
    """Degenerate inputs: every quant -128 (the wrapping negate everywhere), zero scales."""
    rows, n = 64, 512
    rng = wl.Rng(77)
    w = wl.q1_0_weights(rng, rows, n)
    a = wl.q8_0_acts(rng, 1, n).reshape(-1, 34).copy()
    a[:, 2:] = 0x80
    a[::3, 0:2] = 0                                   # d1 = +0 on a third of the blocks
    a = a.reshape(-1)
    w2 = w.reshape(-1, 18).copy()
    w2[::5, 0:2] = [0x00, 0x80]                       # d0 = -0 on a fifth
    w2 = w2.reshape(-1)
    assert_same_bits(gemv(gq, w2, a, rows, n), oracle.q1_q8_gemv(w2, a, rows, n), "degenerate")


def test_golden_cases_on_gpu(gq):
    import json
    import os
    from tests.test_oracle_q1 import build_case
    cases = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "q1_q8_cases.json")))["cases"]
    for case in cases:
        w, a, n = build_case(case)
        y = gemv(gq, w, a, 1, n)
        assert hex(int(y.view(np.uint32)[0])) == case["expected_f32"], case["name"]


def test_f16_weight_scale_every_pattern(gq):
    """All 65536 f16 patterns as d0 (one row each, lane 0 = 1 * 1): the decode of every scale,
    subnormals, signed zeros, Inf and NaN included, matches the oracle's integer decode."""
    rows, n = 65536, 128
    w = np.zeros((rows, 18), dtype=np.uint8)
    w[:, 0:2] = np.arange(rows, dtype=np.uint16).view(np.uint8).reshape(rows, 2)
    w[:, 2] = 0x01                                    # weight 0 of sub-block 0 set
    a = np.zeros((4, 34), dtype=np.uint8)
    a[0, 0:2] = [0x00, 0x3C]                          # d1 = 1
    a[0, 2] = 1                                       # q0 = 1 -> lane 0: s = 1
    y = gemv(gq, w.reshape(-1), a.reshape(-1), rows, n)
    assert_same_bits(y, oracle.q1_q8_gemv(w.reshape(-1), a.reshape(-1), rows, n), "d0 patterns")


def test_f16_activation_scale_every_pattern(gq):
    """All 65536 f16 patterns as d1, spread over the columns of a GEMM (512 blocks per column;
    the Inf/NaN patterns in columns of their own)."""
    n, rows = 16384, 2
    pats = np.arange(65536, dtype=np.uint16)
    finite = pats[((pats >> 10) & 0x1F) != 0x1F]
    nonfin = pats[((pats >> 10) & 0x1F) == 0x1F]
    order = np.concatenate([finite, nonfin])
    per = n // 32
    cols = (order.size + per - 1) // per
    d1 = np.zeros(cols * per, dtype=np.uint16)
    d1[:order.size] = order
    rng = wl.Rng(88)
    a = wl.q8_0_acts(rng, cols, n).reshape(-1, 34)
    a[:, 0:2] = d1.view(np.uint8).reshape(-1, 2)
    a = a.reshape(-1)
    w = wl.q1_0_weights(rng, rows, n)
    packed = gq.q1_0_pack(to_dev(w), rows, n)
    y = gq.q1_q8_gemm(packed, to_dev(a), rows, n, cols, gq.PATH_DP4A).cpu().numpy()
    assert_same_bits(y, oracle.q1_q8_gemm(w, a, rows, n, cols), "d1 patterns")


@pytest.mark.parametrize("path", ["dp4a", "lut4"])
@pytest.mark.parametrize("rows,n,cols,dist", [
    (256, 1024, 5, "page"),           # five activations: a partial tile of four (Q1_MM4_WGSL)
    (130, 512, 1, "uniform"),
    (300, 2560, 9, "page"),
    (64, 6912, 4, "uniform"),
])
def test_gemm_bit_exact(gq, path, rows, n, cols, dist):
    rng = wl.Rng(hash((rows, n, cols, dist)) & 0xFFFF)
    w = wl.q1_0_weights(rng, rows, n, scales=dist)
    a = wl.q8_0_acts(rng, cols, n, scales=dist, quants=dist)
    p = gq.PATH_DP4A if path == "dp4a" else gq.PATH_LUT4
    packed = gq.q1_0_pack(to_dev(w), rows, n)
    y = gq.q1_q8_gemm(packed, to_dev(a), rows, n, cols, p).cpu().numpy()
    assert_same_bits(y, oracle.q1_q8_gemm(w, a, rows, n, cols), f"gemm {path}")


def test_gemm_column_equals_gemv(gq):
    rows, n, cols = 200, 1024, 6
    rng = wl.Rng(9)
    w = wl.q1_0_weights(rng, rows, n)
    a = wl.q8_0_acts(rng, cols, n, quants="page")
    packed = gq.q1_0_pack(to_dev(w), rows, n)
    Y = gq.q1_q8_gemm(packed, to_dev(a), rows, n, cols).cpu().numpy()
    ab = (n // 32) * 34
    for c in range(cols):
        yc = gq.q1_q8_gemv(packed, to_dev(a[c * ab:(c + 1) * ab]), rows, n).cpu().numpy()
        assert_same_bits(Y[c], yc, f"column {c}")


def test_grouped_equals_single_small(gq):
    import torch
    rng = wl.Rng(12)
    shapes = [(256, 1024), (1, 128), (1000, 2560), (129, 6912), (700, 640)]
    items, ref = [], []
    for rows, n in shapes:
        w = wl.q1_0_weights(rng, rows, n, scales="page")
        a = wl.q8_0_acts(rng, 1, n, quants="page")
        packed = gq.q1_0_pack(to_dev(w), rows, n)
        y = torch.empty(rows, dtype=torch.float32, device="cuda")
        items.append((packed, to_dev(a), y, rows, n))
        ref.append(oracle.q1_q8_gemv(w, a, rows, n))
    g = gq.GroupedGemv(items)
    g()
    for (packed, act, y, rows, n), want in zip(items, ref):
        assert_same_bits(y.cpu().numpy(), want, f"grouped {rows}x{n}")
    assert gq.device_error() == 0


def test_grouped_more_tiles_than_warps(gq):
    """More 128-row tiles than the persistent grid has warps, so every warp takes several units
    through the hand-out counter: every row of every matrix (ragged last tiles, several n, Q8_0
    and f32 activations) equals the oracle bit for bit, and a second call over the same outputs
    (counter and constants rebuilt) gives the same bits."""
    import torch
    sms = gq.lib().gq_probe_sm_count()
    rng = wl.Rng(777)
    shapes = [(20_001, 640), (100_005, 384), (40_077, 256), (120_033, 256), (30_001, 128), (70_003, 128)]
    assert sum((r + 127) // 128 for r, _ in shapes) > 16 * sms     # more tiles than warps
    items, want = [], []
    for i, (rows, n) in enumerate(shapes):
        w = wl.q1_0_weights(rng, rows, n, scales="page")
        packed = gq.q1_0_pack(to_dev(w), rows, n)
        y = torch.empty(rows, dtype=torch.float32, device="cuda")
        if i == 4:
            x = _act_f32(rng, n, "normal")
            items.append((packed, to_dev(x), y, rows, n))
            want.append(oracle.q1_q8_gemv(w, _q8_0_blocks(x, n), rows, n))
        else:
            a = wl.q8_0_acts(rng, 1, n, quants="page")
            items.append((packed, to_dev(a), y, rows, n))
            want.append(oracle.q1_q8_gemv(w, a, rows, n))
    g = gq.GroupedGemv(items)
    for call in range(2):
        g()
        torch.cuda.synchronize()
        for (_, _, y, rows, n), wv in zip(items, want):
            assert_same_bits(y.cpu().numpy(), wv, f"many tiles {rows}x{n}, call {call}")
    assert gq.device_error() == 0


def test_bitnet_sweep_full_size_sampled(gq):
    """The BitNet-2B decode sweep (30 layers x 7 matrices, 334.5 MB of Q1_0 weights) in one grouped
    launch, as the benchmark times it: every matrix's output equals its single-matrix GEMV bit for
    bit, and 48 sampled rows of every matrix equal the oracle."""
    import torch
    items, raw = [], []
    for rows, n, w, a in wl.bitnet_sweep(seed=1):
        packed = gq.q1_0_pack(to_dev(w), rows, n)
        y = torch.empty(rows, dtype=torch.float32, device="cuda")
        items.append((packed, to_dev(a), y, rows, n))
        raw.append((w, a))
    g = gq.GroupedGemv(items)
    g()
    torch.cuda.synchronize()
    sel = np.random.default_rng(5)
    for (packed, act, y, rows, n), (w, a) in zip(items, raw):
        got = y.cpu().numpy()
        single = gq.q1_q8_gemv(packed, act, rows, n).cpu().numpy()
        assert_same_bits(got, single, f"grouped vs single {rows}x{n}")
        rb = (n // 128) * 18
        for r in sel.choice(rows, 48, replace=False):
            want, _ = oracle.q1_q8_row(w[r * rb:(r + 1) * rb], a, n)
            assert_same_bits(got[r:r + 1], np.array([want]), f"row {r} of {rows}x{n}")
    assert gq.device_error() == 0


# ----------------------------------------------------------------------------- fused quantization

def _q8_0_blocks(x, n):
    """The Q8_0 bytes (f16 d little-endian, then 32 int8) of the oracle's quantization of x."""
    d, q = oracle.quantize_q8_0(x, 1, n)
    blocks = np.zeros((n // 32, 34), dtype=np.uint8)
    blocks[:, 0:2] = d.reshape(-1, 1).view(np.uint8).reshape(-1, 2)
    blocks[:, 2:] = q.reshape(-1, 32).view(np.uint8)
    return blocks.reshape(-1)


def _act_f32(rng, n, kind):
    x = wl.f32_normal(rng, n)
    if kind == "zeros":                    # every third block all zero: d = 0, q = 0
        x.reshape(-1, 32)[::3] = 0.0
    elif kind == "ties":                   # x = (k + 1/2) * d for the block's own d: round half up
        xb = x.reshape(-1, 32)
        xb[:, 0] = 127.0
        xb[:, 1:] = (np.round(xb[:, 1:] * 20) + 0.5).astype(np.float32)
    elif kind == "range":                  # magnitudes spread over many binades
        x = (x * np.exp2(rng.uniform(n) * 40 - 20)).astype(np.float32)
    return x


@pytest.mark.parametrize("rows,n,kind", [(256, 1024, "normal"), (256, 1024, "zeros"), (130, 2560, "ties"),
                                         (2560, 2560, "range"), (19500, 256, "normal")])
def test_gemv_f32_fused_quantize(gq, rows, n, kind):
    """q1_q8_gemv_f32 == the oracle's Q8_0 quantization followed by the oracle GEMV, bit for bit."""
    rng = wl.Rng(4242 + rows + n)
    w = wl.q1_0_weights(rng, rows, n)
    x = _act_f32(rng, n, kind)
    packed = gq.q1_0_pack(to_dev(w), rows, n)
    y = gq.q1_q8_gemv_f32(packed, to_dev(x), rows, n).cpu().numpy()
    assert_same_bits(y, oracle.q1_q8_gemv(w, _q8_0_blocks(x, n), rows, n), f"gemv_f32 {rows}x{n} {kind}")


def test_grouped_mixed_activation_formats(gq):
    """A grouped sweep mixing Q8_0 and f32 activations: each output equals its own oracle GEMV."""
    import torch
    rng = wl.Rng(5151)
    items, want = [], []
    for i, (rows, n) in enumerate([(2560, 2560), (6912, 2560), (2560, 6912), (300, 1024)]):
        w = wl.q1_0_weights(rng, rows, n)
        packed = gq.q1_0_pack(to_dev(w), rows, n)
        y = torch.empty(rows, dtype=torch.float32, device="cuda")
        if i % 2 == 0:
            x = _act_f32(rng, n, "normal")
            items.append((packed, to_dev(x), y, rows, n))
            want.append(oracle.q1_q8_gemv(w, _q8_0_blocks(x, n), rows, n))
        else:
            a = wl.q8_0_acts(rng, 1, n)
            items.append((packed, to_dev(a), y, rows, n))
            want.append(oracle.q1_q8_gemv(w, a, rows, n))
    g = gq.GroupedGemv(items)
    g()
    for (_, _, y, rows, n), wv in zip(items, want):
        assert_same_bits(y.cpu().numpy(), wv, f"grouped mixed {rows}x{n}")


# ----------------------------------------------------------------------------- the pages' own bytes

@pytest.mark.parametrize("rows,n,dist,seed", [
    (1, 128, "page", 40),
    (33, 1024, "uniform", 41),        # one 8-block step
    (300, 2560, "page", 42),          # ragged rows (300 = 9 x 32 + 12), 20 blocks: a ragged last step
    (257, 1152, "page", 43),          # 9 blocks: a one-block last step
    (1000, 6912, "uniform", 44),
])
def test_gemv_raw_bit_exact(gq, rows, n, dist, seed):
    """q1_q8_gemv_raw reads the 18-byte Q1_0 blocks as stored (no repack): the oracle's bits, and
    the same bits as the resident-layout GEMV."""
    rng = wl.Rng(2000 + seed)
    w = wl.q1_0_weights(rng, rows, n, scales=dist)
    a = wl.q8_0_acts(rng, 1, n, scales=dist, quants=dist)
    y = gq.q1_q8_gemv_raw(to_dev(w), to_dev(a), rows, n).cpu().numpy()
    assert_same_bits(y, oracle.q1_q8_gemv(w, a, rows, n), f"raw {rows}x{n} {dist}")
    assert_same_bits(y, gemv(gq, w, a, rows, n), f"raw vs packed {rows}x{n}")


def test_gemv_raw_degenerate(gq):
    """Every quant -128 and zero scales on the raw path."""
    rows, n = 64, 512
    rng = wl.Rng(78)
    w = wl.q1_0_weights(rng, rows, n)
    a = wl.q8_0_acts(rng, 1, n).reshape(-1, 34).copy()
    a[:, 2:] = 0x80
    a[::3, 0:2] = 0
    a = a.reshape(-1)
    y = gq.q1_q8_gemv_raw(to_dev(w), to_dev(a), rows, n).cpu().numpy()
    assert_same_bits(y, oracle.q1_q8_gemv(w, a, rows, n), "raw degenerate")


@pytest.mark.parametrize("cols,n", [(1, 32), (3, 2560), (5, 96)])
def test_pack_q8_0_layout(gq, cols, n):
    """packQ8: per 32-block the f16 scale decoded to f32 and the 32 quant bytes as eight
    little-endian words; the expected arrays are the input bytes viewed through numpy."""
    a = wl.q8_0_acts(wl.Rng(90 + cols), cols, n, scales="page", quants="page")
    d, q = gq.pack_q8_0(to_dev(a), cols, n)
    blocks = a.reshape(cols * n // 32, 34)
    want_d = blocks[:, :2].copy().view(np.float16).astype(np.float32).reshape(cols, n // 32)
    want_q = blocks[:, 2:].copy().view("<u4").reshape(cols, n // 32, 8)
    assert np.array_equal(d.cpu().numpy().view(np.uint32), want_d.view(np.uint32))
    assert np.array_equal(q.cpu().numpy().view(np.uint32), want_q)
