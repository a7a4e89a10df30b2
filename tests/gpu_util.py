"""Helpers for the GPU parity tests (call the library through its C-ABI binding)."""
import numpy as np
import pytest


def need_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gemm_q1_q8_gb300 import build
    build.build()
    import gemm_q1_q8_gb300 as gq
    gq.lib()
    return gq


def to_dev(a: np.ndarray):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def assert_same_bits(got: np.ndarray, want: np.ndarray, what: str = ""):
    """Bit-for-bit equality of f32 arrays (NaNs compared by class)."""
    g = np.ascontiguousarray(got, dtype=np.float32).reshape(-1)
    w = np.ascontiguousarray(want, dtype=np.float32).reshape(-1)
    assert g.shape == w.shape, (g.shape, w.shape)
    gn, wn = np.isnan(g), np.isnan(w)
    bad = (g.view(np.uint32) != w.view(np.uint32)) & ~(gn & wn)
    if bad.any():
        idx = np.flatnonzero(bad)[:8]
        detail = ", ".join(f"[{i}] got {g[i]!r} ({g.view(np.uint32)[i]:#010x}) want {w[i]!r} "
                           f"({w.view(np.uint32)[i]:#010x})" for i in idx)
        raise AssertionError(f"{what}: {int(bad.sum())} of {g.size} differ: {detail}")
