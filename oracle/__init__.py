"""CPU oracle for the low-bit matvec/matmul path -- TEST INFRASTRUCTURE ONLY.

Thin ctypes wrapper around ``gq_oracle.c`` (plain scalar C, see its header for the sources and
the readings it takes).  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package; the product library never does.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gq_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no contraction, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            S = ctypes.c_size_t
            L.gqo_f16_to_f32.restype = ctypes.c_float
            L.gqo_f16_to_f32.argtypes = [ctypes.c_uint16]
            L.gqo_f32_to_f16_rne.restype = ctypes.c_uint16
            L.gqo_f32_to_f16_rne.argtypes = [ctypes.c_float]
            L.gqo_fma_emulated.restype = ctypes.c_float
            L.gqo_fma_emulated.argtypes = [ctypes.c_float] * 3
            L.gqo_q1_q8_row.restype = ctypes.c_float
            L.gqo_q1_q8_row.argtypes = [P, P, I, P]
            for name, args in [
                ("gqo_q1_q8_gemv", [P, P, P, I, I]),
                ("gqo_q1_q8_gemm", [P, P, P, I, I, I]),
                ("gqo_block_q8_matmul_nt", [P, P, P, P, I, I, I]),
                ("gqo_ternary_direct", [P, P, P, P, I, I, I]),
                ("gqo_ternary_identity", [P, P, P, P, I, I, I]),
                ("gqo_quantize_q8_0", [P, I, I, P, P]),
                ("gqo_prefill_q1s32", [P, P, P, P, P, I, I, I]),
                ("gqo_q1s32_f32_gemv_f64", [P, P, P, P, I, I, I]),
                ("gqo_w8a32_f64", [P, P, P, P, I, I, I]),
                ("gqo_w4a32g128_f64", [P, P, P, P, I, I, I]),
                ("gqo_f16_to_f32_array", [P, P, S]),
                ("gqo_f32_to_f16_array", [P, P, S]),
                ("gqo_fma_emulated_array", [P, P, P, P, S]),
            ]:
                fn = getattr(L, name)
                fn.restype = None
                fn.argtypes = args
            _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


# ----------------------------------------------------------------------------- scalar formats

def f16_to_f32(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16).reshape(-1)
    out = np.empty(h.size, dtype=np.float32)
    lib().gqo_f16_to_f32_array(_p(h), _p(out), h.size)
    return out


def f32_to_f16(f: np.ndarray) -> np.ndarray:
    f = np.ascontiguousarray(f, dtype=np.float32).reshape(-1)
    out = np.empty(f.size, dtype=np.uint16)
    lib().gqo_f32_to_f16_array(_p(f), _p(out), f.size)
    return out


def fma_emulated(a, b, c) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32).reshape(-1)
    b = np.ascontiguousarray(b, dtype=np.float32).reshape(-1)
    c = np.ascontiguousarray(c, dtype=np.float32).reshape(-1)
    out = np.empty(a.size, dtype=np.float32)
    lib().gqo_fma_emulated_array(_p(a), _p(b), _p(c), _p(out), a.size)
    return out


# ----------------------------------------------------------------------------- the path

def q1_q8_row(wrow: np.ndarray, act: np.ndarray, n: int):
    """One row: (result, the eight lane accumulators)."""
    wrow = np.ascontiguousarray(wrow, dtype=np.uint8)
    act = np.ascontiguousarray(act, dtype=np.uint8)
    lanes = np.zeros(8, dtype=np.float32)
    y = lib().gqo_q1_q8_row(_p(wrow), _p(act), n, _p(lanes))
    return np.float32(y), lanes


def q1_q8_gemv(w: np.ndarray, a: np.ndarray, rows: int, n: int) -> np.ndarray:
    w = np.ascontiguousarray(w, dtype=np.uint8).reshape(-1)
    a = np.ascontiguousarray(a, dtype=np.uint8).reshape(-1)
    assert w.size == rows * (n // 128) * 18 and a.size >= (n // 32) * 34
    y = np.empty(rows, dtype=np.float32)
    lib().gqo_q1_q8_gemv(_p(w), _p(a), _p(y), rows, n)
    return y


def q1_q8_gemm(w: np.ndarray, a: np.ndarray, rows: int, n: int, cols: int) -> np.ndarray:
    """Returns O as [cols, rows] (O[c * rows + r])."""
    w = np.ascontiguousarray(w, dtype=np.uint8).reshape(-1)
    a = np.ascontiguousarray(a, dtype=np.uint8).reshape(-1)
    assert w.size == rows * (n // 128) * 18 and a.size == cols * (n // 32) * 34
    y = np.empty(cols * rows, dtype=np.float32)
    lib().gqo_q1_q8_gemm(_p(w), _p(a), _p(y), rows, n, cols)
    return y.reshape(cols, rows)


def block_q8_matmul_nt(x: np.ndarray, quants: np.ndarray, scales: np.ndarray, m: int, k: int, n: int):
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    quants = np.ascontiguousarray(quants, dtype=np.uint32).reshape(-1)
    scales = np.ascontiguousarray(scales, dtype=np.float32).reshape(-1)
    assert x.size == m * k and quants.size == n * k // 4 and scales.size == n * (k // 32)
    y = np.empty(m * n, dtype=np.float32)
    lib().gqo_block_q8_matmul_nt(_p(x), _p(quants), _p(scales), _p(y), m, k, n)
    return y.reshape(m, n)


def _ternary(fn, P, N, X, rows, k, batch):
    P = np.ascontiguousarray(P, dtype=np.uint32).reshape(-1)
    N = np.ascontiguousarray(N, dtype=np.uint32).reshape(-1)
    X = np.ascontiguousarray(X, dtype=np.uint32).reshape(-1)
    assert P.size == rows * k // 32 and N.size == P.size and X.size == batch * k // 32
    y = np.empty(batch * rows, dtype=np.int32)
    fn(_p(P), _p(N), _p(X), _p(y), rows, k, batch)
    return y.reshape(batch, rows)


def ternary_direct(P, N, X, rows, k, batch):
    return _ternary(lib().gqo_ternary_direct, P, N, X, rows, k, batch)


def ternary_identity(P, N, X, rows, k, batch):
    return _ternary(lib().gqo_ternary_identity, P, N, X, rows, k, batch)


def quantize_q8_0(x: np.ndarray, m: int, k: int):
    """Returns (d f16 bits [m, k/32] uint16, q int8 [m, k])."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    assert x.size == m * k
    d = np.empty(m * (k // 32), dtype=np.uint16)
    q = np.empty(m * k, dtype=np.int8)
    lib().gqo_quantize_q8_0(_p(x), m, k, _p(d), _p(q))
    return d.reshape(m, k // 32), q.reshape(m, k)


def prefill_q1s32(signs, ws, xd, xq, M: int, N: int, K: int) -> np.ndarray:
    signs = np.ascontiguousarray(signs, dtype=np.uint32).reshape(-1)
    ws = np.ascontiguousarray(ws, dtype=np.float32).reshape(-1)
    xd = np.ascontiguousarray(xd, dtype=np.uint16).reshape(-1)
    xq = np.ascontiguousarray(xq, dtype=np.int8).reshape(-1)
    assert signs.size == N * K // 32 and ws.size == signs.size
    assert xd.size == M * K // 32 and xq.size == M * K
    y = np.empty(M * N, dtype=np.float32)
    lib().gqo_prefill_q1s32(_p(signs), _p(ws), _p(xd), _p(xq), _p(y), M, N, K)
    return y.reshape(M, N)


def q1s32_f32_gemv(signs, ws, x, M: int, N: int, K: int) -> np.ndarray:
    """Bonsai decode GEMV over f32 activations, the f64 definition: y[m, n] (float64)."""
    signs = np.ascontiguousarray(signs, dtype=np.uint32).reshape(-1)
    ws = np.ascontiguousarray(ws, dtype=np.float32).reshape(-1)
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    assert signs.size == N * K // 32 and ws.size == signs.size and x.size == M * K
    y = np.empty(M * N, dtype=np.float64)
    lib().gqo_q1s32_f32_gemv_f64(_p(signs), _p(ws), _p(x), _p(y), M, N, K)
    return y.reshape(M, N)


def w8a32(w, scale, x, T: int, N: int, K: int) -> np.ndarray:
    """W8A32 matvec/matmul ([P4] matvecQ8 / matmulQ8): w [N, ceil(K/4)] u32 (int8 codes, LSB
    first), scale [N] f32, x [T, K] f32 -> float64 [T, N]."""
    w = np.ascontiguousarray(w, dtype=np.uint32)
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert w.size == N * ((K + 3) // 4) and scale.size == N and x.size == T * K
    y = np.empty((T, N), dtype=np.float64)
    lib().gqo_w8a32_f64(_p(w), _p(scale), _p(x), _p(y), T, N, K)
    return y


def w4a32g128(w, scale, x, T: int, N: int, K: int) -> np.ndarray:
    """W4A32 group-128 matvec/matmul ([P4] matvecQ4G128 / matmulQ4G128): w [N, ceil(K/8)] u32
    (4-bit two's complement codes, LSB first), scale [N, ceil(K/128)] f32, x [T, K] f32 ->
    float64 [T, N]."""
    w = np.ascontiguousarray(w, dtype=np.uint32)
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert w.size == N * ((K + 7) // 8) and scale.size == N * ((K + 127) // 128) and x.size == T * K
    y = np.empty((T, N), dtype=np.float64)
    lib().gqo_w4a32g128_f64(_p(w), _p(scale), _p(x), _p(y), T, N, K)
    return y
