"""gemm_q1_q8_gb300 -- Python binding of libgq (low-bit block-quantized GEMV/GEMM for GB300).

Argument marshalling only: every function checks the torch tensors it is given (device, dtype,
contiguity, size), allocates outputs with torch, and calls the C ABI (include/gq.h) on the
current CUDA stream.  Every step of the computation runs in the library's kernels; there is no
CPU or PyTorch fallback, and a missing library is an error.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

__all__ = [
    "lib", "GQError", "PATH_AUTO", "PATH_DP4A", "PATH_LUT4", "PATH_MMA", "PATH_FMA",
    "q1_0_packed_bytes", "q1_0_pack", "q1_q8_gemv", "q1_q8_gemv_f32", "q1_q8_gemv_noalloc", "GroupedGemv",
    "q1_q8_gemv_raw", "pack_q8_0",
    "q1_q8_gemm", "ACT_Q8_0", "ACT_F32",
    "block_q8_matmul_nt", "ternary_bitplane_gemv", "quantize_q8_0", "q1s32_q8_gemm", "q1s32_f32_gemm",
    "matvec_q8", "matmul_q8", "matmul_q8_mma", "wq_mma_workspace_bytes", "matvec_q4g128", "matmul_q4g128",
    "matmul_q4g128_mma", "q1s32_f32_gemm_mma", "q1s32_mma_workspace_bytes",
    "device_error", "version", "PROBE_KINDS", "probe_fill", "probe_read", "probe_issue", "probe_mma",
]

PATH_AUTO, PATH_DP4A, PATH_LUT4, PATH_MMA, PATH_FMA = 0, 1, 2, 3, 4
_LIB = None


class GQError(RuntimeError):
    pass


class _Desc(ctypes.Structure):
    _fields_ = [("packed_w", ctypes.c_void_p), ("act", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("rows", ctypes.c_int), ("n", ctypes.c_int),
                ("tile_begin", ctypes.c_int), ("act_format", ctypes.c_int)]


ACT_Q8_0, ACT_F32 = 0, 1


def lib():
    """The loaded libgq.so.  Raises if it has not been built (``__graft_entry__.build()``)."""
    global _LIB
    if _LIB is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise GQError(f"libgq.so is not built ({path}); run __graft_entry__.build()")
        L = ctypes.CDLL(path)
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        sig = {
            "gq_version": (ctypes.c_char_p, []),
            "gq_status_string": (ctypes.c_char_p, [I]),
            "gq_last_cuda_error": (I, []),
            "gq_device_error": (I, []),
            "gq_q1_0_packed_bytes": (S, [I, I]),
            "gq_q1_0_pack": (I, [P, I, I, P, P]),
            "gq_q1_q8_workspace_bytes": (S, [I]),
            "q1_q8_gemv": (I, [P, P, P, I, I, P, P]),
            "q1_q8_gemv_noalloc": (I, [P, P, P, I, I, P]),
            "q1_q8_gemv_f32": (I, [P, P, P, I, I, P, P]),
            "q1_q8_gemv_raw": (I, [P, P, P, I, I, P]),
            "gq_pack_q8_0": (I, [P, I, I, P, P, P]),
            "gq_gemv_group_plan": (I, [P, I, P]),
            "q1s32_f32_gemm": (I, [P, P, P, P, I, I, I, I, P]),
            "matvec_q8": (I, [P, P, P, P, I, I, P]),
            "matmul_q8": (I, [P, P, P, P, I, I, I, P]),
            "gq_wq_mma_workspace_bytes": (S, [I, I]),
            "matmul_q8_mma": (I, [P, P, P, P, I, I, I, P, P]),
            "matmul_q4g128_mma": (I, [P, P, P, P, I, I, I, P, P]),
            "gq_q1s32_mma_workspace_bytes": (S, [I, I]),
            "q1s32_f32_gemm_mma": (I, [P, P, P, P, I, I, I, P, P]),
            "matvec_q4g128": (I, [P, P, P, P, I, I, P]),
            "matmul_q4g128": (I, [P, P, P, P, I, I, I, P]),
            "q1_q8_gemv_grouped": (I, [P, I, I, P, P]),
            "q1_q8_gemm": (I, [P, P, P, I, I, I, I, P]),
            "block_q8_matmul_nt": (I, [P, P, P, P, I, I, I, P]),
            "ternary_bitplane_gemv": (I, [P, P, P, P, I, I, I, P]),
            "gq_quantize_q8_0": (I, [P, I, I, P, P, P, P]),
            "q1s32_q8_gemm": (I, [P, P, P, P, P, P, I, I, I, I, P]),
            "gq_probe_sm_count": (I, []),
            "gq_probe_fill": (I, [P, S, ctypes.c_uint32, P]),
            "gq_probe_read": (I, [P, S, P, I, I, P]),
            "gq_probe_issue": (I, [I, I, P, P, P]),
            "gq_probe_issue_insts": (ctypes.c_double, [I, I]),
            "gq_probe_mma": (I, [I, I, I, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def version() -> str:
    return lib().gq_version().decode()


def _check(status: int, what: str):
    if status != 0:
        L = lib()
        msg = L.gq_status_string(status).decode()
        extra = f" (cudaError {L.gq_last_cuda_error()})" if status == 4 else ""
        raise GQError(f"{what}: {msg}{extra}")


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _need(t: torch.Tensor, dtype, numel: int, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise GQError(f"{name}: expected a CUDA tensor")
    if t.dtype != dtype:
        raise GQError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise GQError(f"{name}: must be contiguous")
    if t.numel() != numel:
        raise GQError(f"{name}: expected {numel} elements, got {t.numel()}")


def device_error() -> int:
    """Reads and clears the library's device-side error word (synchronizes the device)."""
    return lib().gq_device_error()


# ----------------------------------------------------------------------------- Q1_0 x Q8_0

def q1_0_packed_bytes(rows: int, n: int) -> int:
    return lib().gq_q1_0_packed_bytes(rows, n)


def q1_0_pack(raw: torch.Tensor, rows: int, n: int) -> torch.Tensor:
    """Repack Q1_0 AoS bytes (uint8, rows*(n/128)*18) into the resident layout."""
    _need(raw, torch.uint8, rows * (n // 128) * 18 if n % 128 == 0 else -1, "raw")
    nbytes = q1_0_packed_bytes(rows, n)
    if nbytes == 0:
        raise GQError("q1_0_pack: invalid shape")
    packed = torch.empty(nbytes, dtype=torch.uint8, device=raw.device)
    _check(lib().gq_q1_0_pack(_ptr(raw), rows, n, _ptr(packed), _stream()), "gq_q1_0_pack")
    return packed


def workspace_bytes(n: int) -> int:
    return lib().gq_q1_q8_workspace_bytes(n)


def q1_q8_gemv(packed: torch.Tensor, act: torch.Tensor, rows: int, n: int, out: torch.Tensor | None = None,
               workspace: torch.Tensor | None = None):
    """y[r] for a packed rows x n Q1_0 matrix and one Q8_0 vector (uint8, n/32*34 bytes)."""
    _need(act, torch.uint8, (n // 32) * 34, "act")
    _need(packed, torch.uint8, q1_0_packed_bytes(rows, n), "packed")
    y = torch.empty(rows, dtype=torch.float32, device=act.device) if out is None else out
    _need(y, torch.float32, rows, "out")
    ws = torch.empty(workspace_bytes(n), dtype=torch.uint8, device=act.device) if workspace is None else workspace
    _need(ws, torch.uint8, workspace_bytes(n), "workspace")
    _check(lib().q1_q8_gemv(_ptr(packed), _ptr(act), _ptr(y), rows, n, _ptr(ws), _stream()), "q1_q8_gemv")
    return y


def q1_q8_gemv_raw(w: torch.Tensor, act: torch.Tensor, rows: int, n: int, out: torch.Tensor | None = None):
    """y[r] for a rows x n Q1_0 matrix in the pages' own 18-byte blocks (uint8, no repack) and one
    Q8_0 vector (uint8, n/32*34 bytes)."""
    _need(w, torch.uint8, rows * (n // 128) * 18 if n % 128 == 0 else -1, "w")
    _need(act, torch.uint8, (n // 32) * 34, "act")
    y = torch.empty(rows, dtype=torch.float32, device=act.device) if out is None else out
    _need(y, torch.float32, rows, "out")
    _check(lib().q1_q8_gemv_raw(_ptr(w), _ptr(act), _ptr(y), rows, n, _stream()), "q1_q8_gemv_raw")
    return y


def pack_q8_0(raw: torch.Tensor, cols: int, n: int):
    """The pages' packQ8: `cols` Q8_0 vectors (uint8, cols*n/32*34 bytes) -> (d f32 [cols, n/32],
    q int32 [cols, n/32, 8], the quant bytes four to a little-endian word)."""
    _need(raw, torch.uint8, cols * (n // 32) * 34 if n % 32 == 0 else -1, "raw")
    d = torch.empty((cols, n // 32), dtype=torch.float32, device=raw.device)
    q = torch.empty((cols, n // 32, 8), dtype=torch.int32, device=raw.device)
    _check(lib().gq_pack_q8_0(_ptr(raw), cols, n, _ptr(d), _ptr(q), _stream()), "gq_pack_q8_0")
    return d, q


def q1_q8_gemv_f32(packed: torch.Tensor, x: torch.Tensor, rows: int, n: int, out: torch.Tensor | None = None,
                   workspace: torch.Tensor | None = None):
    """y[r] for a packed rows x n Q1_0 matrix and one f32 activation vector (n values), quantized to
    Q8_0 inside the call: bit-identical to quantize_q8_0 followed by q1_q8_gemv."""
    _need(x, torch.float32, n, "x")
    _need(packed, torch.uint8, q1_0_packed_bytes(rows, n), "packed")
    y = torch.empty(rows, dtype=torch.float32, device=x.device) if out is None else out
    _need(y, torch.float32, rows, "out")
    ws = torch.empty(workspace_bytes(n), dtype=torch.uint8, device=x.device) if workspace is None else workspace
    _need(ws, torch.uint8, workspace_bytes(n), "workspace")
    _check(lib().q1_q8_gemv_f32(_ptr(packed), _ptr(x), _ptr(y), rows, n, _ptr(ws), _stream()), "q1_q8_gemv_f32")
    return y


def q1_q8_gemv_noalloc(packed: torch.Tensor, act: torch.Tensor, rows: int, n: int,
                       out: torch.Tensor | None = None):
    """q1_q8_gemv without a caller workspace: the library's built-in scratch block is used (for
    callers that cannot allocate device memory; n <= 16384; calls must not overlap on the GPU).
    Only the output tensor, when not given, is allocated here by torch."""
    _need(act, torch.uint8, (n // 32) * 34, "act")
    _need(packed, torch.uint8, q1_0_packed_bytes(rows, n), "packed")
    y = torch.empty(rows, dtype=torch.float32, device=act.device) if out is None else out
    _need(y, torch.float32, rows, "out")
    _check(lib().q1_q8_gemv_noalloc(_ptr(packed), _ptr(act), _ptr(y), rows, n, _stream()), "q1_q8_gemv_noalloc")
    return y


class GroupedGemv:
    """A planned grouped GEMV: one launch over many (packed weights, activation, output) triples."""

    def __init__(self, items, device="cuda"):
        """items: sequence of (packed, act, y, rows, n) with CUDA tensors (kept alive here); an act
        of dtype uint8 holds n/32 Q8_0 blocks, one of dtype float32 n values quantized in the call."""
        self._keep = []
        host = (_Desc * len(items))()
        offs, total = [], 0
        for rows, n in ((it[3], it[4]) for it in items):
            offs.append(total)
            total += (workspace_bytes(n) + 255) // 256 * 256
        self.workspace = torch.empty(total + 256, dtype=torch.uint8, device=device)
        self.counter = self.workspace[total:total + 16].view(torch.int32)
        base = self.workspace.data_ptr()
        for i, (packed, act, y, rows, n) in enumerate(items):
            fmt = ACT_F32 if act.dtype == torch.float32 else ACT_Q8_0
            if fmt == ACT_F32:
                _need(act, torch.float32, n, f"act[{i}]")
            else:
                _need(act, torch.uint8, (n // 32) * 34, f"act[{i}]")
            _need(packed, torch.uint8, q1_0_packed_bytes(rows, n), f"packed[{i}]")
            _need(y, torch.float32, rows, f"y[{i}]")
            host[i] = _Desc(packed.data_ptr(), act.data_ptr(), y.data_ptr(), base + offs[i], rows, n, 0, fmt)
            self._keep += [packed, act, y]
        tiles = ctypes.c_int(0)
        _check(lib().gq_gemv_group_plan(ctypes.cast(host, ctypes.c_void_p), len(items), ctypes.byref(tiles)),
               "gq_gemv_group_plan")
        raw = bytes(host)
        self.descs = torch.frombuffer(bytearray(raw), dtype=torch.uint8).to(device)
        self.count, self.tiles = len(items), tiles.value

    def __call__(self):
        _check(lib().q1_q8_gemv_grouped(_ptr(self.descs), self.count, self.tiles, _ptr(self.counter), _stream()),
               "q1_q8_gemv_grouped")


def q1s32_f32_gemm(signs: torch.Tensor, wscale: torch.Tensor, x: torch.Tensor, path: int = PATH_AUTO,
                   out: torch.Tensor | None = None):
    """Bonsai 1-bit weights times f32 activations: signs [N, K/32] int32 (u32 bits), wscale
    [N, K/32] f32, x [M, K] f32 (16-byte aligned) -> y [M, N] f32.  path: PATH_LUT4 (AUTO) or
    PATH_FMA."""
    N, nbk = signs.shape
    M, K = x.shape
    _need(signs, torch.int32, N * nbk, "signs")
    _need(wscale, torch.float32, N * nbk, "wscale")
    _need(x, torch.float32, M * K, "x")
    if K != 32 * nbk:
        raise GQError("q1s32_f32_gemm: x has K columns, signs K/32 words per row")
    y = torch.empty((M, N), dtype=torch.float32, device=x.device) if out is None else out
    _need(y, torch.float32, M * N, "out")
    _check(lib().q1s32_f32_gemm(_ptr(signs), _ptr(wscale), _ptr(x), _ptr(y), M, N, K, path, _stream()),
           "q1s32_f32_gemm")
    return y


def q1s32_mma_workspace_bytes(M: int, K: int) -> int:
    """Bytes of the workspace q1s32_f32_gemm_mma needs for M tokens of K columns (3 * M * K bf16)."""
    return lib().gq_q1s32_mma_workspace_bytes(M, K)


def q1s32_f32_gemm_mma(signs: torch.Tensor, wscale: torch.Tensor, x: torch.Tensor, out: torch.Tensor | None = None,
                       workspace: torch.Tensor | None = None):
    """q1s32_f32_gemm on the tensor cores (x split exactly into three bf16 planes): signs [N, K/32]
    int32, wscale [N, K/32] f32, x [M, K] f32 -> y [M, N] f32.  workspace: a uint8 CUDA tensor of at
    least q1s32_mma_workspace_bytes(M, K) bytes (allocated here when None)."""
    N, nbk = signs.shape
    M, K = x.shape
    _need(signs, torch.int32, N * nbk, "signs")
    _need(wscale, torch.float32, N * nbk, "wscale")
    _need(x, torch.float32, M * K, "x")
    if K != 32 * nbk:
        raise GQError("q1s32_f32_gemm_mma: x has K columns, signs K/32 words per row")
    y = torch.empty((M, N), dtype=torch.float32, device=x.device) if out is None else out
    _need(y, torch.float32, M * N, "out")
    need = q1s32_mma_workspace_bytes(M, K)
    if need == 0:
        raise GQError("q1s32_f32_gemm_mma: invalid shape")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    _need(workspace, torch.uint8, workspace.numel(), "workspace")
    if workspace.numel() < need:
        raise GQError(f"q1s32_f32_gemm_mma: workspace holds {workspace.numel()} bytes, needs {need}")
    _check(lib().q1s32_f32_gemm_mma(_ptr(signs), _ptr(wscale), _ptr(x), _ptr(y), M, N, K, _ptr(workspace),
                                    _stream()), "q1s32_f32_gemm_mma")
    return y


def _wq(bits: int, w: torch.Tensor, scale: torch.Tensor, x: torch.Tensor, out, name: str):
    N = w.shape[0]
    T, K = x.shape
    _need(w, torch.int32, N * K * bits // 32, "w")
    _need(scale, torch.float32, N if bits == 8 else N * ((K + 127) // 128), "scale")
    _need(x, torch.float32, T * K, "x")
    y = torch.empty((T, N), dtype=torch.float32, device=x.device) if out is None else out
    _need(y, torch.float32, T * N, "out")
    fn = getattr(lib(), name)
    if name.startswith("matvec"):
        if T != 1:
            raise GQError(f"{name}: x must hold one token")
        _check(fn(_ptr(w), _ptr(scale), _ptr(x), _ptr(y), N, K, _stream()), name)
    else:
        _check(fn(_ptr(w), _ptr(scale), _ptr(x), _ptr(y), T, N, K, _stream()), name)
    return y


def matvec_q8(w: torch.Tensor, scale: torch.Tensor, x: torch.Tensor, out: torch.Tensor | None = None):
    """W8A32 GEMV: w [N, K/4] int32 (int8 codes, LSB first), scale [N] f32, x [1, K] f32 -> y [1, N]."""
    return _wq(8, w, scale, x, out, "matvec_q8")


def matmul_q8(w: torch.Tensor, scale: torch.Tensor, x: torch.Tensor, out: torch.Tensor | None = None):
    """W8A32 GEMM: w [N, K/4] int32, scale [N] f32, x [T, K] f32 -> y [T, N] f32."""
    return _wq(8, w, scale, x, out, "matmul_q8")


def wq_mma_workspace_bytes(T: int, K: int) -> int:
    """Bytes of the workspace matmul_q8_mma needs for T tokens of K columns (3 * T * K bf16)."""
    return lib().gq_wq_mma_workspace_bytes(T, K)


def _wq_mma(bits: int, w, scale, x, out, workspace, name: str):
    N = w.shape[0]
    T, K = x.shape
    _need(w, torch.int32, N * K * bits // 32, "w")
    _need(scale, torch.float32, N if bits == 8 else N * ((K + 127) // 128), "scale")
    _need(x, torch.float32, T * K, "x")
    y = torch.empty((T, N), dtype=torch.float32, device=x.device) if out is None else out
    _need(y, torch.float32, T * N, "out")
    need = wq_mma_workspace_bytes(T, K)
    if need == 0:
        raise GQError(f"{name}: invalid shape")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    _need(workspace, torch.uint8, workspace.numel(), "workspace")
    if workspace.numel() < need:
        raise GQError(f"{name}: workspace holds {workspace.numel()} bytes, needs {need}")
    _check(getattr(lib(), name)(_ptr(w), _ptr(scale), _ptr(x), _ptr(y), T, N, K, _ptr(workspace), _stream()), name)
    return y


def matmul_q8_mma(w: torch.Tensor, scale: torch.Tensor, x: torch.Tensor, out: torch.Tensor | None = None,
                  workspace: torch.Tensor | None = None):
    """matmul_q8 on the tensor cores (x split exactly into three bf16 planes): w [N, K/4] int32,
    scale [N] f32, x [T, K] f32 -> y [T, N] f32.  workspace: a uint8 CUDA tensor of at least
    wq_mma_workspace_bytes(T, K) bytes (allocated here when None)."""
    return _wq_mma(8, w, scale, x, out, workspace, "matmul_q8_mma")


def matmul_q4g128_mma(w: torch.Tensor, scale: torch.Tensor, x: torch.Tensor, out: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None):
    """matmul_q4g128 on the tensor cores: w [N, K/8] int32, scale [N, ceil(K/128)] f32, x [T, K] f32
    -> y [T, N] f32; workspace as matmul_q8_mma."""
    return _wq_mma(4, w, scale, x, out, workspace, "matmul_q4g128_mma")


def matvec_q4g128(w: torch.Tensor, scale: torch.Tensor, x: torch.Tensor, out: torch.Tensor | None = None):
    """W4A32 group-128 GEMV: w [N, K/8] int32 (4-bit codes, LSB first), scale [N, ceil(K/128)] f32,
    x [1, K] f32 -> y [1, N]."""
    return _wq(4, w, scale, x, out, "matvec_q4g128")


def matmul_q4g128(w: torch.Tensor, scale: torch.Tensor, x: torch.Tensor, out: torch.Tensor | None = None):
    """W4A32 group-128 GEMM: w [N, K/8] int32, scale [N, ceil(K/128)] f32, x [T, K] f32 -> y [T, N]."""
    return _wq(4, w, scale, x, out, "matmul_q4g128")


def q1_q8_gemm(packed: torch.Tensor, act: torch.Tensor, rows: int, n: int, cols: int, path: int = PATH_AUTO,
               out: torch.Tensor | None = None):
    """O[c, r] ([cols, rows] f32) for `cols` Q8_0 vectors (uint8, cols*(n/32)*34 bytes)."""
    _need(act, torch.uint8, cols * (n // 32) * 34, "act")
    _need(packed, torch.uint8, q1_0_packed_bytes(rows, n), "packed")
    y = torch.empty((cols, rows), dtype=torch.float32, device=act.device) if out is None else out
    _need(y, torch.float32, rows * cols, "out")
    _check(lib().q1_q8_gemm(_ptr(packed), _ptr(act), _ptr(y), rows, n, cols, path, _stream()), "q1_q8_gemm")
    return y


# ----------------------------------------------------------------------------- block_q8_matmul_nt

def block_q8_matmul_nt(x: torch.Tensor, quants: torch.Tensor, scales: torch.Tensor, out: torch.Tensor | None = None):
    """y = x . w^T: x [m, k] f32, quants int32/uint32 words (n*k/4), scales [n, k/32] f32."""
    m, k = x.shape
    n = scales.shape[0]
    _need(x, torch.float32, m * k, "x")
    if quants.dtype not in (torch.int32, torch.uint32):
        raise GQError("quants: expected int32 or uint32 words")
    _need(quants, quants.dtype, n * k // 4, "quants")
    _need(scales, torch.float32, n * (k // 32), "scales")
    y = torch.empty((m, n), dtype=torch.float32, device=x.device) if out is None else out
    _need(y, torch.float32, m * n, "out")
    _check(lib().block_q8_matmul_nt(_ptr(x), _ptr(quants), _ptr(scales), _ptr(y), m, k, n, _stream()),
           "block_q8_matmul_nt")
    return y


# ----------------------------------------------------------------------------- ternary

def ternary_bitplane_gemv(P: torch.Tensor, N: torch.Tensor, X: torch.Tensor, out: torch.Tensor | None = None):
    """y [batch, rows] int32 for P, N [rows, k/32] and X [batch, k/32] bitplanes (int32/uint32)."""
    rows, kw = P.shape
    batch = X.shape[0]
    for t, nm, cnt in ((P, "P", rows * kw), (N, "N", rows * kw), (X, "X", batch * kw)):
        if t.dtype not in (torch.int32, torch.uint32):
            raise GQError(f"{nm}: expected int32 or uint32 words")
        _need(t, t.dtype, cnt, nm)
    y = torch.empty((batch, rows), dtype=torch.int32, device=P.device) if out is None else out
    _need(y, torch.int32, batch * rows, "out")
    _check(lib().ternary_bitplane_gemv(_ptr(P), _ptr(N), _ptr(X), _ptr(y), rows, kw * 32, batch, _stream()),
           "ternary_bitplane_gemv")
    return y


# ----------------------------------------------------------------------------- prefill

def quantize_q8_0(x: torch.Tensor, mma_operand: bool = False, out=None):
    """(d [m, k/32] f16 bits as int16, q [m, k] int8, operand [3, m, k] bf16 bits or None: the
    three bf16 parts of f16(d) * q that the prefill MMA path reads).  `out` = (d, q, op) reuses
    caller buffers of those shapes (op None unless mma_operand)."""
    m, k = x.shape
    _need(x, torch.float32, m * k, "x")
    if out is None:
        d = torch.empty((m, k // 32), dtype=torch.int16, device=x.device)
        q = torch.empty((m, k), dtype=torch.int8, device=x.device)
        op = torch.empty((3, m, k), dtype=torch.int16, device=x.device) if mma_operand else None
    else:
        d, q, op = out
        _need(d, torch.int16, m * (k // 32), "d")
        _need(q, torch.int8, m * k, "q")
        if mma_operand:
            _need(op, torch.int16, 3 * m * k, "op")
        else:
            op = None
    _check(lib().gq_quantize_q8_0(_ptr(x), m, k, _ptr(d), _ptr(q), _ptr(op), _stream()), "gq_quantize_q8_0")
    return d, q, op


def q1s32_q8_gemm(signs: torch.Tensor, wscale: torch.Tensor, xd: torch.Tensor, xq: torch.Tensor,
                  xq_mma: torch.Tensor | None = None, path: int = PATH_AUTO, out: torch.Tensor | None = None):
    """y [M, N] f32 for 1-bit weights (signs [N, K/32] words, wscale [N, K/32] f32) and Q8_0
    activations (xd [M, K/32] f16 bits, xq [M, K] int8, optional MMA operand [3, M, K] from
    quantize_q8_0)."""
    M, K = xq.shape
    N = signs.shape[0]
    if signs.dtype not in (torch.int32, torch.uint32):
        raise GQError("signs: expected int32 or uint32 words")
    _need(signs, signs.dtype, N * (K // 32), "signs")
    _need(wscale, torch.float32, N * (K // 32), "wscale")
    _need(xd, torch.int16, M * (K // 32), "xd")
    _need(xq, torch.int8, M * K, "xq")
    if xq_mma is not None:
        _need(xq_mma, torch.int16, 3 * M * K, "xq_mma")
    y = torch.empty((M, N), dtype=torch.float32, device=xq.device) if out is None else out
    _need(y, torch.float32, M * N, "out")
    _check(lib().q1s32_q8_gemm(_ptr(signs), _ptr(wscale), _ptr(xd), _ptr(xq), _ptr(xq_mma), _ptr(y), M, N, K,
                               path, _stream()), "q1s32_q8_gemm")
    return y


# ----------------------------------------------------------------------------- roofline probes

PROBE_KINDS = {
    "ffma": 0, "ffma2": 1, "fadd2": 2, "fadd": 3, "dp4a": 4, "lop3": 5, "popc": 6, "prmt": 7, "shf": 8,
    "imad": 9, "shfl": 10, "lds": 11, "dp4a+ffma2": 12, "lds+shfl": 13, "ffma+ffma2": 14, "lop3+dp4a": 15,
    "fadd+ffma2": 16, "lop3+ffma2": 17, "mma_sync_f16": 18, "mma_sync_bf16": 19, "mma_sync_e4m3": 20,
    "mma_sync_s8": 21, "mma_sync_f16_mix": 22, "mma_sync_e4m3_mix": 23, "lop3+popc": 24,
}
PROBE_MMA_F16, PROBE_MMA_F8, PROBE_MMA_F16_TMEM_A = 0, 1, 2


def probe_fill(buf: torch.Tensor, seed: int = 1):
    """Fill a contiguous CUDA tensor (size a multiple of 16 bytes) with a non-zero pattern."""
    nbytes = buf.numel() * buf.element_size()
    _check(lib().gq_probe_fill(_ptr(buf), nbytes, seed & 0xFFFFFFFF, _stream()), "gq_probe_fill")


def probe_read(buf: torch.Tensor, sink: torch.Tensor, blocks_per_sm: int = 2, threads: int = 1024):
    """One read-only pass over buf (XOR of everything read folded into the int32 sink)."""
    _need(sink, torch.int32, 1, "sink")
    nbytes = buf.numel() * buf.element_size()
    _check(lib().gq_probe_read(_ptr(buf), nbytes, _ptr(sink), blocks_per_sm, threads, _stream()), "gq_probe_read")


def probe_issue(kind: str, iters: int = 2000):
    """Warp instructions per SM per cycle for one instruction kind (median over the SMs)."""
    L = lib()
    sms = L.gq_probe_sm_count()
    if sms <= 0:
        raise GQError("probe_issue: no device")
    cyc = torch.zeros(sms, dtype=torch.int64, device="cuda")
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    k = PROBE_KINDS[kind]
    _check(L.gq_probe_issue(k, iters, _ptr(cyc), _ptr(sink), _stream()), "gq_probe_issue")
    c = cyc.cpu().double()
    return L.gq_probe_issue_insts(k, iters) / float(c.median())


def probe_mma(kind: int, n: int, iters: int = 2000):
    """Dense MMA flops per SM per cycle (median over the SMs) for M = 128, N = n."""
    L = lib()
    sms = L.gq_probe_sm_count()
    cyc = torch.zeros(sms, dtype=torch.int64, device="cuda")
    _check(L.gq_probe_mma(kind, n, iters, _ptr(cyc), _stream()), "gq_probe_mma")
    c = float(cyc.cpu().double().median())
    k = 32 if kind == PROBE_MMA_F8 else 16
    return 2.0 * 128 * n * k * iters / c, c / iters
