"""The C-ABI library without a GPU: it loads, exports every entry point include/gq.h declares, and
rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gq.h")


@pytest.fixture(scope="module")
def L():
    from gemm_q1_q8_gb300 import build
    build.build()
    import gemm_q1_q8_gb300 as gq
    L = gq.lib()
    return L


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "sizeof")))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("q1_q8_gemv", "q1_q8_gemm", "block_q8_matmul_nt", "ternary_bitplane_gemv",
                 "gq_q1_0_pack", "q1_q8_gemv_grouped", "gq_quantize_q8_0", "q1s32_q8_gemm", "q1_q8_gemv_raw",
                 "gq_pack_q8_0"):
        assert must in names


def test_library_exports_every_declared_symbol(L):
    from gemm_q1_q8_gb300 import build
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True, check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing


def test_version_and_status_strings(L):
    assert L.gq_version().decode().startswith("gq ")
    assert L.gq_status_string(0).decode() == "ok"
    assert "shape" in L.gq_status_string(1).decode()


N = ctypes.c_void_p(0)
X = ctypes.c_void_p(0x1000)     # never dereferenced: validation fails first


@pytest.mark.parametrize("call,expect", [
    (lambda L: L.q1_q8_gemv(X, X, X, 0, 1024, X, N), 1),
    (lambda L: L.q1_q8_gemv(X, X, X, 16, 1000, X, N), 1),
    (lambda L: L.q1_q8_gemv(X, X, X, 16, (1 << 20) + 128, X, N), 1),
    (lambda L: L.q1_q8_gemv(N, X, X, 16, 1024, X, N), 2),
    (lambda L: L.q1_q8_gemv(ctypes.c_void_p(0x1008), X, X, 16, 1024, X, N), 2),
    (lambda L: L.q1_q8_gemv(X, ctypes.c_void_p(0x1001), X, 16, 1024, X, N), 2),
    (lambda L: L.q1_q8_gemv(X, X, X, 16, 1024, N, N), 2),
    (lambda L: L.q1_q8_gemv(X, X, X, 16, 1024, ctypes.c_void_p(0x1004), N), 2),
    (lambda L: L.q1_q8_gemm(X, X, X, 16, 1024, 0, 0, N), 1),
    (lambda L: L.q1_q8_gemm(X, X, X, 16, 1024, 4, 3, N), 3),
    (lambda L: L.q1_q8_gemm(X, X, X, 16, 1024, 4, 9, N), 3),
    (lambda L: L.block_q8_matmul_nt(X, X, X, X, 1, 48, 8, N), 1),
    (lambda L: L.block_q8_matmul_nt(X, ctypes.c_void_p(0x1004), X, X, 1, 64, 8, N), 2),
    (lambda L: L.ternary_bitplane_gemv(X, X, X, X, 8, 1000, 1, N), 1),
    (lambda L: L.ternary_bitplane_gemv(X, X, X, X, 8, 1024, 65, N), 1),
    (lambda L: L.ternary_bitplane_gemv(X, N, X, X, 8, 1024, 1, N), 2),
    (lambda L: L.gq_quantize_q8_0(X, 1, 33, X, X, N, N), 1),
    (lambda L: L.gq_quantize_q8_0(X, 1, 64, X, N, N, N), 2),
    (lambda L: L.q1s32_q8_gemm(X, X, X, X, N, X, 8, 8, 96, 2, N), 1),
    (lambda L: L.q1s32_q8_gemm(X, X, X, X, N, X, 8, 8, 128, 1, N), 3),
    (lambda L: L.q1s32_q8_gemm(X, X, X, X, N, X, 8, 8, 128, 3, N), 2),
    (lambda L: L.q1_q8_gemv_f32(X, X, X, 16, 1000, X, N), 1),
    (lambda L: L.q1_q8_gemv_f32(X, ctypes.c_void_p(0x1008), X, 16, 1024, X, N), 2),
    (lambda L: L.q1_q8_gemv_f32(X, X, X, 16, 1024, N, N), 2),
    (lambda L: L.matvec_q8(X, X, X, X, 8, 48, N), 1),
    (lambda L: L.matmul_q8(X, X, X, X, 0, 8, 64, N), 1),
    (lambda L: L.matvec_q4g128(X, X, X, X, 0, 64, N), 1),
    (lambda L: L.matmul_q4g128(X, X, X, X, 2, 8, 65568, N), 1),
    (lambda L: L.matvec_q8(ctypes.c_void_p(0x1008), X, X, X, 8, 64, N), 2),
    (lambda L: L.matmul_q4g128(X, X, ctypes.c_void_p(0x1004), X, 3, 8, 64, N), 2),
    (lambda L: L.matvec_q4g128(X, N, X, X, 8, 64, N), 2),
    (lambda L: L.matmul_q8_mma(X, X, X, X, 4, 8, 32, X, N), 1),
    (lambda L: L.matmul_q8_mma(X, X, X, X, 4, 8, 96, N, N), 2),
    (lambda L: L.matmul_q4g128_mma(X, X, X, X, 4, 8, 128, ctypes.c_void_p(0x1008), N), 2),
    (lambda L: L.matmul_q4g128_mma(X, X, X, X, 0, 8, 128, X, N), 1),
    (lambda L: L.q1s32_f32_gemm_mma(X, X, X, X, 4, 8, 96, X, N), 1),
    (lambda L: L.q1s32_f32_gemm_mma(X, ctypes.c_void_p(0x1004), X, X, 4, 8, 128, X, N), 2),
    (lambda L: L.q1s32_f32_gemm_mma(X, X, X, X, 4, 8, 128, N, N), 2),
    (lambda L: L.q1s32_q8_gemm(X, ctypes.c_void_p(0x1004), X, X, X, X, 8, 8, 128, 3, N), 2),
    (lambda L: L.q1s32_f32_gemm(X, X, X, X, 1, 8, 48, 0, N), 1),
    (lambda L: L.q1s32_f32_gemm(X, X, X, X, 0, 8, 64, 0, N), 1),
    (lambda L: L.q1s32_f32_gemm(X, X, X, X, 1, 0, 64, 0, N), 1),
    (lambda L: L.q1s32_f32_gemm(X, X, X, X, 1, 8, 64, 1, N), 3),
    (lambda L: L.q1s32_f32_gemm(X, X, X, X, 1, 8, 64, 3, N), 3),
    (lambda L: L.q1s32_f32_gemm(X, N, X, X, 1, 8, 64, 0, N), 2),
    (lambda L: L.q1s32_f32_gemm(X, X, ctypes.c_void_p(0x1008), X, 1, 8, 64, 2, N), 2),
    (lambda L: L.q1s32_f32_gemm(X, X, X, ctypes.c_void_p(0x1002), 1, 8, 64, 4, N), 2),
    (lambda L: L.gq_q1_0_pack(X, 8, 100, X, N), 1),
    (lambda L: L.gq_q1_0_pack(X, 8, 128, ctypes.c_void_p(0x1004), N), 2),
    (lambda L: L.q1_q8_gemv_raw(X, X, X, 0, 1024, N), 1),
    (lambda L: L.q1_q8_gemv_raw(X, X, X, 8, 1000, N), 1),
    (lambda L: L.q1_q8_gemv_raw(ctypes.c_void_p(0x1001), X, X, 8, 1024, N), 2),
    (lambda L: L.q1_q8_gemv_raw(X, X, ctypes.c_void_p(0x1002), 8, 1024, N), 2),
    (lambda L: L.gq_pack_q8_0(X, 1, 48, X, X, N), 1),
    (lambda L: L.gq_pack_q8_0(X, 0, 64, X, X, N), 1),
    (lambda L: L.gq_pack_q8_0(X, 1, 64, N, X, N), 2),
    (lambda L: L.gq_probe_fill(X, 24, 1, N), 1),
    (lambda L: L.gq_probe_fill(ctypes.c_void_p(0x1008), 32, 1, N), 2),
    (lambda L: L.gq_probe_read(X, 4096, X, 0, 256, N), 1),
    (lambda L: L.gq_probe_read(X, 4096, X, 2, 100, N), 1),
    (lambda L: L.gq_probe_read(X, 4096, N, 2, 256, N), 2),
    (lambda L: L.gq_probe_issue(99, 10, X, X, N), 1),
    (lambda L: L.gq_probe_issue(0, 0, X, X, N), 1),
    (lambda L: L.gq_probe_issue(0, 10, ctypes.c_void_p(0x1004), X, N), 2),
    (lambda L: L.gq_probe_mma(5, 64, 10, X, N), 3),
    (lambda L: L.gq_probe_mma(0, 24, 10, X, N), 1),
    (lambda L: L.gq_probe_mma(1, 64, 10, N, N), 2),
])
def test_host_validation_rejects_without_launching(L, call, expect):
    assert call(L) == expect


def test_workspace_bytes(L):
    assert L.gq_q1_q8_workspace_bytes(2560) == 80 * 96 + 16
    assert L.gq_q1_q8_workspace_bytes(100) == 0


def test_wq_mma_workspace_bytes(L):
    assert L.gq_wq_mma_workspace_bytes(512, 4096) == 3 * 512 * 4096 * 2
    assert L.gq_wq_mma_workspace_bytes(1, 32) == 0
    assert L.gq_wq_mma_workspace_bytes(0, 64) == 0


def test_packed_bytes(L):
    assert L.gq_q1_0_packed_bytes(256, 1024) == 2 * 8 * 2304
    assert L.gq_q1_0_packed_bytes(129, 128) == 2 * 1 * 2304
    assert L.gq_q1_0_packed_bytes(1, 100) == 0


def test_group_plan_host_only(L):
    import gemm_q1_q8_gb300 as gq
    descs = (gq._Desc * 3)()
    for i, (rows, n) in enumerate([(256, 1024), (1000, 2560), (1, 128)]):
        descs[i] = gq._Desc(0x1000 * (i + 1), 0x2000, 0x3000, 0x4000, rows, n, -1, 0)
    tiles = ctypes.c_int(0)
    assert L.gq_gemv_group_plan(ctypes.cast(descs, ctypes.c_void_p), 3, ctypes.byref(tiles)) == 0
    # sorted by n descending: (1000, 2560) [8 tiles], (256, 1024) [2 tiles], (1, 128) [1 tile]
    assert [descs[i].n for i in range(3)] == [2560, 1024, 128]
    assert [descs[i].packed_w for i in range(3)] == [0x2000, 0x1000, 0x3000]
    assert [descs[i].tile_begin for i in range(3)] == [0, 8, 10]
    assert tiles.value == 11
    descs[1].n = 2500
    assert L.gq_gemv_group_plan(ctypes.cast(descs, ctypes.c_void_p), 3, ctypes.byref(tiles)) == 1


def test_group_plan_act_format(L):
    """act_format must be Q8_0 (0) or F32 (1); an f32 activation must be 16-byte aligned."""
    import gemm_q1_q8_gb300 as gq
    tiles = ctypes.c_int(0)
    for fmt, act, want in [(gq.ACT_F32, 0x2000, 0), (gq.ACT_F32, 0x2008, 2), (2, 0x2000, 1), (gq.ACT_Q8_0, 0x2002, 0)]:
        descs = (gq._Desc * 1)()
        descs[0] = gq._Desc(0x1000, act, 0x3000, 0x4000, 256, 1024, -1, fmt)
        assert L.gq_gemv_group_plan(ctypes.cast(descs, ctypes.c_void_p), 1, ctypes.byref(tiles)) == want
        if want == 0:
            assert descs[0].act_format == fmt
