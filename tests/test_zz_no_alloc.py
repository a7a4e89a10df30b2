"""q1_q8_gemv_noalloc: the decode GEMV for callers that cannot allocate device memory (it takes its
workspace from scratch memory built into the library).  Called directly through the C ABI and
checked against q1_q8_gemv, bit for bit, on calls in a row with different inputs, so whatever one
call left in the shared scratch cannot leak into the next result.  The first two shapes have at
least as many 128-row tiles as the GPU has SMs, so they take the two-launch path whose constants
and tile counter live in the scratch array (n = 16384, the largest accepted, then a smaller n);
the last takes the one-launch path that needs no scratch.  Collected last (file name) so that a
run stopping at the first failure has run everything else."""
import ctypes

import numpy as np
import pytest

import workloads as wl
from tests.gpu_util import need_gpu, to_dev

pytestmark = pytest.mark.gpu


def test_noalloc_matches_gemv_calls_in_a_row():
    gq = need_gpu()
    import torch
    L = gq.lib()
    sms = L.gq_probe_sm_count()
    assert sms > 0
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    big = 128 * sms
    cases = [(big + 300, 16384, 31), (big + 77, 2560, 32), (1000, 6912, 33)]
    for rows, n, seed in cases:
        tiles = (rows + 127) // 128
        assert (tiles >= sms) == (rows > big - 128)       # the scratch path for the first two
        rng = wl.Rng(seed)
        w = wl.q1_0_weights(rng, rows, n, scales="page")
        a = wl.q8_0_acts(rng, 1, n, quants="page")
        packed = gq.q1_0_pack(to_dev(w), rows, n)
        act = to_dev(a)
        y_ref = gq.q1_q8_gemv(packed, act, rows, n)
        y = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
        st = L.q1_q8_gemv_noalloc(ctypes.c_void_p(packed.data_ptr()), ctypes.c_void_p(act.data_ptr()),
                                  ctypes.c_void_p(y.data_ptr()), rows, n, stream)
        assert st == 0, L.gq_status_string(st)
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy().view(np.uint32), y_ref.cpu().numpy().view(np.uint32)), (rows, n)
    assert gq.device_error() == 0


def test_noalloc_rejects_oversize():
    gq = need_gpu()
    L = gq.lib()
    X = ctypes.c_void_p(0x1000)
    assert L.q1_q8_gemv_noalloc(X, X, X, 16, 16384 + 128, ctypes.c_void_p(0)) == 1
