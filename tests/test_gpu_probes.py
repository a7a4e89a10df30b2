"""The roofline probes the bench quotes its fractions against (csrc/probes.cu).

The read probe is pinned exactly: the fill pattern is a fixed function of the item index, so the
XOR of every word of the buffer is known on the host, and the probe's XOR-reduced sink must equal
it -- every 16-byte item read once, none missed, none read twice (a second read would cancel).
The issue and MMA probes are timing instruments; here they must run, return rates inside what an
SM can issue, and leave the device error word clear."""
import numpy as np
import pytest

from tests.gpu_util import need_gpu

pytestmark = pytest.mark.gpu


def _host_xor(n16: int, seed: int) -> int:
    """XOR over the buffer gq_probe_fill writes: item i holds h|1, (h^0xA5A5A5A5)|1, (3h)|1 and
    (h+0x01234567)|1 with h = i * 0x9E3779B1 + seed, all modulo 2^32."""
    i = np.arange(n16, dtype=np.uint64).astype(np.uint32)
    h = i * np.uint32(0x9E3779B1) + np.uint32(seed)
    w = (h | np.uint32(1)) ^ ((h ^ np.uint32(0xA5A5A5A5)) | np.uint32(1)) ^ \
        ((h * np.uint32(3)) | np.uint32(1)) ^ ((h + np.uint32(0x01234567)) | np.uint32(1))
    return int(np.bitwise_xor.reduce(w))


@pytest.mark.parametrize("n16,blocks_per_sm,threads", [(4 * 1024 * 1024 + 7, 2, 1024), (1000003, 1, 256),
                                                      (16, 4, 512), (1, 1, 32)])
def test_read_probe_reads_every_item_once(n16, blocks_per_sm, threads):
    gq = need_gpu()
    import torch
    buf = torch.empty(n16 * 16, dtype=torch.uint8, device="cuda")
    gq.probe_fill(buf, seed=7)
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    gq.probe_read(buf, sink, blocks_per_sm=blocks_per_sm, threads=threads)
    torch.cuda.synchronize()
    assert (int(sink.item()) & 0xFFFFFFFF) == _host_xor(n16, 7)


def test_host_xor_matches_a_direct_fill():
    """The host formula against the device fill itself, word by word, on a small buffer."""
    gq = need_gpu()
    import torch
    n16 = 4099
    buf = torch.empty(n16 * 16, dtype=torch.uint8, device="cuda")
    gq.probe_fill(buf, seed=12345)
    words = buf.cpu().numpy().view(np.uint32).reshape(n16, 4)
    i = np.arange(n16, dtype=np.uint64).astype(np.uint32)
    h = i * np.uint32(0x9E3779B1) + np.uint32(12345)
    assert np.array_equal(words[:, 0], h | np.uint32(1))
    assert np.array_equal(words[:, 1], (h ^ np.uint32(0xA5A5A5A5)) | np.uint32(1))
    assert np.array_equal(words[:, 2], (h * np.uint32(3)) | np.uint32(1))
    assert np.array_equal(words[:, 3], (h + np.uint32(0x01234567)) | np.uint32(1))


def test_issue_probes_run_within_the_issue_limit():
    gq = need_gpu()
    for kind in gq.PROBE_KINDS:
        rate = gq.probe_issue(kind, 200)
        # four SMSPs, one warp instruction each per cycle at most
        assert 0.0 < rate <= 4.05, (kind, rate)
    assert gq.device_error() == 0


@pytest.mark.parametrize("kind", [0, 1, 2])
def test_mma_probes_run(kind):
    gq = need_gpu()
    flop_per_cycle, cycles_per_mma = gq.probe_mma(kind, 128, 200)
    # a 128 x 128 x K MMA per SM: dense bf16 is ~8 K flop per SM-cycle, e4m3 twice that
    assert 1000.0 < flop_per_cycle < 40000.0, (kind, flop_per_cycle)
    assert cycles_per_mma > 0.0
    assert gq.device_error() == 0
