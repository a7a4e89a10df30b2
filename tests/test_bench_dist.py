"""The multi-GPU bench path is replicas only (no exchange step on the path): each rank times its
own sweep, the job reports total bytes over the slowest rank's time, and only rank 0 prints.
These check that host-side logic with two gloo ranks on the CPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(0.25 + rank * 0.5, dist, "cpu")   # rank 1 is the slow one
        dist.barrier()
        q.put((rank, t, bench.whole_job_rate(world, 1000, 10, t)))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_and_weak_rate():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, rate in got:
        assert t == 0.75                                   # both ranks see the slowest time
        assert rate == pytest.approx(2 * 1000 * 10 / 0.75 / 1e9)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.5, None, "cpu") == 1.5


def test_reference_arm_prints_on_rank_zero_only(tmp_path):
    """Under torchrun only rank 0 runs the reference arm; another rank exits 0 without output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_reference_arm_line():
    """Rank 0's reference arm: the oracle timed on the host cores, one JSON line with the contract's keys."""
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--ref-step-seconds", "0.2"], env=env, capture_output=True, text=True,
                       timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "higher_is_better", "cpu_baseline", "e2e"):
        assert key in line
    assert line["value"] > 0 and line["e2e"]["h2d_bytes_per_step"] == 0


def test_parallel_cpu_baseline():
    """The parallel CPU baseline runs the unchanged oracle in spawned processes started together and
    reports all their bytes over the slowest one's time."""
    sys.path.insert(0, ROOT)
    import bench
    r = bench.cpu_baseline_parallel(budget_s=0.5)
    assert r["kind"] == "oracle" and r["unit"] == "GB/s"
    assert r["cores"] == max(1, min(os.cpu_count() or 1, 64))
    assert r["value"] > 0 and r["seconds"] >= 0.5
    assert str(r["cores"]) in r["sample"]


def test_recorded_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    """The DRAM-traffic figure in the bench line comes from the committed record only while the
    GEMV's sources hash to the value stored with it; any other hash gives null."""
    sys.path.insert(0, ROOT)
    import bench
    current = bench.kernel_hash(*bench.GEMV_SOURCES)
    assert len(current) == 16
    rec = tmp_path / "profiles"
    rec.mkdir()
    (rec / "t.json").write_text(json.dumps({"kernel_source_hash": current, "dram_bytes_per_launch": 123}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("t.json", current) == 123
    assert bench.recorded_traffic("t.json", "0" * 16) is None
    assert bench.recorded_traffic("missing.json", current) is None

