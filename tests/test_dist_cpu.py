"""The multi-rank paths of bench.py on CPU with the gloo backend, world size 2.

The hot path shards without any exchange (replicas over heads and sequences),
so the only collective is the timing reduction: every rank times its own
steps, the job takes the slowest rank's time, and rank 0 alone prints the
whole-job line.  The reference arm (the oracle on host cores) runs on rank 0
only; the other ranks exit 0 without work."""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        got = bench.max_over_ranks(dist, times[rank], "cpu")
        out[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_timing_reduction_takes_the_slowest_rank():
    world, port = 2, _free_port()
    times = [12.5, 17.25]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, times, out), nprocs=world, join=True)
        got = dict(out)
    assert got == {0: 17.25, 1: 17.25}


def test_whole_job_value_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    # 2 replicas, 3 steps of 1e12 FLOP each per rank, slowest rank 1.5 s
    assert bench.whole_job_tflops(2, 1e12, 3, 1500.0) == pytest.approx(4.0)
    assert bench.max_over_ranks(None, 3.0, "cpu") == 3.0


def test_reference_arm_prints_once_under_torchrun():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--config", "1", "--steps", "1", "--warmup", "0",
           "--cpu-seconds", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0
