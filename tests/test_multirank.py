"""The N > 1 host path of bench.py on CPU, world size 2 over gloo.

Verification shards by sequence with no collective on the data path
(replicas): each rank verifies its own batches, the step time of the job is
the slowest rank's, and rank 0 alone prints.  These tests run the helpers
bench.py uses for that under a real two-process gloo group, and the
reference arm under torchrun.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _ranks_body(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        step_ms = [7.5, 9.25][rank]  # rank 1 is the slowest
        slowest = bench.max_over_ranks(step_ms, "cpu")
        out[rank] = (slowest, bench.replica_seed(0, rank))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_step_time():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_ranks_body, args=(world, _free_port(), out), nprocs=world, join=True)
        got = dict(out)
    assert got[0][0] == got[1][0] == 9.25          # every rank sees the maximum
    assert got[0][1] != got[1][1]                   # each rank draws its own batches


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.replica_seed(5, 0) == 5


def test_job_rate_counts_every_rank():
    import bench
    # 2 ranks x 10 steps x 1456 positions in 10 ms of the slowest rank
    assert bench.job_rate(2, 10, 1456, 10.0) == pytest.approx(2 * 10 * 1456 / 0.010)
    assert bench.job_rate(1, 10, 1456, 10.0) * 2 == bench.job_rate(2, 10, 1456, 10.0)


def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
