"""Multi-rank host logic of bench.py on CPU: two gloo ranks (world size 2).

The path has no exchange step, so N GPUs run N independent replicas; what
needs checking across processes is the harness: process-group set-up, the
barrier, the maximum over ranks, the whole-job rate (all ranks' units over
the slowest rank's time), and that only rank 0 prints under torchrun.
No GPU is used.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    r, w, local = bench.dist_setup()
    try:
        assert (r, w, local) == (rank, world, rank)
        assert dist.get_backend() == "gloo"
        bench.barrier(w)
        # each rank's own number; every rank sees the largest
        mx = bench.max_over_ranks(1.5 + rank, w)
        # rank r took (r + 1) seconds for 10 units: the job did 10 * w units
        # in the slowest rank's w seconds
        rate = bench.whole_job_rate(10.0, float(rank + 1), w)
        results[rank] = (mx, rate)
    finally:
        dist.destroy_process_group()


def test_gloo_two_ranks_max_and_rate():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_rank_main, args=(world, free_port(), results), nprocs=world, join=True,
                           start_method="spawn")
        got = dict(results)
    assert sorted(got) == [0, 1]
    for rank in range(world):
        mx, rate = got[rank]
        assert mx == 2.5
        assert rate == pytest.approx(10.0 * world / world)  # 20 units over the slowest rank's 2 s


def test_single_rank_rate_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.whole_job_rate(32 * 5, 0.5, 1) == pytest.approx(320.0)


def test_reference_arm_under_torchrun_prints_once():
    """`bench.py --impl reference` launched as the driver launches N > 1:
    rank 0 alone times the oracle and prints one JSON line; the other rank
    exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--cpu-seconds", "0.1"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
