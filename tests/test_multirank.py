"""The bench's replica mode (N > 1) on CPU: world_size 2 over gloo.

The layer runs as independent replicas, one per GPU, with no data-path collective; what the ranks
share is the timing protocol (a barrier on both sides of the timed region, the slowest rank's time,
all ranks' work over it) and the reference arm's rule that rank 0 alone runs and prints.  Both are
host logic and run here without a GPU.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        local_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        job_ms = bench.max_over_ranks(local_ms, dist, "cpu")
        rate = bench.whole_job_rate(world, 1000.0, job_ms)
        dist.barrier()
        out.put((rank, job_ms, rate))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, job_ms, rate in res:
        assert job_ms == 15.0  # every rank sees the slowest rank's time
        assert rate == pytest.approx(world * 1000.0 / 15e-3)  # all ranks' units over that time


def test_max_over_ranks_without_a_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.whole_job_rate(1, 10.0, 2.0) == pytest.approx(5000.0)


def test_reference_arm_under_torchrun_prints_once():
    """`bench.py --impl reference` launched as two ranks: rank 0 times the oracle and prints one line,
    rank 1 exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "tiny"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
