"""bench.py's N > 1 path on CPU with the gloo backend.  The step does not
shard (replicas only: one process per GPU, each with its own model and no
collective on the data path); the ranks meet only to time the job: the job's
time is the slowest rank's, its value counts every rank's rows, and the
reference arm (the oracle) runs on rank 0 alone."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", init_method="env://")
    w, r, _ = bench.dist_env()
    local = 10.0 + 5.0 * r  # rank 1 is the slower one
    t = bench.max_over_ranks(local, w)
    rate = bench.whole_job_rate(512 * 3, w, t)
    dist.barrier()
    dist.destroy_process_group()
    q.put((r, w, t, rate))


def test_job_time_is_the_slowest_rank_and_value_counts_every_rank():
    import multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    ps = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for r, w, t, rate in got:
        assert w == 2 and t == 15.0
        assert rate == pytest.approx(512 * 3 * 2 / 15.0)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.whole_job_rate(100, 1, 2.0) == 50.0


def test_reference_arm_under_torchrun_prints_one_line_from_rank_zero():
    """The driver's launch of the reference arm at N = 2: rank 0 times the
    oracle and prints one line; rank 1 exits 0 without work."""
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
