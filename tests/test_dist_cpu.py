"""The bench's multi-rank path on CPU: two gloo ranks.

With N ranks every rank runs an independent replica (token data
parallelism does not shard the expert bytes); the job's time is the
slowest rank's and the value counts every rank's units.  The reference arm
runs on rank 0 only; the other ranks exit at once without printing.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    import torch.distributed as dist

    import bench
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, loc = bench.dist_env()
    slow = bench.max_over_ranks(times[rank], w, "cpu")
    dist.barrier()
    out.put((r, w, loc, slow, bench.whole_job_rate(16 * 100, slow, w)))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_max_over_ranks_and_whole_job_rate(world):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    times = [0.5 + 0.25 * r for r in range(world)]
    port = free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, times, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    slow = max(times)
    for r, (rank, w, loc, got_slow, rate) in enumerate(res):
        assert (rank, w, loc) == (r, world, r)
        assert got_slow == slow
        assert rate == pytest.approx(16 * 100 * world / slow)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(1.25, 1, "cpu") == 1.25
    assert bench.whole_job_rate(160, 2.0, 1) == 80.0


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
