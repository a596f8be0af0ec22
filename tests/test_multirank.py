"""The benchmark's multi-rank host logic on CPU: two gloo ranks (world size 2,
127.0.0.1 rendezvous).  The decode does not shard, so N GPUs run N
independent replicas; what N > 1 adds is the slowest-rank timing, the
whole-job rate and rank 0 alone reporting (and the reference arm running on
rank 0 only)."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, times, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(times[rank], dist, "cpu")
        dist.barrier()
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_job_time_on_every_rank():
    world, times = 2, [12.5, 40.25]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = dict(q.get(timeout=10) for _ in range(world))
    assert res == {0: 40.25, 1: 40.25}


def test_whole_job_rate_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    # 2 replicas x 64 tokens per step, 100 steps, slowest rank 20 ms in total
    assert bench.whole_job_rate(2, 64, 100, 20.0) == pytest.approx(2 * 64 / (0.020 / 100))
    assert bench.whole_job_rate(1, 64, 100, 20.0) == pytest.approx(64 / (0.020 / 100))
    assert bench.max_over_ranks(3.5) == 3.5          # one process: no reduction


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        steps, warmup, gpus = 1, 0, 2

    monkeypatch.setenv("RANK", "1")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(Args(), None)
    assert buf.getvalue() == ""                      # rank 1: no work, no line
