"""Multi-rank host logic of bench.py, on the CPU with two gloo ranks.

The benchmark runs one replica of the product per GPU (the path has no exchange
step).  What the ranks share is host logic: the environment they are launched
with, the timing taken as the slowest rank's, the whole-job value over all
ranks, and the reference arm printing on rank 0 only.
"""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def worker(rank, world, port, results):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        t = bench.max_over_ranks(1.0 + rank, dist)          # rank r took 1 + r seconds
        value = bench.whole_job_gbs(1_000_000_000, 10, w, t)
        results[rank] = {"env": (r, w, local), "t": t, "value": value}
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world, port = 2, free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(worker, args=(world, port, results), nprocs=world, join=True)
        res = dict(results)
    for rank in range(world):
        assert res[rank]["env"] == (rank, world, rank)
        assert res[rank]["t"] == 2.0                         # the max over ranks, on every rank
        assert res[rank]["value"] == pytest.approx(1e9 * 10 * 2 / 2.0 / 1e9)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(0.25, None) == 0.25
    assert bench.whole_job_gbs(2_000_000_000, 1, 1, 1.0) == pytest.approx(2.0)


def test_reference_arm_prints_on_rank_zero_only():
    class Args:
        steps, warmup, cpu_seconds, gpus = 5, 3, 0.2, 2
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(Args, 1, 2)                       # rank 1: no work, no output
    assert buf.getvalue() == ""
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(Args, 0, 2)
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    # exactly the requested steps: W untimed, K timed, each a bounded sample of the workload
    assert line["steps"] == 5 and line["warmup"] == 3
    assert line["cpu_baseline"]["sample"].startswith("5 timed steps after 3 warm-up steps")
