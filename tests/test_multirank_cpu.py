"""The bench's multi-rank logic on the CPU (two gloo ranks, no GPU): every
rank gets the slowest rank's timings, the whole-job value counts every rank's
work over that time, and the reference arm runs on rank 0 only."""
import contextlib
import io
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [1.0 + rank, 5.0 - rank, 0.25 * (rank + 1)]
        got = bench.max_over_ranks(mine, world, device="cpu")
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in (0, 1):
        assert results[rank] == [2.0, 5.0, 0.5]


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks([3.0, 1.5], 1) == [3.0, 1.5]


def test_job_value_counts_every_rank():
    # 2 ranks, 1e12 FLOP each, slowest rank 1 ms -> 2000 TFLOP/s for the job
    assert bench.job_tflops(1e12, 2, 1.0) == pytest.approx(2000.0)
    assert bench.job_tflops(1e12, 1, 1.0) == pytest.approx(1000.0)


def test_reference_arm_runs_on_rank_0_only():
    class Args:
        reference_rows = 4
        warmup = 0
        steps = 1
        gpus = 2
    w = bench.headline_workload("two_shard_256")
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        bench.run_reference(Args(), w, rank=1, world=2)
    assert out.getvalue() == ""
