"""bench.py's multi-rank logic on CPU: two gloo ranks (one process each, as
under torchrun) agree on the slowest rank's time, the job throughput counts
the work of every rank, and the reference arm runs on rank 0 only."""
import io
import os
import socket
import sys
import contextlib

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(100.0 + 25.0 * rank)
        out.put((rank, slowest))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 125.0, 1: 125.0}


def test_max_over_ranks_without_group():
    assert not dist.is_initialized()
    assert bench.max_over_ranks(3.5) == 3.5


def test_job_tflops_counts_every_rank():
    ff = 1e12                      # forward flop of one step on one rank
    one = bench.job_tflops(ff, steps=2, world=1, ms=1000.0)
    assert one == pytest.approx(3.5 * ff * 2 / 1.0 / 1e12)
    # weak scaling: N ranks doing the same work in the same time = N times the throughput
    assert bench.job_tflops(ff, steps=2, world=4, ms=1000.0) == pytest.approx(4 * one)


def test_reference_arm_runs_on_rank0_only(monkeypatch):
    called = []
    monkeypatch.setattr(bench, "cpu_oracle", lambda *a, **k: called.append(1))
    monkeypatch.setenv("RANK", "1")
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(bench.parse(["--impl", "reference", "--gpus", "2"]))
    assert called == [] and buf.getvalue() == ""
