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


def test_reference_arm_json_contract():
    """`bench.py --impl reference` (the oracle on the host cores) prints one JSON
    line with the benchmark contract's keys, on a small workload."""
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--seqlen", "2048", "--heads", "2", "--steps", "1", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "TFLOP/s"
    assert d["higher_is_better"] is True and d["steps"] == 1 and d["warmup"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["S"] == 2048 and d["config"]["H"] == 2


def test_traffic_counters_only_for_the_captured_workload(monkeypatch):
    """roofline.traffic comes from committed ncu counters: reported for the
    workloads and kernel code they were taken on, null for anything else."""
    import json
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        stored = json.load(f)["bwd_main"]
    entries = stored if isinstance(stored, list) else [stored]
    h = entries[0]["source_hash"]
    assert all(e["source_hash"] == h for e in entries)
    monkeypatch.setattr(bench, "source_hash", lambda: h)
    default = bench.traffic_workload(bench.parse([]))
    captured = {e["workload"] for e in entries}
    assert default in captured
    for e in entries:
        assert bench.ncu_traffic("bwd_main", e["workload"]) == e["bytes_per_launch_full"]
    for flags in (["--causal"], ["--deterministic"], ["--dtype", "f16"], ["--head-dim", "64"],
                  ["--seqlen", "65536"]):
        w = bench.traffic_workload(bench.parse(flags))
        assert w != default
        if w not in captured:
            assert bench.ncu_traffic("bwd_main", w) is None, flags
    monkeypatch.setattr(bench, "source_hash", lambda: "0" * 16)
    assert bench.ncu_traffic("bwd_main", default) is None
