"""The benchmark's multi-replica bookkeeping on CPU (gloo, world size 2).

With N GPUs the layer runs as N independent replicas (it has no exchange step); the
benchmark takes the slowest rank's time and reports the blocks of all ranks over it.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slow = bench.max_over_ranks(1.5 + rank, world)  # rank 1 is the slow one
        bench.barrier(world)
        q.put((rank, slow, bench.whole_job_rate(100, world, slow)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, slow, rate in got:
        assert slow == pytest.approx(2.5)            # every rank sees the slowest time
        assert rate == pytest.approx(100 * 2 / 2.5)  # blocks of both ranks / slowest time


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.whole_job_rate(10, 1, 2.0) == 5.0


def test_reference_arm_runs_on_rank0_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert capsys.readouterr().out == ""


def test_reference_arm_line_on_rank0(monkeypatch, capsys):
    """The reference arm (the CPU oracle, timed on bounded samples) prints one JSON line
    with the contract's keys, its cpu_baseline and e2e describing the same run."""
    import json
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
