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
