"""Multi-rank plumbing of bench.py on CPU (gloo, world size 2): the timed
region's max over ranks, and the reference arm running on rank 0 only. The
linear and accept calls are single-GPU operations, so several GPUs run
independent replicas; these are the only cross-rank steps."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank's local time differs; every rank must end with the largest
        out[rank] = bench.max_over_ranks(10.0 + 3.5 * rank, world, "cpu")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()  # one rendezvous port for both ranks
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        assert dict(out) == {0: 13.5, 1: 13.5}


def test_max_over_ranks_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(4.25, 1, "cpu") == 4.25


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench

    calls = []
    monkeypatch.setattr(bench, "cpu_baseline_sample", lambda **kw: calls.append(kw) or {"value": 1.0})
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    class A:
        steps, warmup, cpu_cols = 2, 1, 8

    bench.run_reference(A())
    assert calls == [] and capsys.readouterr().out == ""
