"""Host-side logic of the multi-rank bench path, on CPU with gloo (world size 2).

The product path does not shard across GPUs (replicas only): each rank runs
the same workload on its own GPU, the timed region is bracketed by barriers,
and the elapsed time is the maximum over ranks. These tests run that logic on
CPU processes: the rank environment, the max-over-ranks reduction, the
barrier, and the reference arm's rule that only rank 0 works and prints.
"""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        bench.barrier(ws)
        # rank-dependent elapsed times: the job time is the slowest rank's
        got = bench.max_over_ranks(1.5 + rank, ws)
        bench.barrier(ws)
        q.put((rank, ws, r, local, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, (r0, ws, r, local, got) in enumerate(res):
        assert (r0, ws, r, local) == (rank, 2, rank, rank)
        assert got == 2.5  # max(1.5, 2.5) on every rank


def test_single_rank_identity(monkeypatch):
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.max_over_ranks(3.25, 1) == 3.25
    bench.barrier(1)  # no process group needed at world size 1


def test_reference_arm_only_rank0_works(monkeypatch, capsys):
    import argparse
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    args = argparse.Namespace(gpus=2, steps=1, warmup=1)
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""  # rank 1 prints nothing and does no work
