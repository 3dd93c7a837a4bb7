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


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` at world size 1: one JSON line with the
    contract's keys, the oracle timed on host cores, no device bytes moved."""
    import json
    import subprocess
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "3",
                        "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1
    assert (d["steps"], d["warmup"]) == (3, 3)
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert "workload" in d["config"]
    # value is weight bytes per second: bytes per step / seconds per step
    assert abs(d["value"] - d["config"]["weight_bytes_per_step"] / (d["ms_per_step"] * 1e6)) \
        < 1e-6 * d["value"]
