"""Host logic of bench.py under torch.distributed, as two gloo ranks on the CPU.

With several ranks the job's time is the maximum over ranks and only rank 0
prints; the ranks split one batch (dp) unless replicas are asked for.  These tests run that logic without a GPU.
"""

from __future__ import annotations

import os
import socket
import sys
from pathlib import Path

import pytest
import torch
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parents[1]


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, str(ROOT))
    import bench
    ctx = bench.DistCtx(torch)
    try:
        assert ctx.world == world and ctx.rank == rank
        ctx.barrier()
        mx = ctx.max(1.5 + rank)          # per-rank "time"; the job takes the slowest
        out.put((rank, mx))
        ctx.barrier()
    finally:
        ctx.close()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    world, port = 2, _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=10) for _ in range(world))
    assert got == [(0, 2.5), (1, 2.5)]


def test_reference_arm_idle_on_other_ranks(monkeypatch):
    """Under torchrun the oracle baseline runs on rank 0 only; other ranks return at once."""
    sys.path.insert(0, str(ROOT))
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        workload = bench.DEFAULT_WORKLOAD
        steps, warmup = 3, 3

    def boom(*a, **k):
        raise AssertionError("rank 1 must not run the oracle")

    monkeypatch.setattr(bench, "time_oracle", boom)
    monkeypatch.setattr(bench, "oracle_step", boom)
    assert bench.run_reference(Args()) == {}


def test_single_process_context():
    sys.path.insert(0, str(ROOT))
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(k, None)
    ctx = bench.DistCtx(torch)
    assert ctx.world == 1 and ctx.rank == 0
    assert ctx.max(3.25) == 3.25
    ctx.barrier()
    ctx.close()


if __name__ == "__main__":
    sys.exit(pytest.main([__file__, "-q"]))


def test_parallelism_choice():
    """Several ranks split one batch (dp) unless replicas are asked for; one GPU
    runs the fused step, and dp on one rank is refused."""
    sys.path.insert(0, str(ROOT))
    import bench
    assert bench.parallelism_of("auto", 1) == "replicas"
    assert bench.parallelism_of("auto", 4) == "dp"
    assert bench.parallelism_of("replicas", 8) == "replicas"
    assert bench.parallelism_of("dp", 2) == "dp"
    with pytest.raises(SystemExit):
        bench.parallelism_of("dp", 1)
