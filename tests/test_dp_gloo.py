"""Host logic of the data-parallel statistics (moe_expert_routing_router_gb300.dp)
as two gloo ranks on the CPU: the all-gather of every rank's counts, P and
token count, in rank order, and the gradient coefficient's rescaling.  The
combine itself is a kernel (tests/test_gpu_dp.py)."""

from __future__ import annotations

import os
import socket
import sys
from pathlib import Path

import numpy as np
import torch
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parents[1]
E = 12


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _shard(rank: int):
    rng = np.random.default_rng(100 + rank)
    counts = rng.integers(0, 50, size=E).astype(np.int32)
    P = rng.random(E).astype(np.float32)
    return counts, P, 1000 + 37 * rank


def _rank_main(rank: int, world: int, port: int, out) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, str(ROOT))
    import torch.distributed as dist
    from moe_expert_routing_router_gb300 import dp
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        counts, P, T = _shard(rank)
        c_all, p_all, t_all = dp.gather_shard_stats(torch.from_numpy(counts), torch.from_numpy(P), T)
        out.put((rank, c_all.numpy(), p_all.numpy(), t_all))
    finally:
        dist.destroy_process_group()


def test_gather_shard_stats_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    world, port = 2, _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    want = [_shard(r) for r in range(world)]
    for rank, c_all, p_all, t_all in got:
        assert c_all.shape == (world, E) and c_all.dtype == np.int32
        for r in range(world):
            assert np.array_equal(c_all[r], want[r][0])
            assert np.array_equal(p_all[r].view(np.uint32), want[r][1].view(np.uint32))
        assert t_all == [want[r][2] for r in range(world)]


def test_shard_grad_scale():
    sys.path.insert(0, str(ROOT))
    from moe_expert_routing_router_gb300 import dp
    # alpha*E/T_local * g * T_local/T_total = alpha*E/T_total * g
    assert dp.shard_grad_scale(2.0, 300, 1200) == 0.5
    assert dp.shard_grad_scale(1.0, 4096, 4096) == 1.0
