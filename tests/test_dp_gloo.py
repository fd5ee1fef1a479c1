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
        known = [_shard(r)[2] for r in range(world)]
        c2, p2, t2 = dp.gather_shard_stats(torch.from_numpy(counts), torch.from_numpy(P), T, T_shard=known)
        same = (torch.equal(c2, c_all) and torch.equal(p2.view(torch.int32), p_all.view(torch.int32)) and t2 == t_all)
        try:
            dp.gather_shard_stats(torch.from_numpy(counts), torch.from_numpy(P), T, T_shard=known[::-1])
            rejected = False
        except ValueError:
            rejected = True
        out.put((rank, c_all.numpy(), p_all.numpy(), t_all, same, rejected))
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
    for rank, c_all, p_all, t_all, same, rejected in got:
        assert same and rejected
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


# Global-capacity dispatch over two gloo ranks.  The exchange and the choice of
# rank and batch size are dp's host logic; the two kernel calls are replaced by
# stand-ins built from the oracle (cap_base = the counts of the lower ranks;
# slot = cap_base + the rank-local order, dropped at the batch's capacity), so
# that a wrong rank, rank order or token count changes the slots.
E_D, K_D, CF_D = 7, 2, 0.8


def _dispatch_shard(rank: int):
    rng = np.random.default_rng(300 + rank)
    T = 90 + 41 * rank
    idx = np.stack([rng.choice(E_D, size=K_D, replace=False) for _ in range(T)]).astype(np.int32)
    return idx


def _rank_dispatch_main(rank: int, world: int, port: int, out) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, str(ROOT))
    import torch.distributed as dist
    import oracle
    from moe_expert_routing_router_gb300 import dp

    def fake_base(counts, r, out=None, stream=None):
        c = counts.numpy()
        return torch.from_numpy(c[:r].sum(axis=0).astype(np.int32))

    def fake_dispatch(idx, E, cf, T_total, base, ws=None, out=None, stream=None):
        i = idx.numpy()
        C = oracle.dispatch.capacity(int(T_total), i.shape[1], E, cf)
        local = oracle.dispatch.dispatch(i, E, 10 ** 9)["slot"]
        g = base.numpy()[i.ravel()] + local
        return {"slot": np.where(g < C, g, -1), "capacity": C}

    dp.api.moe_shard_capacity_base = fake_base
    dp.api.moe_dispatch_sharded = fake_dispatch
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        idx = _dispatch_shard(rank)
        counts = torch.from_numpy(np.bincount(idx.ravel(), minlength=E_D).astype(np.int32))
        c_all, _, T_shard = dp.gather_shard_stats(counts, torch.zeros(E_D), idx.shape[0])
        batch = {"counts_all": c_all, "rank": dist.get_rank(), "T_total": sum(T_shard)}
        got = dp.data_parallel_dispatch(torch.from_numpy(idx), batch, E_D, CF_D)
        out.put((rank, got["slot"], got["cap_base"].numpy(), got["capacity"]))
    finally:
        dist.destroy_process_group()


def test_global_capacity_dispatch_gloo():
    sys.path.insert(0, str(ROOT))
    import oracle
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    world, port = 2, _free_port()
    procs = [ctx.Process(target=_rank_dispatch_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted((q.get(timeout=120) for _ in range(world)), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    shards = [_dispatch_shard(r) for r in range(world)]
    whole_idx = np.concatenate(shards)
    C = oracle.dispatch.capacity(whole_idx.shape[0], K_D, E_D, CF_D)
    whole = oracle.dispatch.dispatch(whole_idx, E_D, C)
    assert all(g[3] == C for g in got)
    assert np.array_equal(got[0][2], np.zeros(E_D, np.int32))
    assert np.array_equal(got[1][2], np.bincount(shards[0].ravel(), minlength=E_D))
    assert np.array_equal(np.concatenate([g[1] for g in got]), whole["slot"])
    assert (whole["slot"] < 0).any() and (whole["slot"] >= 0).any()    # the capacity binds


# A rank with no rows of the batch (a ragged split): it must still take part in
# the exchange, so that the other rank's collectives complete, and return empty
# per-row outputs; the batch's statistics and capacity are those of the rows
# that exist.  The kernel calls are stand-ins built from the oracle, and each
# records that it ran, so that the empty rank is seen to launch none of them.
E_Z, K_Z, CF_Z, T_Z = 6, 2, 1.0, 40


def _rank_empty_main(rank: int, world: int, port: int, out) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, str(ROOT))
    import torch.distributed as dist
    import oracle
    from moe_expert_routing_router_gb300 import dp
    ran = []

    def fake_fwd(logits, k, alpha, renorm=-1, n_ranks=0, ws=None, stream=None):
        ran.append("fwd")
        fw = oracle.router.router_forward(logits.numpy(), "fp32", k, alpha)
        return {"idx": torch.from_numpy(fw["idx"].astype(np.int32)), "gate": torch.from_numpy(fw["gate"]),
                "counts": torch.from_numpy(fw["counts"].astype(np.int32)),
                "P": torch.from_numpy(fw["P"].astype(np.float32))}

    def fake_combine(c_all, p_all, T_shard, k, alpha, n_ranks=0, stream=None):
        T = sum(T_shard)
        counts = c_all.numpy().sum(axis=0)
        P = (p_all.numpy().astype(np.float64) * np.asarray(T_shard, np.float64)[:, None]).sum(axis=0) / T
        return {"counts": counts, "P": P, "f": torch.from_numpy((counts / (T * k)).astype(np.float32))}

    def fake_base(counts, r, out=None, stream=None):
        return torch.from_numpy(counts.numpy()[:r].sum(axis=0).astype(np.int32))

    def fake_dispatch(idx, E, cf, T_total, base, ws=None, out=None, stream=None):
        ran.append("dispatch")
        i = idx.numpy()
        C = oracle.dispatch.capacity(int(T_total), i.shape[1], E, cf)
        g = base.numpy()[i.ravel()] + oracle.dispatch.dispatch(i, E, 10 ** 9)["slot"]
        return {"slot": np.where(g < C, g, -1), "capacity": C}

    def fake_bwd(logits, f, alpha, g, dlogits=None, stream=None):
        ran.append("bwd")
        return torch.zeros(logits.shape, dtype=torch.float32)

    dp.api.moe_router_fwd = fake_fwd
    dp.api.moe_router_combine = fake_combine
    dp.api.moe_shard_capacity_base = fake_base
    dp.api.moe_dispatch_sharded = fake_dispatch
    dp.api.moe_dispatch_capacity = lambda T, E, k, cf: oracle.dispatch.capacity(int(T), k, E, cf)
    dp.api.moe_router_bwd = fake_bwd
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rows = T_Z if rank == 0 else 0
        x = torch.from_numpy(np.random.default_rng(7).standard_normal((T_Z, E_Z)).astype(np.float32)[:rows].copy())
        b = dp.data_parallel_step(x, K_Z, 0.01, CF_Z)
        out.put((rank, ran, tuple(b["idx"].shape), np.asarray(b["slot"]), tuple(b["dlogits"].shape),
                 b["T_local"], b["T_total"], b["capacity"], np.asarray(b["counts"])))
    finally:
        dist.destroy_process_group()


def test_a_rank_without_rows_gloo():
    sys.path.insert(0, str(ROOT))
    import oracle
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    world, port = 2, _free_port()
    procs = [ctx.Process(target=_rank_empty_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted((q.get(timeout=120) for _ in range(world)), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    x = np.random.default_rng(7).standard_normal((T_Z, E_Z)).astype(np.float32)
    fw = oracle.router.router_forward(x, "fp32", K_Z, 0.01)
    C = oracle.dispatch.capacity(T_Z, K_Z, E_Z, CF_Z)
    whole = oracle.dispatch.dispatch(fw["idx"], E_Z, C)
    (_, ran0, idx0, slot0, dl0, tl0, tt0, c0, n0), (_, ran1, idx1, slot1, dl1, tl1, tt1, c1, n1) = got
    assert ran0 == ["fwd", "dispatch", "bwd"] and ran1 == []
    assert idx0 == (T_Z, K_Z) and dl0 == (T_Z, E_Z) and tl0 == T_Z
    assert idx1 == (0, K_Z) and slot1.shape == (0,) and dl1 == (0, E_Z) and tl1 == 0
    assert tt0 == tt1 == T_Z and c0 == c1 == C
    assert np.array_equal(n0, fw["counts"]) and np.array_equal(n1, fw["counts"])
    assert np.array_equal(slot0, whole["slot"])
