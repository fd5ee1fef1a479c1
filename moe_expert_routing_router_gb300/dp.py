"""Data-parallel batch statistics over ranks that each route their own tokens.

The Switch balance terms f and P are means over the whole batch.  When the
batch is split over data-parallel ranks, each rank routes its tokens with
``moe_router_fwd``, the ranks exchange their per-expert counts and P (one
all-gather of 2E values, plus the token count per rank unless every rank
knows them), ``moe_router_combine``
turns them into the batch's f, P and scalars, and each rank's
``moe_router_bwd`` takes the batch's f with its coefficient scaled from its own
T to the batch's.  The exchange is ``torch.distributed`` plumbing (NCCL between
GPUs, gloo on CPU); every number is computed by the library's kernels.

Dispatch with the capacity of the whole batch reuses the gathered counts: each
rank's ``moe_shard_capacity_base`` is the exclusive scan of the counts across
the ranks below it, and ``moe_dispatch_sharded`` places the rank's assignments
after them in each expert's buffer, so the ranks' slots together are those of
one dispatch over the whole batch.

A rank that holds no rows of the batch still takes part in the exchange, with
zero counts and P and a token count of 0, so that the other ranks' collectives
complete; its per-row outputs are empty.
"""

from __future__ import annotations

import torch
import torch.distributed as dist

from . import api


def gather_shard_stats(counts: torch.Tensor, P: torch.Tensor, T_local: int, group=None, T_shard=None):
    """All-gathers one rank's counts [E] (int32) and P [E] (fp32), packed into
    one buffer of 2E 32-bit words (one collective), and the ranks' token counts
    unless T_shard (every rank's T, known to all) is given; returns
    (counts [G, E], P [G, E], T_shard list of G ints), in rank order."""
    G = dist.get_world_size(group)
    E = counts.numel()
    packed = torch.empty(2 * E, dtype=torch.int32, device=counts.device)
    packed[:E].copy_(counts.reshape(-1))
    packed[E:].copy_(P.contiguous().reshape(-1).view(torch.int32))
    parts = [torch.empty_like(packed) for _ in range(G)]
    dist.all_gather(parts, packed, group=group)
    rows = torch.stack(parts)
    c_all = rows[:, :E].contiguous()
    p_all = rows[:, E:].contiguous().view(torch.float32)
    if T_shard is None:
        t = torch.tensor([int(T_local)], dtype=torch.int64, device=counts.device)
        t_all = [torch.empty_like(t) for _ in range(G)]
        dist.all_gather(t_all, t, group=group)
        T_shard = [int(x.item()) for x in t_all]
    elif len(T_shard) != G or int(T_shard[dist.get_rank(group)]) != int(T_local):
        raise ValueError("T_shard must list every rank's token count, this rank's included")
    return c_all, p_all, [int(x) for x in T_shard]


def shard_grad_scale(grad_scale: float, T_local: int, T_total: int) -> float:
    """The grad_scale that turns a shard's aux-loss coefficient alpha*E/T_local
    into the batch's alpha*E/T_total."""
    return float(grad_scale) * float(T_local) / float(T_total)


def data_parallel_forward(logits: torch.Tensor, k: int, alpha: float, renorm: int = -1, n_ranks: int = 0,
                          group=None, ws=None, stream=None, T_shard=None) -> dict:
    """This rank's routing (idx, gate) and the whole batch's counts, f, P,
    scalars and rank loads; also the batch's T and this rank's T."""
    T_local, E = int(logits.shape[0]), int(logits.shape[1])
    if T_local > 0:
        local = api.moe_router_fwd(logits, k, alpha, renorm=renorm, n_ranks=n_ranks, ws=ws, stream=stream)
    else:
        with api._on(stream):
            local = {"idx": torch.empty((0, k), dtype=torch.int32, device=logits.device),
                     "gate": torch.empty((0, k), dtype=torch.float32, device=logits.device),
                     "counts": torch.zeros(E, dtype=torch.int32, device=logits.device),
                     "P": torch.zeros(E, dtype=torch.float32, device=logits.device)}
    # The torch side of the exchange (packing copies, collectives, slices) on the
    # stream of the library's calls: after the forward that wrote counts and P,
    # before the combine that reads them.
    with api._on(stream):
        c_all, p_all, T_shard = gather_shard_stats(local["counts"], local["P"], T_local, group, T_shard)
    batch = api.moe_router_combine(c_all, p_all, T_shard, k, alpha, n_ranks=n_ranks, stream=stream)
    batch.update(idx=local["idx"], gate=local["gate"], T_total=sum(T_shard), T_local=T_local,
                 counts_all=c_all, rank=dist.get_rank(group))
    return batch


def data_parallel_dispatch(idx: torch.Tensor, batch: dict, E: int, capacity_factor: float, ws=None,
                           stream=None) -> dict:
    """This rank's dispatch with the whole batch's capacity: slots after the
    lower ranks' assignments to each expert, from the counts the forward's
    exchange gathered (``batch`` as data_parallel_forward returns it)."""
    base = api.moe_shard_capacity_base(batch["counts_all"], batch["rank"], stream=stream)
    if idx.shape[0] == 0:
        k, dev = int(idx.shape[1]), idx.device
        with api._on(stream):
            out = {"perm": torch.empty(0, dtype=torch.int32, device=dev),
                   "slot": torch.empty(0, dtype=torch.int32, device=dev),
                   "offsets": torch.zeros(E + 1, dtype=torch.int32, device=dev),
                   "kept": torch.zeros(E, dtype=torch.int32, device=dev),
                   "n_dropped": torch.zeros(1, dtype=torch.int32, device=dev)}
        out["capacity"] = api.moe_dispatch_capacity(batch["T_total"], E, k, capacity_factor)
    else:
        out = api.moe_dispatch_sharded(idx, E, capacity_factor, batch["T_total"], base, ws=ws, stream=stream)
    out["cap_base"] = base
    return out


def data_parallel_step(logits: torch.Tensor, k: int, alpha: float, capacity_factor: float, renorm: int = -1,
                       n_ranks: int = 0, grad_scale: float = 1.0, group=None, ws=None, stream=None,
                       T_shard=None) -> dict:
    """One pass of the hot path over this rank's rows of a data-parallel batch:
    the local forward, the exchange of counts, P and T, the combine, the
    dispatch with the batch's capacity and the backward of the batch's loss."""
    batch = data_parallel_forward(logits, k, alpha, renorm=renorm, n_ranks=n_ranks, group=group, ws=ws,
                                  stream=stream, T_shard=T_shard)
    batch.update(data_parallel_dispatch(batch["idx"], batch, logits.shape[1], capacity_factor, ws=ws, stream=stream))
    batch["dlogits"] = data_parallel_backward(logits, batch, alpha, grad_scale=grad_scale, stream=stream)
    return batch


def data_parallel_backward(logits: torch.Tensor, batch: dict, alpha: float, grad_scale: float = 1.0,
                           dlogits=None, stream=None) -> torch.Tensor:
    """dL_aux/dlogits of this rank's rows for the whole batch's loss."""
    if batch["T_local"] == 0:
        if dlogits is not None:
            return dlogits
        with api._on(stream):
            return torch.empty((0, logits.shape[1]), dtype=torch.float32, device=logits.device)
    g = shard_grad_scale(grad_scale, batch["T_local"], batch["T_total"])
    return api.moe_router_bwd(logits, batch["f"], alpha, g, dlogits=dlogits, stream=stream)
