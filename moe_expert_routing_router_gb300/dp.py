"""Data-parallel batch statistics over ranks that each route their own tokens.

The Switch balance terms f and P are means over the whole batch.  When the
batch is split over data-parallel ranks, each rank routes its tokens with
``moe_router_fwd``, the ranks exchange their per-expert counts and P (one
all-gather of 2E values and the token count per rank), ``moe_router_combine``
turns them into the batch's f, P and scalars, and each rank's
``moe_router_bwd`` takes the batch's f with its coefficient scaled from its own
T to the batch's.  The exchange is ``torch.distributed`` plumbing (NCCL between
GPUs, gloo on CPU); every number is computed by the library's kernels.
"""

from __future__ import annotations

import torch
import torch.distributed as dist

from . import api


def gather_shard_stats(counts: torch.Tensor, P: torch.Tensor, T_local: int, group=None):
    """All-gathers one rank's counts [E] (int32) and P [E] (fp32) and its token
    count; returns (counts [G, E], P [G, E], T_shard list of G ints), in rank order."""
    G = dist.get_world_size(group)
    c_all = [torch.empty_like(counts) for _ in range(G)]
    p_all = [torch.empty_like(P) for _ in range(G)]
    t = torch.tensor([int(T_local)], dtype=torch.int64, device=counts.device)
    t_all = [torch.empty_like(t) for _ in range(G)]
    dist.all_gather(c_all, counts.contiguous(), group=group)
    dist.all_gather(p_all, P.contiguous(), group=group)
    dist.all_gather(t_all, t, group=group)
    return torch.stack(c_all), torch.stack(p_all), [int(x.item()) for x in t_all]


def shard_grad_scale(grad_scale: float, T_local: int, T_total: int) -> float:
    """The grad_scale that turns a shard's aux-loss coefficient alpha*E/T_local
    into the batch's alpha*E/T_total."""
    return float(grad_scale) * float(T_local) / float(T_total)


def data_parallel_forward(logits: torch.Tensor, k: int, alpha: float, renorm: int = -1, n_ranks: int = 0,
                          group=None, ws=None, stream=None) -> dict:
    """This rank's routing (idx, gate) and the whole batch's counts, f, P,
    scalars and rank loads; also the batch's T and this rank's T."""
    local = api.moe_router_fwd(logits, k, alpha, renorm=renorm, n_ranks=n_ranks, ws=ws, stream=stream)
    c_all, p_all, T_shard = gather_shard_stats(local["counts"], local["P"], logits.shape[0], group)
    batch = api.moe_router_combine(c_all, p_all, T_shard, k, alpha, n_ranks=n_ranks, stream=stream)
    batch.update(idx=local["idx"], gate=local["gate"], T_total=sum(T_shard), T_local=int(logits.shape[0]))
    return batch


def data_parallel_backward(logits: torch.Tensor, batch: dict, alpha: float, grad_scale: float = 1.0,
                           dlogits=None, stream=None) -> torch.Tensor:
    """dL_aux/dlogits of this rank's rows for the whole batch's loss."""
    g = shard_grad_scale(grad_scale, batch["T_local"], batch["T_total"])
    return api.moe_router_bwd(logits, batch["f"], alpha, g, dlogits=dlogits, stream=stream)
