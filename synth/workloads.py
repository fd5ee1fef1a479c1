"""Seeded synthetic router workloads.

Every workload is a token-by-expert matrix of router logits z[T, E]:

  * ``switch-top1-T4096-E8``: fp32 logits drawn i.i.d. N(0, 1); Switch top-1
    routing over 8 experts (the 8-expert setting of the MoE article's
    capacity example, section 4.5 of the untitled HPC load-balancing article at
    mhpq.cn/news/998159).
  * ``zipf-top2-T65536-E64``: 16 sequences x 4096 tokens, 64 experts, top-2 with
    the gate renormalised over the two picks.  Logits are N(0, 1) plus a
    per-expert bias b_e = 1.5 * ln(w_e), where w is a Zipf(s=1.1) law laid over
    a seeded permutation of the experts (a few hot experts, a long cold tail).
  * ``zipf-hot-top8-T131072-E256``: as above with s=1.2, 256 experts, top-8, and
    5% of the tokens carrying +3.0 on one randomly chosen hot expert; capacity
    factor 1.0 so that the dispatch drops tokens.
  * ``zipf-ep64-top6-T262144-E384``: s=1.3, 384 experts, top-6 (the expert
    count and fan-out of the model family named in the introduction of the
    TAOT article), experts mapped contiguously onto 64 simulated
    expert-parallel ranks of 6 experts, 8 ranks per node.

The bf16 workloads are formed in fp64, rounded to fp32 and then to bf16 with
round-to-nearest-even, and are returned as the raw uint16 bit patterns.

Random streams: ``numpy.random.Generator(PCG64(SeedSequence(seed,
spawn_key=(workload_id,))))``.  Draw order: expert permutation, the [T, E]
standard normals (row-major), then the hot expert and the hot token set.
"""

from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np


@dataclass(frozen=True)
class RouterWorkload:
    name: str
    workload_id: int
    T: int
    E: int
    k: int
    dtype: str                 # "fp32" or "bf16"
    alpha: float
    capacity_factor: float
    renorm: bool               # gate renormalised over the k picks
    zipf_s: float | None       # None: no per-expert bias
    bias_scale: float = 1.5
    hot_frac: float = 0.0
    hot_bump: float = 0.0
    n_ranks: int = 0           # simulated expert-parallel ranks (0: none)
    ranks_per_node: int = 0

    def with_tokens(self, T: int) -> "RouterWorkload":
        """Same recipe at another token count (a fresh draw, not a prefix)."""
        return replace(self, T=int(T), name=f"{self.name}@T{T}")


@dataclass(frozen=True)
class SinkhornWorkload:
    name: str
    B: int                     # microbatches
    R: int                     # simulated expert-parallel ranks
    ranks_per_node: int
    lam: float                 # cross-node cost lambda
    eps: float                 # entropic regulariser (epsilon = lambda)
    iters: int
    tokens_per_microbatch: int
    source: str                # router workload whose generator is re-seeded per microbatch


ROUTER_WORKLOADS: dict[str, RouterWorkload] = {
    w.name: w
    for w in (
        RouterWorkload("switch-top1-T4096-E8", 1, 4096, 8, 1, "fp32", 0.01, 1.25,
                       renorm=False, zipf_s=None),
        RouterWorkload("zipf-top2-T65536-E64", 2, 65536, 64, 2, "bf16", 0.01, 1.25,
                       renorm=True, zipf_s=1.1),
        RouterWorkload("zipf-hot-top8-T131072-E256", 3, 131072, 256, 8, "bf16", 0.001, 1.0,
                       renorm=True, zipf_s=1.2, hot_frac=0.05, hot_bump=3.0),
        RouterWorkload("zipf-ep64-top6-T262144-E384", 4, 262144, 384, 6, "bf16", 0.001, 1.25,
                       renorm=True, zipf_s=1.3, n_ranks=64, ranks_per_node=8),
    )
}

SINKHORN_WORKLOADS: dict[str, SinkhornWorkload] = {
    "taot-sinkhorn-B1024-R64": SinkhornWorkload(
        "taot-sinkhorn-B1024-R64", B=1024, R=64, ranks_per_node=8, lam=10.0, eps=10.0,
        iters=50, tokens_per_microbatch=4096, source="zipf-ep64-top6-T262144-E384"),
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bit patterns.

    Inputs must be finite.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(seed: int, workload_id: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(workload_id,))))


def _encode(z64: np.ndarray, dtype: str) -> np.ndarray:
    z32 = z64.astype(np.float32)
    if dtype == "fp32":
        return z32
    if dtype == "bf16":
        return f32_to_bf16_bits(z32)
    raise ValueError(f"unknown dtype {dtype!r}")


@dataclass(frozen=True)
class EplbWorkload:
    """Per-expert token counts of B independent problems (layers or
    microbatches) for the replication and packing planner."""
    name: str
    workload_id: int
    B: int
    E: int
    assignments: int           # T * k per problem
    zipf_s: float
    num_phys: int              # physical expert slots
    num_gpus: int
    num_nodes: int
    num_groups: int            # contiguous expert groups (0: none)


EPLB_WORKLOADS: dict[str, EplbWorkload] = {
    "eplb-zipf-E384-B1024": EplbWorkload("eplb-zipf-E384-B1024", 5, B=1024, E=384, assignments=4096 * 6,
                                         zipf_s=1.3, num_phys=448, num_gpus=64, num_nodes=8, num_groups=32),
}


def eplb_loads(w: EplbWorkload, B: int | None = None) -> np.ndarray:
    """int64 [B, E] expert token counts: problem b draws a seeded permutation of
    the experts, Zipf(s) probabilities over it, and a multinomial of
    ``assignments`` draws."""
    B = w.B if B is None else B
    rng = _rng(0, w.workload_id)
    out = np.empty((B, w.E), dtype=np.int64)
    for b in range(B):
        perm = rng.permutation(w.E)
        p = (perm + 1.0) ** (-w.zipf_s)
        out[b] = rng.multinomial(w.assignments, p / p.sum())
    return out


def router_logits(w: RouterWorkload, seed: int = 0) -> np.ndarray:
    """Logits of workload ``w``: float32 [T, E] for fp32, uint16 bf16 bits [T, E] for bf16."""
    rng = _rng(seed, w.workload_id)
    T, E = w.T, w.E
    bias = np.zeros(E)
    if w.zipf_s is not None:
        perm = rng.permutation(E)                      # rank of expert e in the Zipf law
        weights = (perm + 1.0) ** (-w.zipf_s)
        weights /= weights.sum()
        bias = w.bias_scale * np.log(weights)
    z = rng.standard_normal((T, E))
    z += bias[None, :]
    if w.hot_frac > 0.0:
        hot_expert = int(rng.integers(E))
        n_hot = int(np.floor(w.hot_frac * T + 0.5))
        hot_tokens = rng.choice(T, size=n_hot, replace=False)
        z[hot_tokens, hot_expert] += w.hot_bump
    return _encode(z, w.dtype)


def sinkhorn_microbatch_logits(s: SinkhornWorkload, m: int) -> np.ndarray:
    """Logits of microbatch ``m``: the source router workload re-seeded with seed ``m``."""
    src = ROUTER_WORKLOADS[s.source].with_tokens(s.tokens_per_microbatch)
    return router_logits(src, seed=m)


def random_logits(T: int, E: int, dtype: str, seed: int, scale: float = 1.0,
                  integer_levels: int = 0) -> np.ndarray:
    """Small ad-hoc inputs for edge cases.

    ``integer_levels > 0`` draws integers in [0, integer_levels) so that equal
    logits (ties) are common.
    """
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(1000,))))
    if integer_levels > 0:
        z = rng.integers(0, integer_levels, size=(T, E)).astype(np.float64)
    else:
        z = scale * rng.standard_normal((T, E))
    return _encode(z, dtype)
