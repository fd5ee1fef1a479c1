"""Oracle: TAOT Phase 1, the topology-aware Sinkhorn-Knopp flow plan.

TEST INFRASTRUCTURE (see the package docstring): plain float64 numpy.

[P4] §2, Phase 1: each rank's overload is a supply and each rank's idle
capacity a demand; the optimal transport between them under a topology cost
matrix W, relaxed with a negative-entropy term, has the Gibbs form
T = diag(u) * M * diag(v) with M = exp(-W / eps), and alternating
Sinkhorn-Knopp matrix-vector iterations find u and v.  Taking eps equal to the
cross-node cost lambda makes the intra-node to cross-node kernel ratio
greater than one (the "soft topology preference").  [P4] §3: 50 iterations,
each a matrix-vector product plus a clamp.

Readings where the page is silent:
  * supply_r = max(load_r - mean, 0), demand_r = max(mean - load_r, 0), each
    normalised to unit mass; with no supply (all loads equal) the plan is
    empty: u = v = 0, plan = 0, status 1.
  * W[r, s] = 0 on the same rank, 1 within a node, lambda across nodes; rank
    r sits on node floor(r / ranks_per_node).
  * v starts at 1; each iteration updates u, then v; the clamp bounds each
    denominator below by 1e-30.
"""

from __future__ import annotations

import numpy as np

DENOMINATOR_FLOOR = 1e-30
STATUS_OK = 0
STATUS_NO_MASS = 1


def supply_demand(load: np.ndarray) -> tuple[np.ndarray, np.ndarray, bool]:
    """Unit-mass supply a (overloaded ranks) and demand b (idle ranks) of one load vector.

    Pinned by: hand cases ([3, 1, 1, 3] -> a = [1, 0, 0, 1] / 2, b = [0, 1, 1, 0] / 2;
    [5, 1, 0, 2] -> b = [0, 1, 2, 0] / 3); equal loads carry no mass.
    """
    load = np.asarray(load, dtype=np.float64)
    mean = load.mean()
    a = np.maximum(load - mean, 0.0)
    b = np.maximum(mean - load, 0.0)
    sa, sb = a.sum(), b.sum()
    if sa <= 0.0 or sb <= 0.0:
        return np.zeros_like(a), np.zeros_like(b), False
    return a / sa, b / sb, True


def topology_cost(R: int, ranks_per_node: int, lam: float) -> np.ndarray:
    """W[r, s]: 0 on the same rank, 1 within a node, ``lam`` across nodes.

    Pinned by: the 4-rank, 2-per-node matrix written out by hand; the intra- to
    cross-node kernel ratio at eps = lambda.
    """
    node = np.arange(R) // ranks_per_node
    W = np.where(node[:, None] == node[None, :], 1.0, float(lam))
    np.fill_diagonal(W, 0.0)
    return W


def gibbs_kernel(W: np.ndarray, eps: float) -> np.ndarray:
    """M = exp(-W / eps).  Pinned by: exp(-1/2) and exp(-5) at eps = 2 by hand; the kernel ratio."""
    return np.exp(-W / float(eps))


def sinkhorn_knopp(a: np.ndarray, b: np.ndarray, M: np.ndarray, iters: int) -> tuple[np.ndarray, np.ndarray]:
    """v = 1; ``iters`` times: u = a / (M v), then v = b / (M^T u).

    Works for any positive M (not only the symmetric topology kernel).
    Pinned by: the marginals of diag(u) M diag(v); an independent dual
    optimiser (scipy) on small problems; a two-rank closed form.
    """
    v = np.ones(len(b))
    u = np.zeros(len(a))
    for _ in range(iters):
        Mv = (M * v[None, :]).sum(axis=1)
        u = a / np.maximum(Mv, DENOMINATOR_FLOOR)
        Mtu = (M * u[:, None]).sum(axis=0)
        v = b / np.maximum(Mtu, DENOMINATOR_FLOOR)
    return u, v


def transport_plan(u: np.ndarray, M: np.ndarray, v: np.ndarray) -> np.ndarray:
    """T = diag(u) M diag(v).  Pinned by: the plan's marginals a and b; the independent dual solve."""
    return u[:, None] * M * v[None, :]


def taot_phase1(loads: np.ndarray, ranks_per_node: int, lam: float, eps: float | None = None,
                iters: int = 50) -> dict:
    """Batched Phase 1 over microbatches: loads [B, R] -> u, v [B, R], plan [B, R, R], status [B].

    Pinned by its parts' pins; 50 iterations reach the 10,000-iteration plan;
    equal loads give status 1 and an empty plan.
    """
    loads = np.atleast_2d(np.asarray(loads, dtype=np.float64))
    B, R = loads.shape
    if eps is None or eps <= 0:
        eps = lam
    M = gibbs_kernel(topology_cost(R, ranks_per_node, lam), eps)
    U = np.zeros((B, R))
    V = np.zeros((B, R))
    plan = np.zeros((B, R, R))
    status = np.zeros(B, dtype=np.int32)
    for m in range(B):
        a, b, ok = supply_demand(loads[m])
        if not ok:
            status[m] = STATUS_NO_MASS
            continue
        u, v = sinkhorn_knopp(a, b, M, iters)
        U[m], V[m] = u, v
        plan[m] = transport_plan(u, M, v)
    return {"u": U, "v": V, "plan": plan, "status": status, "M": M}
