"""Oracle: EPLB expert replication and balanced packing ([P3] §4.1.2).

TEST INFRASTRUCTURE (see the package docstring): plain Python / numpy.

What the page fixes:
  * replicate_experts: heavy experts get extra replicas until the physical
    expert count reaches its target; each step computes weight / count (the
    load one replica of each expert carries) and replicates the expert where
    that is largest.
  * balanced_packing: items with weights go into a fixed number of bins that
    each take the same number of items; items are taken heaviest first and
    each goes to the currently lightest bin that is not full.  Worked example:
    group loads [9, 7, 5, 3] onto 2 nodes of 2 groups: 9 -> node 0, 7 -> node 1,
    5 -> node 1 (12), 3 -> node 0: both nodes carry 12.
  * Two policies: hierarchical (used when the node count divides the group
    count): groups are packed onto nodes, experts are replicated within each
    node, and the node's replicas are packed onto its GPUs; global (otherwise):
    experts are replicated over the whole system and the replicas packed onto
    all GPUs.

Readings where the page is silent:
  * Loads are integer token counts.  The replication choice compares
    w_a / c_a with w_b / c_b exactly (as w_a * c_b against w_b * c_a); ties go
    to the lower expert index.
  * A replica's weight in the packing is fp32(w) / fp32(c) in fp32 (one
    correctly rounded division); a group's weight is fp32 of its integer sum;
    a bin's total is the fp32 sum of its items in the order they were placed.
    These decide integers (the bin of each item), so both sides take them in
    the same fp32 arithmetic (the kernel's precision).
  * Packing order: weight descending, ties to the lower item index; the
    lightest non-full bin, ties to the lower bin index.
  * Physical expert slots are numbered GPU-major: GPU g holds slots
    [g*S, (g+1)*S), S = num_phys / num_gpus, filled in the order the packing
    placed them.  Replica r >= 1 of the replication is item E + (order of
    its creation); item e < E is the expert's first copy.
  * Groups are contiguous blocks of E / num_groups experts.  Hierarchically,
    node n's logical experts are those of its groups, in the order the groups
    were placed on it, each group's experts in ascending index; node n owns
    GPUs [n*G/N, (n+1)*G/N) and num_phys / num_nodes physical slots.
"""

from __future__ import annotations

import numpy as np


def replicate_experts(weights, num_phys: int) -> tuple[np.ndarray, np.ndarray]:
    """Replicate the expert with the largest weight/count until there are num_phys copies.

    Returns (phy2log [num_phys], count [E]): item e < E is expert e's first
    copy, item E + r the r-th replica created.
    Pinned by: brute force over all count vectors (the greedy reaches the
    smallest possible max_e w_e / c_e); a hand case; num_phys = E is the identity.
    """
    w = [int(x) for x in weights]
    E = len(w)
    assert num_phys >= E
    count = [1] * E
    phy2log = list(range(E))
    for _ in range(num_phys - E):
        best = 0
        for e in range(1, E):
            if w[e] * count[best] > w[best] * count[e]:     # w_e/c_e > w_best/c_best, exactly
                best = e
        count[best] += 1
        phy2log.append(best)
    return np.asarray(phy2log, dtype=np.int64), np.asarray(count, dtype=np.int64)


def balanced_packing(weights, num_bins: int) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Greedy equal-cardinality packing ([P3] §4.1.2).

    weights: per item, taken as fp32; len(weights) must be a multiple of num_bins.
    Returns (bin [N], position within its bin [N], bin totals [num_bins], fp32).
    Pinned by: the page's [9, 7, 5, 3] example; equal weights fill the bins
    round-robin; every bin gets N / num_bins items.
    """
    w = [np.float32(x) for x in weights]
    N = len(w)
    assert N % num_bins == 0
    cap = N // num_bins
    order = sorted(range(N), key=lambda i: (-float(w[i]), i))
    totals = [np.float32(0.0)] * num_bins
    fill = [0] * num_bins
    bin_of = [0] * N
    pos = [0] * N
    for i in order:
        best = -1
        for b in range(num_bins):
            if fill[b] < cap and (best < 0 or totals[b] < totals[best]):
                best = b
        bin_of[i] = best
        pos[i] = fill[best]
        fill[best] += 1
        totals[best] = np.float32(totals[best] + w[i])
    return np.asarray(bin_of), np.asarray(pos), np.asarray(totals, dtype=np.float32)


def _replica_weights(weights, phy2log, count) -> list:
    return [np.float32(weights[e]) / np.float32(count[e]) for e in phy2log]


def _place(phy2log_local, bins, pos, gpu0: int, S: int, out: np.ndarray) -> None:
    for item, e in enumerate(phy2log_local):
        out[(gpu0 + bins[item]) * S + pos[item]] = e


def plan_global(weights, num_phys: int, num_gpus: int) -> dict:
    """Global policy: replicate over all experts, pack the replicas onto all GPUs.

    Pinned by: the hand case [6, 2, 1, 3] onto 6 slots of 2 GPUs (6 / 6); the
    plan invariants (S slots per GPU, copies equal counts, loads add up).
    """
    E = len(weights)
    S = num_phys // num_gpus
    p2l, count = replicate_experts(weights, num_phys)
    rw = _replica_weights(weights, p2l, count)
    bins, pos, totals = balanced_packing(rw, num_gpus)
    phy2log = np.empty(num_phys, dtype=np.int64)
    _place(p2l, bins, pos, 0, S, phy2log)
    return {"phy2log": phy2log, "log_count": count, "gpu_load": totals, "hierarchical": False}


def plan_hierarchical(weights, num_phys: int, num_gpus: int, num_nodes: int, num_groups: int) -> dict:
    """Hierarchical policy: groups onto nodes, then replication and packing within each node.

    Pinned by: the page's groups [9, 7, 5, 3] on 2 nodes worked by hand (12 / 12);
    the plan invariants, with every copy on the node its group went to.
    """
    w = [int(x) for x in weights]
    E = len(w)
    gsize = E // num_groups
    gpn = num_gpus // num_nodes
    S = num_phys // num_gpus
    phys_per_node = num_phys // num_nodes
    group_w = [np.float32(sum(w[g * gsize:(g + 1) * gsize])) for g in range(num_groups)]
    gbin, gpos, _ = balanced_packing(group_w, num_nodes)
    phy2log = np.empty(num_phys, dtype=np.int64)
    count = np.zeros(E, dtype=np.int64)
    gpu_load = np.zeros(num_gpus, dtype=np.float32)
    for n in range(num_nodes):
        groups = sorted((g for g in range(num_groups) if gbin[g] == n), key=lambda g: gpos[g])
        experts = [g * gsize + j for g in groups for j in range(gsize)]
        p2l, cnt = replicate_experts([w[e] for e in experts], phys_per_node)
        for j, e in enumerate(experts):
            count[e] = cnt[j]
        rw = _replica_weights([w[e] for e in experts], p2l, cnt)
        bins, pos, totals = balanced_packing(rw, gpn)
        _place([experts[j] for j in p2l], bins, pos, n * gpn, S, phy2log)
        gpu_load[n * gpn:(n + 1) * gpn] = totals
    return {"phy2log": phy2log, "log_count": count, "gpu_load": gpu_load, "hierarchical": True}


def plan(weights, num_phys: int, num_gpus: int, num_nodes: int, num_groups: int) -> dict:
    """The page's choice of policy: hierarchical when num_groups > 0 and the node
    count divides the group count, global otherwise.  Pinned by: both branches
    taken in the plan pins (3 nodes do not divide 8 groups: global)."""
    if num_groups > 0 and num_groups % num_nodes == 0:
        return plan_hierarchical(weights, num_phys, num_gpus, num_nodes, num_groups)
    return plan_global(weights, num_phys, num_gpus)
