"""Oracle: TAOT Phase 2, column-first iterative matching of hot experts to cold ranks ([P4] §2, §3).

TEST INFRASTRUCTURE (see the package docstring): plain Python integers.

What the page fixes:
  * Replica placement is an integer decision: a cold rank hosts at most K whole
    replicas of hot experts, and several cold ranks may want the same hot
    expert in one round, so conflicts are arbitrated.
  * Every (cold rank, hot expert) pair gets a three-level score: first the
    tokens the match moves (its balance gain), then the topology preference,
    and only then Phase 1's transport flow as a global hint for ties.
  * Column-first: in each round every cold rank picks its best expert on its
    own, conflicts are arbitrated, and a rank that lost picks again in the
    next round.  The rounds run in one fused launch.

Readings where the page is silent (parity unpinned: these are choices):
  * Experts sit on home ranks contiguously, E / R per rank; a rank's load is
    the sum of its experts' loads, the mean is total / R.  A rank is hot when
    its load is above the mean and cold when below (compared exactly, as
    load * R against total).
  * A match (c, e) moves x(c, e) = min(w_rem[e], floor(load[h] - mean),
    floor(mean - load[c])) tokens of expert e from its home rank h to cold
    rank c, where w_rem[e] is the part of e's load still at home.  Only
    matches with x > 0 count, and a cold rank takes an expert once.
  * Score of (c, e): x first; then topology, 1 when c and h share a node and 0
    when not; then the flow plan[h, c] of Phase 1 (fp32, compared as given);
    last the lower expert index.  Arbitration among the cold ranks that chose
    one expert uses the same score with the lower rank index last.
  * Each round's winners commit in ascending cold-rank order, each move taken
    again against the loads as they stand at that moment (so two winners
    drawing on one hot rank never push it below the mean); a move that has
    become empty is dropped.  K caps the replicas of a cold rank; rounds repeat
    until no cold rank finds a positive match.  (Read instead as exactly K
    rounds, column-first left more imbalance than an expert-major greedy on
    mildly skewed loads, the opposite of the page's 1-2 % against 7-10 %;
    repeated to convergence it leaves 1-4 %, below the expert-major greedy.)
"""

from __future__ import annotations

import numpy as np


def _floor_div(a: int, b: int) -> int:
    return a // b


def match(expert_loads, plan, R: int, ranks_per_node: int, K: int) -> dict:
    """Column-first matching of one microbatch.

    expert_loads: [E] integer token counts; plan: [R, R] fp32 Phase 1 flow
    (plan[h, c] from hot rank h to cold rank c).
    Returns slot_expert [R, K] (-1 where empty), slot_tokens [R, K] (tokens
    moved into each slot, in the round order), rank_load [R] after the moves,
    and moved (total tokens moved).
    Pinned by: hand cases; invariants (total kept, no rank crosses the mean,
    at most K slots, no pair twice, an expert never gives more than its load).
    """
    w = [int(x) for x in expert_loads]
    E = len(w)
    per = E // R
    home = [e // per for e in range(E)]
    load = [sum(w[r * per:(r + 1) * per]) for r in range(R)]
    total = sum(load)
    w_rem = list(w)
    used = [[False] * E for _ in range(R)]
    slot_e = [[-1] * K for _ in range(R)]
    slot_x = [[0] * K for _ in range(R)]
    n_slots = [0] * R
    P = np.asarray(plan, dtype=np.float32)

    def excess(r):       # floor(load - mean), for a hot rank
        return _floor_div(load[r] * R - total, R)

    def spare(r):        # floor(mean - load), for a cold rank
        return _floor_div(total - load[r] * R, R)

    def moved(c, e):
        h = home[e]
        if load[h] * R <= total or load[c] * R >= total or used[c][e] or w_rem[e] <= 0:
            return 0
        return max(0, min(w_rem[e], excess(h), spare(c)))

    def score(c, e):
        h = home[e]
        return (moved(c, e), 1 if h // ranks_per_node == c // ranks_per_node else 0, float(P[h, c]))

    while True:
        choice = {}
        for c in range(R):
            if n_slots[c] >= K:
                continue
            best, best_s = -1, None
            for e in range(E):
                s = score(c, e)
                if s[0] <= 0:
                    continue
                if best < 0 or s > best_s:          # ties keep the lower expert index
                    best, best_s = e, s
            if best >= 0:
                choice[c] = (best, best_s)
        if not choice:
            break
        winner = {}
        for c in sorted(choice):
            e, s = choice[c]
            if e not in winner or s > winner[e][1]:  # ties keep the lower rank index
                winner[e] = (c, s)
        for c in sorted(cw for cw, _ in winner.values()):
            e = choice[c][0]
            x = moved(c, e)
            if x <= 0:
                continue
            h = home[e]
            load[h] -= x
            load[c] += x
            w_rem[e] -= x
            used[c][e] = True
            slot_e[c][n_slots[c]] = e
            slot_x[c][n_slots[c]] = x
            n_slots[c] += 1
    return {"slot_expert": np.asarray(slot_e, dtype=np.int64), "slot_tokens": np.asarray(slot_x, dtype=np.int64),
            "rank_load": np.asarray(load, dtype=np.int64), "moved": int(sum(map(sum, slot_x)))}


def residual_imbalance(rank_load) -> float:
    """(max load - mean) / mean: the imbalance measure of [P4] §2 (1-2 % column-first vs 7-10 % row-first).

    Pinned by: hand values ([6, 4, 5, 5] -> 0.2, [9, 1] -> 0.8, equal loads -> 0).
    """
    rl = np.asarray(rank_load, dtype=np.float64)
    return float((rl.max() - rl.mean()) / rl.mean())
