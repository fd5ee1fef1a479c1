"""Oracle: expert capacity and the capacity-limited, stable token->expert dispatch.

TEST INFRASTRUCTURE (see the package docstring): plain numpy, integers only.

[P1] §4.5: every expert takes at most ``capacity`` tokens per batch; the
assignments beyond it are dropped.  Readings where the page is silent:
  * For top-k the batch holds T*k assignments, so
    C = ceil(ceil(T*k / E) * capacity_factor)  (the page's 1024 tokens,
    8 experts and factor 1.25 give 160).
  * Which assignments are dropped: the dispatch is a stable sort of the
    flattened assignments a = t*k + j by expert, so an expert keeps its
    first C assignments in token order and drops the rest.
  * perm holds assignment ids; offsets[e] is the exclusive prefix of the
    pre-drop counts (offsets[E] = T*k); the kept assignments of expert e are
    perm[offsets[e] : offsets[e] + kept[e]].
"""

from __future__ import annotations

import math

import numpy as np


def capacity(T: int, k: int, E: int, capacity_factor: float) -> int:
    """C = ceil(ceil(T*k/E) * capacity_factor), the product taken in float64.  [P1] §4.5.

    Pinned by: the page's worked example (1024 tokens, 8 experts, 1.25 -> 160).
    """
    per_expert = -(-(T * k) // E)          # integer ceil(T*k / E)
    return int(math.ceil(per_expert * float(capacity_factor)))


def dispatch(idx: np.ndarray, E: int, C: int) -> dict:
    """Stable counting-sort dispatch of the assignments in ``idx`` [T, k].

    Returns perm [T*k] (assignment ids sorted by expert, ascending id within an
    expert), slot [T*k] (rank of the assignment within its expert, -1 when the
    rank is >= C), offsets [E+1], counts [E], kept [E] = min(counts, C) and
    n_dropped.  Pinned by: an O((T*k)^2) brute force on small inputs and the
    counting identities (sum kept + n_dropped == T*k, offsets[E] == T*k).
    """
    flat = np.asarray(idx, dtype=np.int64).ravel()
    n = flat.size
    perm = np.argsort(flat, kind="stable")
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    rank = np.empty(n, dtype=np.int64)
    rank[perm] = np.arange(n, dtype=np.int64) - offsets[flat[perm]]
    slot = np.where(rank < C, rank, -1)
    kept = np.minimum(counts, C)
    return {
        "perm": perm, "slot": slot, "offsets": offsets, "counts": counts,
        "kept": kept, "n_dropped": int((counts - kept).sum()), "capacity": int(C),
    }
