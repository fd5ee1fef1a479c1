"""Oracle: router forward (softmax, top-k, gates, f, P, L_aux, CV) and dL_aux/dlogits.

TEST INFRASTRUCTURE (see the package docstring): plain float64 numpy.

Notation follows [P1] §4.2 and [P2] §2.2: N (here ``E``) experts, T tokens,
router logits z[t, e], p[t, e] = softmax(z[t, :])[e],
    f_i = share of the T*k assignments routed to expert i,
    P_i = (1/T) * sum_t p[t, i]          (mean router probability, all tokens),
    L_aux = alpha * N * sum_i f_i * P_i.

Readings where the pages are silent or disagree:
  * P_i is the unmasked mean of [P1] §4.2.  [P2] §2.2/§3.1 and the code of
    [P1] §4.4 mask P to the selected experts, but then sum_i P_i != 1, which
    [P1] §5.3 asserts, and the closed-form gradient below no longer holds.
  * f_i divides by T*k ([P1] §4.4: the top-k total is T*k, not T).  The eps of
    [P2] §3.1 is dropped.  f uses the pre-drop counts.
  * Top-k ranks the raw logits, descending, ties to the lower expert index;
    the selected experts are returned in that order.
  * The gate is p itself for k == 1 (Switch) and p renormalised over the k
    picks for k > 1 (``renorm`` overrides).
  * CV is the population standard deviation over the mean ([P3] §3.1/§5.1
    say only "standard deviation / mean").
"""

from __future__ import annotations

import numpy as np

from synth import bf16_bits_to_f32

SCALAR_NAMES = ("l_aux", "balance", "cv", "max_over_mean", "min_over_mean",
                "rank_cv", "rank_max_over_mean")


def widen(logits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 copy of fp32 logits or of bf16 bit patterns (uint16).

    Pinned by: torch's bfloat16 -> float32 conversion over every finite bf16
    pattern (subnormals, -0.0); hand values (0x3F80 = 1, 0xC040 = -3).
    """
    if dtype == "bf16":
        return bf16_bits_to_f32(logits).astype(np.float64)
    if dtype == "fp32":
        return np.asarray(logits, dtype=np.float32).astype(np.float64)
    raise ValueError(dtype)


def softmax(z: np.ndarray) -> np.ndarray:
    """Row softmax p[t, e] = exp(z[t,e] - max_e z[t,:]) / sum_e exp(...).

    [P1] §4.2 (P_i is the mean of softmax(router(x))_i); [P2] §3.1 step 3.
    Pinned by: scipy.special.softmax; rows sum to 1; shift invariance.
    """
    m = z.max(axis=1, keepdims=True)
    e = np.exp(z - m)
    return e / e.sum(axis=1, keepdims=True)


def top_k(z: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest logits per row, largest first, ties to the lower index.

    [P1] §4.4 (top-k routing), [P2] §3.1 (argmax / top-k decides the expert).
    A stable sort of -z keeps equal logits in ascending index order.
    Pinned by: brute-force enumeration of k-subsets; np.argmax for k == 1.
    """
    order = np.argsort(-z, axis=1, kind="stable")
    return order[:, :k]


def gates(p: np.ndarray, idx: np.ndarray, renorm: bool) -> np.ndarray:
    """Gate weights of the selected experts: p, or p / sum of the picked p.

    [P1] §4.4; [P2] §3.1.  Pinned by: hand examples (z = [0, ln 3]: top-1 gate
    3/4, renormalised top-2 [3/4, 1/4]; z = [ln 2, 0, ln 6]: [6/9, 2/9] plain).
    """
    g = np.take_along_axis(p, idx, axis=1)
    if renorm:
        g = g / g.sum(axis=1, keepdims=True)
    return g


def expert_counts(idx: np.ndarray, E: int) -> np.ndarray:
    """tokens_per_expert: assignments per expert, zero for unused experts.

    [P2] §3.1 (bincount with minlength=num_experts); [P1] §4.4 (scatter_add).
    Pinned by: sum == T*k; a brute-force loop on small inputs.
    """
    return np.bincount(np.asarray(idx).ravel(), minlength=E).astype(np.int64)


def token_fraction(counts: np.ndarray, T: int, k: int) -> np.ndarray:
    """f_i = counts_i / (T * k).  [P1] §4.4.  Pinned by: sum_i f_i == 1."""
    return counts / float(T * k)


def mean_router_prob(p: np.ndarray) -> np.ndarray:
    """P_i = (1/T) sum_t p[t, i] over all tokens.  [P1] §4.2.  Pinned by: sum_i P_i == 1."""
    return p.sum(axis=0) / p.shape[0]


def balance(f: np.ndarray, P: np.ndarray) -> float:
    """N * sum_i f_i P_i: equals 1 under uniform routing ([P2] §2.2).

    Pinned by: uniform P and uniform f both give 1; the two-token hand example 5/4.
    """
    return float(len(f) * np.sum(f * P))


def aux_loss(f: np.ndarray, P: np.ndarray, alpha: float) -> float:
    """L_aux = alpha * N * sum_i f_i P_i.  [P2] §2.2; [P1] §4.2.

    Pinned by: alpha at balance 1; the two-token hand example (0.0125 at alpha 0.01);
    the finite differences of the gradient, which differentiate it.
    """
    return alpha * balance(f, P)


def load_cv(loads: np.ndarray) -> float:
    """Coefficient of variation std/mean (population std) of a load vector.  [P3] §3.1, §5.1.

    Pinned by: closed forms ([1, 3] -> 1/2, [0, 0, 0, 4] -> sqrt 3, equal loads -> 0).
    """
    loads = np.asarray(loads, dtype=np.float64)
    mean = loads.mean()
    return float(loads.std() / mean) if mean > 0 else 0.0


def rank_loads(counts: np.ndarray, n_ranks: int) -> np.ndarray:
    """Token load of each simulated expert-parallel rank; experts are mapped
    contiguously, E / n_ranks per rank ([P4] introduction: a rank's load is the
    tokens routed to the experts it hosts).
    Pinned by: a hand-worked 12-expert, 4-rank case; one expert per rank gives
    the counts back, one rank the total."""
    E = len(counts)
    return np.asarray(counts).reshape(n_ranks, E // n_ranks).sum(axis=1)


def batch_statistics(counts: np.ndarray, P: np.ndarray, T: int, k: int, alpha: float,
                     n_ranks: int = 0) -> dict:
    """f and the batch scalars from the expert counts and P of a whole batch.

    max/mean and min/mean divide by the mean assignments per expert T*k/E;
    the rank max/mean by the mean per rank T*k/n_ranks ([P3] §5.1: max load
    over mean load); both CVs use the population deviation.
    Pinned by: a hand-worked 4-expert, 2-rank case (every scalar); the [P1]
    §5.3 log line (8192 tokens, 4320 on one expert: max/mean 4.21875)."""
    E = len(counts)
    f = token_fraction(counts, T, k)
    mean = T * k / E
    out = {
        "counts": counts, "f": f, "P": P,
        "l_aux": aux_loss(f, P, alpha), "balance": balance(f, P),
        "cv": load_cv(counts), "max_over_mean": counts.max() / mean,
        "min_over_mean": counts.min() / mean,
        "rank_cv": 0.0, "rank_max_over_mean": 0.0, "rank_load": np.zeros(0, np.int64),
    }
    if n_ranks > 0:
        rl = rank_loads(counts, n_ranks)
        out["rank_load"] = rl
        out["rank_cv"] = load_cv(rl)
        out["rank_max_over_mean"] = rl.max() / (T * k / n_ranks)
    return out


def router_forward(logits: np.ndarray, dtype: str, k: int, alpha: float,
                   renorm: bool | None = None, n_ranks: int = 0) -> dict:
    """The whole forward of the router on one batch, in float64.

    Returns idx [T,k], gate [T,k], counts [E], f [E], P [E], the scalars
    (l_aux, balance, cv, max_over_mean, min_over_mean, rank_cv,
    rank_max_over_mean) and rank_load [n_ranks].
    Pinned by its parts' pins and, whole, by the two-token hand example, the
    uniform-P and uniform-f cases and sum f = sum P = 1 on every workload recipe.
    """
    z = widen(logits, dtype)
    T, E = z.shape
    if renorm is None:
        renorm = k > 1
    p = softmax(z)
    idx = top_k(z, k)
    out = batch_statistics(expert_counts(idx, E), mean_router_prob(p), T, k, alpha, n_ranks)
    out["idx"] = idx
    out["gate"] = gates(p, idx, renorm)
    return out


def aux_loss_of_logits(z: np.ndarray, f: np.ndarray, alpha: float, grad_scale: float = 1.0) -> float:
    """g * L_aux as a function of the logits with f held fixed (f carries no gradient,
    [P1] §4.2, [P2] §2.2).  Used by the finite-difference pin of ``aux_loss_grad``;
    it composes softmax, mean_router_prob and aux_loss, each pinned on its own."""
    return grad_scale * aux_loss(f, mean_router_prob(softmax(z)), alpha)


def aux_loss_grad(logits: np.ndarray, dtype: str, f: np.ndarray, alpha: float,
                  grad_scale: float = 1.0, T: int | None = None) -> np.ndarray:
    """dL_aux/dz[t, j] = g * (alpha * N / T) * p[t, j] * (f_j - sum_i p[t, i] f_i).

    Differentiating alpha*N*sum_i f_i*(1/T)*sum_t p[t,i] through the softmax
    Jacobian dp_i/dz_j = p_i (delta_ij - p_j), with f constant.
    ``T`` is the batch size when ``logits`` holds only some of its rows.
    Pinned by: central finite differences of ``aux_loss_of_logits``; rows sum
    to zero; the uniform-p special case (alpha/T)*(f_j - 1/N).
    """
    z = widen(logits, dtype)
    E = z.shape[1]
    T = z.shape[0] if T is None else T
    p = softmax(z)
    s = (p * np.asarray(f, dtype=np.float64)[None, :]).sum(axis=1)
    return grad_scale * (alpha * E / T) * p * (f[None, :] - s[:, None])


def cv_grade(cv: float) -> str:
    """CV bands of [P3] §5.1: below 0.1 excellent, [0.1, 0.3) good, [0.3, 0.5) fair,
    0.5 and above severely imbalanced.  Pinned by: the band edges as golden cases."""
    if cv < 0.1:
        return "excellent"
    if cv < 0.3:
        return "good"
    if cv < 0.5:
        return "fair"
    return "severe"


def balance_degree(max_over_mean: float) -> float:
    """[P3] §5.1: 1 - (max load - mean load) / mean load.

    Pinned by: 1 at the mean, 0 at twice the mean, 1/4 at 1.75.
    """
    return 1.0 - (max_over_mean - 1.0)


def is_ratio_imbalanced(max_over_mean: float) -> bool:
    """[P1] §5.4: max_tokens_per_expert / mean_tokens_per_expert above 2 means imbalance.

    Pinned by: the [P1] §5.3 log line is flagged; a ratio of exactly 2 is not.
    """
    return max_over_mean > 2.0

