"""Oracle: the router's next steps -- aux-loss-free bias routing, the masked
P_i variant, and the full router backward through the gates.

TEST INFRASTRUCTURE (see the package docstring): plain float64 numpy, except
where a decision is taken in fp32 on purpose (stated below).

Readings where the pages are silent:

  * Bias routing ([P1] §4.3).  Every expert i has one scalar bias b_i,
    initialised to 0, added to its router logit.  The page says the bias
    steers which experts get *selected* and that no loss term is added; it
    gives the direction of the update (an overloaded expert's b_i goes down,
    an idle one's goes up) but no rule.  This build reads it as follows.
      - Selection ranks s[t, i] = fp32(z[t, i]) + b_i, added in fp32 and
        rounded to nearest: the selection is an integer decision, so both
        sides take it in the same (the kernel's) precision.  Ties go to the
        lower expert index, as for plain top-k.
      - Softmax, gates, P and the aux-loss gradient use the unbiased z: the
        bias moves selection only and carries no gradient.
      - After a batch, b_i <- b_i + gamma * sign(mean - count_i), with
        mean = T*k/E, sign(0) = 0, in fp32 (one rounding).  The comparison
        is exact: it is taken as count_i * E against T * k in integers.
  * Masked P ([P2] §3.1 and the code of [P1] §4.4):
        P_i = (1/(T*k)) * sum_t p[t, i] * [expert i is one of t's picks].
    The unmasked P_i of [P1] §4.2 stays the default; this is a flag.
  * Full backward.  The upstream gradient of the main loss arrives as
    dgate[t, j] = dL_main/dgate[t, j] for the k gates of each token; the
    picks are held fixed (top-k is piecewise constant in z).  The gradient
    flows through the gate (p itself, or p renormalised over the picks) and
    the softmax, and is added to the aux-loss gradient.
"""

from __future__ import annotations

import numpy as np

from . import router as R


def selection_scores(logits: np.ndarray, dtype: str, bias: np.ndarray) -> np.ndarray:
    """s[t, i] = z[t, i] + b_i, added in fp32 ([P1] §4.3: the bias sits on the logits).

    The logits widen exactly to fp32 (bf16 and fp32 inputs both do); the sum
    is one fp32 addition, rounded to nearest even.
    Pinned by: 1 + 2^-24 rounds to 1 (a tie the lower expert wins), 1 + 2^-23
    does not; brute-force top-k of z + b on integer inputs.
    """
    z32 = R.widen(logits, dtype).astype(np.float32)
    b32 = np.asarray(bias, dtype=np.float32)
    return z32 + b32[None, :]


def top_k_biased(logits: np.ndarray, dtype: str, bias: np.ndarray, k: int) -> np.ndarray:
    """The k experts of largest biased score per row, largest first, ties to the lower index.

    [P1] §4.3 (the bias changes which experts are picked), [P1] §4.4 (top-k).
    Pinned by: brute-force enumeration of k-subsets on tiny integer inputs;
    a zero bias gives plain top-k; a dominant bias forces its expert in.
    """
    s = selection_scores(logits, dtype, bias).astype(np.float64)
    return R.top_k(s, k)


def bias_update(bias: np.ndarray, counts: np.ndarray, T: int, k: int, gamma: float) -> np.ndarray:
    """b_i + gamma * sign(T*k/E - count_i) in fp32 ([P1] §4.3: an overloaded
    expert's bias goes down, an idle one's goes up; the step size gamma is the
    caller's).

    Pinned by: a hand case with an expert exactly at the mean (no change);
    repeated routing + update lowers the load CV of a skewed batch.
    """
    counts = np.asarray(counts, dtype=np.int64)
    E = len(counts)
    total = int(T) * int(k)
    direction = np.sign(total - counts * E).astype(np.float32)   # sign(mean - count), exact
    step = np.float32(gamma) * direction                         # +-gamma or 0, exact
    return (np.asarray(bias, dtype=np.float32) + step).astype(np.float32)


def pick_mask(idx: np.ndarray, E: int) -> np.ndarray:
    """m[t, i] = 1 if expert i is one of token t's picks, else 0.

    Pinned by: the masked-P hand case and the k == E closed form, which go through it.
    """
    m = np.zeros((idx.shape[0], E), dtype=np.float64)
    np.put_along_axis(m, np.asarray(idx), 1.0, axis=1)
    return m


def mean_router_prob_masked(p: np.ndarray, idx: np.ndarray, k: int) -> np.ndarray:
    """P_i = (1/(T*k)) sum_t p[t, i] m[t, i] -- the masked reading of [P2] §3.1 / [P1] §4.4.

    Pinned by: k == E (every expert picked) gives the unmasked P_i / k;
    a per-token loop on small inputs.
    """
    T, E = p.shape
    return (p * pick_mask(idx, E)).sum(axis=0) / float(T * k)


def router_forward_ex(logits: np.ndarray, dtype: str, k: int, alpha: float,
                      renorm: bool | None = None, n_ranks: int = 0,
                      bias: np.ndarray | None = None, masked_p: bool = False,
                      gamma: float | None = None) -> dict:
    """The router forward with the optional bias selection and masked P.

    Same outputs as ``router.router_forward``; with ``gamma`` also
    ``bias_out`` = ``bias_update(bias, counts, T, k, gamma)``.
    Pinned by: a zero bias with unmasked P reproduces router.router_forward
    exactly; with a bias P and the gates stay those of the unbiased softmax
    ([P1] §4.3: the bias moves the choice only); the masked-P hand case.
    """
    z = R.widen(logits, dtype)
    T, E = z.shape
    if renorm is None:
        renorm = k > 1
    b = np.zeros(E, np.float32) if bias is None else np.asarray(bias, np.float32)
    p = R.softmax(z)
    idx = top_k_biased(logits, dtype, b, k)
    counts = R.expert_counts(idx, E)
    P = mean_router_prob_masked(p, idx, k) if masked_p else R.mean_router_prob(p)
    out = R.batch_statistics(counts, P, T, k, alpha, n_ranks)
    out["idx"] = idx
    out["gate"] = R.gates(p, idx, renorm)
    if gamma is not None:
        out["bias_out"] = bias_update(b, counts, T, k, gamma)
    return out


def grad_wrt_probs(p: np.ndarray, idx: np.ndarray, f: np.ndarray, alpha: float, grad_scale: float,
                   T: int, k: int, dgate: np.ndarray | None, renorm: bool, masked_p: bool) -> np.ndarray:
    """dL/dp[t, i] of L = sum_{t,j} dgate[t,j] * gate[t,j] + grad_scale * L_aux, picks fixed.

    Aux part ([P1] §4.2, f constant): grad_scale * alpha * E * f_i * dP_i/dp[t,i],
    with dP_i/dp[t,i] = 1/T (unmasked) or m[t,i]/(T*k) (masked).
    Gate part: gate_j = p[t, i_j] (no renormalisation) or p[t, i_j] / S_t with
    S_t = sum_m p[t, i_m]; by the quotient rule
        d gate_j / d p[t, i_m] = [j == m] / S_t - p[t, i_j] / S_t^2.
    Pinned by: central differences in p of the gate and aux terms (picks fixed),
    for plain and renormalised gates, with masked and unmasked P.
    """
    E = p.shape[1]
    f = np.asarray(f, dtype=np.float64)
    if masked_p:
        dp = grad_scale * alpha * E * f[None, :] * pick_mask(idx, E) / float(T * k)
    else:
        dp = np.broadcast_to(grad_scale * alpha * E * f[None, :] / float(T), p.shape).copy()
    if dgate is not None:
        dg = np.asarray(dgate, dtype=np.float64)
        rows = np.arange(p.shape[0])
        picked = np.take_along_axis(p, idx, axis=1)                  # p[t, i_j]
        if renorm:
            S = picked.sum(axis=1)
            for j in range(idx.shape[1]):
                for m in range(idx.shape[1]):
                    d = (1.0 / S if j == m else 0.0) - picked[:, j] / S ** 2
                    dp[rows, idx[:, m]] += dg[:, j] * d
        else:
            for j in range(idx.shape[1]):
                dp[rows, idx[:, j]] += dg[:, j]
    return dp


def softmax_backward(p: np.ndarray, dp: np.ndarray) -> np.ndarray:
    """dz[t, j] = sum_i dp[t, i] * p[t, i] * (delta_ij - p[t, j]) (the softmax Jacobian).

    Pinned by: torch autograd through torch.softmax in float64 (random rows and
    a saturated one).
    """
    return p * (dp - (p * dp).sum(axis=1, keepdims=True))


def router_backward_full(logits: np.ndarray, dtype: str, f: np.ndarray, alpha: float,
                         grad_scale: float, idx: np.ndarray, dgate: np.ndarray | None,
                         renorm: bool, masked_p: bool = False, T: int | None = None) -> np.ndarray:
    """dL/dz for L = sum_{t,j} dgate[t,j] * gate[t,j](z) + grad_scale * L_aux(z).

    ``T`` is the batch size when ``logits`` holds only some of its rows.
    Pinned by: central finite differences of ``full_loss_of_logits`` (picks
    frozen); rows sum to zero; dgate = None and unmasked P give
    ``router.aux_loss_grad``; with renormalised gates the gate part vanishes
    on the unpicked experts.
    """
    z = R.widen(logits, dtype)
    T = z.shape[0] if T is None else T
    k = idx.shape[1]
    p = R.softmax(z)
    dp = grad_wrt_probs(p, idx, f, alpha, grad_scale, T, k, dgate, renorm, masked_p)
    return softmax_backward(p, dp)


def full_loss_of_logits(z: np.ndarray, f: np.ndarray, alpha: float, grad_scale: float,
                        idx: np.ndarray, dgate: np.ndarray | None, renorm: bool,
                        masked_p: bool = False) -> float:
    """sum_{t,j} dgate[t,j] * gate[t,j](z) + grad_scale * alpha * E * sum_i f_i P_i(z),
    picks and f held fixed.  Used by the finite-difference pin of ``router_backward_full``;
    it composes softmax, gates and the (masked) P, each pinned on its own."""
    T, E = z.shape
    k = idx.shape[1]
    p = R.softmax(z)
    P = mean_router_prob_masked(p, idx, k) if masked_p else R.mean_router_prob(p)
    loss = grad_scale * R.aux_loss(np.asarray(f, np.float64), P, alpha)
    if dgate is not None:
        loss += float((np.asarray(dgate, np.float64) * R.gates(p, idx, renorm)).sum())
    return loss
