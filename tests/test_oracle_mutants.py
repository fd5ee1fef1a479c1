"""Plausible mistakes planted in the oracle (on the CPU) must fail a pin.

Each case monkeypatches one oracle function with a wrong variant and checks
that at least one of the pins raises.  This is what makes the pins worth
trusting: a dropped term, a wrong sign, a transposed operand or a changed
tie rule cannot slip through.
"""

import math

import numpy as np
import pytest

import oracle
import pins
import synth

R, D, S = oracle.router, oracle.dispatch, oracle.sinkhorn
X = oracle.routing_ext
B = oracle.eplb
M = oracle.taot_match


def _masked_forward(logits, dtype, k, alpha, renorm=None, n_ranks=0):
    # [P2]'s masked P_i: only the selected experts' probabilities, over T*k
    out = _orig_forward(logits, dtype, k, alpha, renorm, n_ranks)
    z = R.widen(logits, dtype)
    p = R.softmax(z)
    mask = np.zeros_like(p)
    np.put_along_axis(mask, out["idx"], 1.0, axis=1)
    out["P"] = (p * mask).sum(axis=0) / (z.shape[0] * k)
    out["balance"] = R.balance(out["f"], out["P"])
    out["l_aux"] = alpha * out["balance"]
    return out


_orig_forward = R.router_forward

MUTANTS = {
    "P masked to the selected experts": (
        [(R, "router_forward", _masked_forward)],
        [lambda: pins.check_fp_sums(R, synth), lambda: pins.check_balance_uniform_P(R)]),
    "f divided by T instead of T*k": (
        [(R, "token_fraction", lambda counts, T, k: counts / float(T))],
        [lambda: pins.check_fp_sums(R, synth)]),
    "top-k ties to the higher index": (
        [(R, "top_k", lambda z, k: (z.shape[1] - 1 - np.argsort(-z[:, ::-1], axis=1, kind="stable"))[:, :k])],
        [lambda: pins.check_topk_bruteforce(R), lambda: pins.check_top1_argmax(R)]),
    "top-k picks the smallest logits": (
        [(R, "top_k", lambda z, k: np.argsort(z, axis=1, kind="stable")[:, :k])],
        [lambda: pins.check_topk_bruteforce(R)]),
    "softmax normalised over the token axis": (
        [(R, "softmax", lambda z: np.exp(z) / np.exp(z).sum(axis=0, keepdims=True))],
        [lambda: pins.check_softmax_library(R)]),
    "balance without the factor N": (
        [(R, "balance", lambda f, P: float(np.sum(f * P)))],
        [lambda: pins.check_balance_uniform_P(R), lambda: pins.check_switch_hand_example(R)]),
    "gradient with the wrong sign": (
        [(R, "aux_loss_grad", lambda *a, **kw: -_orig_grad(*a, **kw))],
        [lambda: pins.check_grad_finite_difference(R)]),
    "gradient without the sum_i p_i f_i term": (
        [(R, "aux_loss_grad", lambda logits, dtype, f, alpha, grad_scale=1.0:
          grad_scale * (alpha * len(f) / R.widen(logits, dtype).shape[0]) * R.softmax(R.widen(logits, dtype)) * f[None, :])],
        [lambda: pins.check_grad_finite_difference(R), lambda: pins.check_grad_structure(R)]),
    "bf16 bit patterns read as IEEE half precision": (
        [(R, "widen", lambda logits, dtype: np.asarray(logits).view(np.float16).astype(np.float64)
          if dtype == "bf16" else _orig_widen(logits, dtype))],
        [lambda: pins.check_widen_library(R)]),
    "bf16 widened without the 16-bit shift": (
        [(R, "widen", lambda logits, dtype: np.asarray(logits).astype(np.uint32).view(np.float32).astype(np.float64)
          if dtype == "bf16" else _orig_widen(logits, dtype))],
        [lambda: pins.check_widen_library(R)]),
    "balance degree over the max instead of the mean": (
        [(R, "balance_degree", lambda r: 1.0 - (r - 1.0) / r)],
        [lambda: pins.check_balance_degree_hand(R)]),
    "imbalance flag at a ratio of 2 and above": (
        [(R, "is_ratio_imbalanced", lambda r: r >= 2.0)],
        [lambda: pins.check_balance_degree_hand(R), lambda: pins.check_log_example(R)]),
    "CV with the sample (n-1) deviation": (
        [(R, "load_cv", lambda x: float(np.std(np.asarray(x, float), ddof=1) / np.mean(x)))],
        [lambda: pins.check_cv_closed_forms(R)]),
    "rank loads from a strided expert mapping (e mod R)": (
        [(R, "rank_loads", lambda counts, n: np.asarray(counts).reshape(len(counts) // n, n).sum(axis=0))],
        [lambda: pins.check_rank_loads_contiguous(R), lambda: pins.check_batch_scalars_hand(R)]),
    "max/min over mean divided by T instead of T*k": (
        [(R, "batch_statistics", lambda *a, **kw: _stats_over_T(*a, **kw))],
        [lambda: pins.check_batch_scalars_hand(R), lambda: pins.check_log_example(R)]),
    "rank max/mean over the per-expert mean": (
        [(R, "batch_statistics", lambda *a, **kw: _stats_rank_mean_per_expert(*a, **kw))],
        [lambda: pins.check_batch_scalars_hand(R)]),
    "rank CV with the sample (n-1) deviation": (
        [(R, "batch_statistics", lambda *a, **kw: _stats_rank_cv_ddof1(*a, **kw))],
        [lambda: pins.check_batch_scalars_hand(R)]),
    "dispatch keeps the last C instead of the first": (
        [(D, "dispatch", lambda idx, E, C: _reverse_dispatch(idx, E, C))],
        [lambda: pins.check_dispatch_bruteforce(D, R)]),
    "dispatch keeps C + 1": (
        [(D, "dispatch", lambda idx, E, C: _orig_dispatch(idx, E, C + 1))],
        [lambda: pins.check_dispatch_bruteforce(D, R)]),
    "capacity floors the per-expert share": (
        [(D, "capacity", lambda T, k, E, cf: int(math.ceil((T * k // E) * cf)))],
        [lambda: pins.check_dispatch_bruteforce(D, R), lambda: _capacity_ragged()]),
    "Sinkhorn uses M^T where M belongs": (
        [(S, "sinkhorn_knopp", lambda a, b, M, iters: _orig_sk(a, b, M.T.copy(), iters))],
        [lambda: pins.check_sinkhorn_dual(S)]),
    "Sinkhorn kernel exp(-W * eps)": (
        [(S, "gibbs_kernel", lambda W, eps: np.exp(-W * float(eps)))],
        [lambda: pins.check_sinkhorn_topology_kernel(S)]),
    "supply and demand swapped": (
        [(S, "supply_demand", lambda load: _orig_sd(load)[1::-1] + (_orig_sd(load)[2],))],
        [lambda: pins.check_supply_demand_hand(S), lambda: pins.check_sinkhorn_marginals(S, _loads()),
         lambda: pins.check_sinkhorn_two_rank(S)]),
    "supply and demand left unnormalised": (
        [(S, "supply_demand", lambda load: _unnormalised_sd(load))],
        [lambda: pins.check_supply_demand_hand(S)]),
    "cross-node cost and intra-node cost swapped": (
        [(S, "topology_cost", lambda R_, rpn, lam: np.where(_orig_tc(R_, rpn, lam) == 1.0, lam, np.where(_orig_tc(R_, rpn, lam) == lam, 1.0, 0.0)))],
        [lambda: pins.check_topology_cost_hand(S), lambda: pins.check_sinkhorn_topology_kernel(S)]),
    "topology cost 1 on the diagonal (a rank's own slot priced as intra-node)": (
        [(S, "topology_cost", lambda R_, rpn, lam: np.where(np.eye(R_, dtype=bool), 1.0, _orig_tc(R_, rpn, lam)))],
        [lambda: pins.check_topology_cost_hand(S)]),
    "bias added in float64 instead of fp32": (
        [(X, "selection_scores", lambda logits, dtype, bias: R.widen(logits, dtype) + np.asarray(bias, np.float64)[None, :])],
        [lambda: pins.check_biased_sum_is_fp32(X)]),
    "bias subtracted from the logits": (
        [(X, "selection_scores", lambda logits, dtype, bias: _orig_sel(logits, dtype, -np.asarray(bias, np.float32)))],
        [lambda: pins.check_biased_topk_bruteforce(X), lambda: pins.check_biased_topk_dominant(X)]),
    "softmax and gates taken on the biased scores": (
        [(X, "router_forward_ex", lambda *a, **kw: _softmax_on_biased(*a, **kw))],
        [lambda: pins.check_forward_ex_reductions(X, R)]),
    "bias update with the wrong sign": (
        [(X, "bias_update", lambda bias, counts, T, k, gamma: _orig_bu(bias, counts, T, k, -gamma))],
        [lambda: pins.check_bias_update_hand(X), lambda: pins.check_bias_update_balances(X, R)]),
    "bias update against the floor of the mean": (
        [(X, "bias_update", lambda bias, counts, T, k, gamma: (np.asarray(bias, np.float32) + np.float32(gamma) * np.sign(
            (T * k) // len(counts) - np.asarray(counts)).astype(np.float32)).astype(np.float32))],
        [lambda: pins.check_bias_update_hand(X)]),
    "masked P divided by T instead of T*k": (
        [(X, "mean_router_prob_masked", lambda p, idx, k: (p * X.pick_mask(idx, p.shape[1])).sum(axis=0) / p.shape[0])],
        [lambda: pins.check_masked_p_closed_forms(X, R)]),
    "renormalised gate gradient without the p/S^2 term": (
        [(X, "grad_wrt_probs", lambda *a: _no_quotient_term(*a))],
        [lambda: pins.check_grad_wrt_probs_finite_difference(X, R), lambda: pins.check_full_grad_finite_difference(X, R)]),
    "masked aux gradient without the mask": (
        [(X, "grad_wrt_probs", lambda p, idx, f, a, g, T, k, dg, rn, masked: _orig_gwp(p, idx, f, a, g * (1.0 / k if masked else 1.0), T, k, dg, rn, False))],
        [lambda: pins.check_grad_wrt_probs_finite_difference(X, R), lambda: pins.check_full_grad_finite_difference(X, R)]),
    "softmax backward without the row-sum term": (
        [(X, "softmax_backward", lambda p, dp: p * dp)],
        [lambda: pins.check_softmax_backward_autograd(X), lambda: pins.check_full_grad_finite_difference(X, R),
         lambda: pins.check_full_grad_structure(X, R)]),
    "softmax backward with the row sum of dp instead of p*dp": (
        [(X, "softmax_backward", lambda p, dp: p * (dp - dp.sum(axis=1, keepdims=True)))],
        [lambda: pins.check_softmax_backward_autograd(X)]),
    "packing takes the lightest item first": (
        [(B, "balanced_packing", lambda w, n: _orig_bp([-x for x in w], n)[:2] + (_totals(w, *_orig_bp([-x for x in w], n)[:2], n),))],
        [lambda: pins.check_packing_worked_example(B)]),
    "packing ignores the bins' capacity": (
        [(B, "balanced_packing", lambda w, n: _uncapped_packing(w, n))],
        [lambda: pins.check_packing_cardinality_and_mass(B), lambda: pins.check_packing_worked_example(B)]),
    "replication by weight instead of weight per copy": (
        [(B, "replicate_experts", lambda w, n: _by_weight(w, n))],
        [lambda: pins.check_replication_bruteforce(B), lambda: pins.check_replication_hand_case(B)]),
    "replication ties to the higher index": (
        [(B, "replicate_experts", lambda w, n: _ties_high(w, n))],
        [lambda: pins.check_replication_hand_case(B)]),
    "residual imbalance over the max instead of the mean": (
        [(M, "residual_imbalance", lambda rl: float((np.max(rl) - np.mean(rl)) / np.max(rl)))],
        [lambda: pins.check_residual_imbalance_hand(M)]),
    "matching ignores the topology": (
        [(M, "match", lambda w, plan, R, ranks_per_node, K: _orig_match(w, plan, R, R, K))],
        [lambda: pins.check_match_hand_arbitration(M)]),
    "matching stops after K rounds": (
        [(M, "match", lambda w, plan, R, ranks_per_node, K: _k_rounds_match(w, plan, R, ranks_per_node, K))],
        [lambda: pins.check_match_column_first_claim(M, S), lambda: pins.check_match_hand_arbitration(M)]),
    "matching prefers the smaller flow": (
        [(M, "match", lambda w, plan, R, ranks_per_node, K: _orig_match(w, -np.asarray(plan), R, ranks_per_node, K))],
        [lambda: pins.check_match_hand_arbitration(M)]),
}

_orig_match = M.match


def _k_rounds_match(w, plan, R, rpn, K):
    """The matching cut to exactly K rounds (a rank that lost does not get its slot back)."""
    w = [int(x) for x in w]
    E = len(w)
    per = E // R
    load = [sum(w[r * per:(r + 1) * per]) for r in range(R)]
    total = sum(load)
    w_rem, used, n = list(w), set(), [0] * R
    se, st = np.full((R, K), -1), np.zeros((R, K), np.int64)
    P = np.asarray(plan, np.float32)

    def mv(c, e):
        h = e // per
        if load[h] * R <= total or load[c] * R >= total or (c, e) in used or w_rem[e] <= 0:
            return 0
        return max(0, min(w_rem[e], (load[h] * R - total) // R, (total - load[c] * R) // R))

    for _ in range(K):
        ch = {}
        for c in range(R):
            if n[c] >= K:
                continue
            best = None
            for e in range(E):
                x = mv(c, e)
                if x > 0:
                    sc = (x, 1 if (e // per) // rpn == c // rpn else 0, float(P[e // per, c]))
                    if best is None or sc > best[0]:
                        best = (sc, e)
            if best:
                ch[c] = best
        win = {}
        for c in sorted(ch):
            sc, e = ch[c]
            if e not in win or sc > win[e][0]:
                win[e] = (sc, c)
        for c in sorted(c for _, c in win.values()):
            e = ch[c][1]
            x = mv(c, e)
            if x > 0:
                load[e // per] -= x
                load[c] += x
                w_rem[e] -= x
                used.add((c, e))
                se[c, n[c]], st[c, n[c]] = e, x
                n[c] += 1
    return {"slot_expert": se, "slot_tokens": st, "rank_load": np.asarray(load), "moved": int(st.sum())}
_orig_pg = B.plan_global
_orig_bp = B.balanced_packing


def _totals(w, bins, pos, n):
    t = np.zeros(n)
    for i, b in enumerate(bins):
        t[b] += w[i]
    return t


def _uncapped_packing(w, n):
    order = sorted(range(len(w)), key=lambda i: (-w[i], i))
    t, fill, bins, pos = [0.0] * n, [0] * n, [0] * len(w), [0] * len(w)
    for i in order:
        b = min(range(n), key=lambda j: (t[j], j))
        bins[i], pos[i] = b, fill[b]
        fill[b] += 1
        t[b] += w[i]
    return np.asarray(bins), np.asarray(pos), np.asarray(t)


def _by_weight(w, num_phys):
    E = len(w)
    count, p2l = [1] * E, list(range(E))
    for _ in range(num_phys - E):
        best = max(range(E), key=lambda e: (w[e], -e))
        count[best] += 1
        p2l.append(best)
    return np.asarray(p2l), np.asarray(count)


def _ties_high(w, num_phys):
    E = len(w)
    count, p2l = [1] * E, list(range(E))
    for _ in range(num_phys - E):
        best = 0
        for e in range(1, E):
            if w[e] * count[best] >= w[best] * count[e]:
                best = e
        count[best] += 1
        p2l.append(best)
    return np.asarray(p2l), np.asarray(count)


_orig_sel = X.selection_scores
_orig_fwd_ex = X.router_forward_ex


def _softmax_on_biased(logits, dtype, k, alpha, renorm=None, n_ranks=0, bias=None, masked_p=False, gamma=None):
    if bias is None:
        return _orig_fwd_ex(logits, dtype, k, alpha, renorm, n_ranks, bias, masked_p, gamma)
    s = X.selection_scores(logits, dtype, bias)             # the biased scores feed the softmax too
    return _orig_fwd_ex(s, "fp32", k, alpha, renorm, n_ranks, np.zeros_like(np.asarray(bias, np.float32)),
                        masked_p, gamma)
_orig_bu = X.bias_update
_orig_gwp = X.grad_wrt_probs


def _no_quotient_term(p, idx, f, alpha, grad_scale, T, k, dgate, renorm, masked_p):
    dp = _orig_gwp(p, idx, f, alpha, grad_scale, T, k, None, renorm, masked_p)
    if dgate is not None:
        rows = np.arange(p.shape[0])
        S = np.take_along_axis(p, idx, axis=1).sum(axis=1) if renorm else 1.0
        for j in range(idx.shape[1]):
            dp[rows, idx[:, j]] += dgate[:, j] / S
    return dp


_orig_grad = R.aux_loss_grad
_orig_widen = R.widen
_orig_dispatch = D.dispatch
_orig_sk = S.sinkhorn_knopp
_orig_sd = S.supply_demand
_orig_tc = S.topology_cost


def _unnormalised_sd(load):
    a, b, ok = _orig_sd(load)
    load = np.asarray(load, dtype=np.float64)
    mean = load.mean()
    return (np.maximum(load - mean, 0.0), np.maximum(mean - load, 0.0), ok)


_orig_stats = R.batch_statistics


def _stats_over_T(counts, P, T, k, alpha, n_ranks=0):
    out = _orig_stats(counts, P, T, k, alpha, n_ranks)
    out["max_over_mean"] = counts.max() / (T / len(counts))
    out["min_over_mean"] = counts.min() / (T / len(counts))
    return out


def _stats_rank_mean_per_expert(counts, P, T, k, alpha, n_ranks=0):
    out = _orig_stats(counts, P, T, k, alpha, n_ranks)
    if n_ranks > 0:
        out["rank_max_over_mean"] = out["rank_load"].max() / (T * k / len(counts))
    return out


def _stats_rank_cv_ddof1(counts, P, T, k, alpha, n_ranks=0):
    out = _orig_stats(counts, P, T, k, alpha, n_ranks)
    if n_ranks > 0:
        rl = np.asarray(out["rank_load"], dtype=np.float64)
        out["rank_cv"] = float(rl.std(ddof=1) / rl.mean())
    return out


def _reverse_dispatch(idx, E, C):
    out = _orig_dispatch(idx, E, C)
    counts = out["counts"]
    slot = np.full_like(out["slot"], -1)
    for e in range(E):
        seg = out["perm"][out["offsets"][e]:out["offsets"][e + 1]]
        for r, a in enumerate(seg[::-1]):
            slot[a] = r if r < C else -1
        out["perm"][out["offsets"][e]:out["offsets"][e + 1]] = seg[::-1]
    out["slot"] = slot
    out["counts"] = counts
    return out


def _capacity_ragged():
    # T*k/E not an integer: 10 tokens, 4 experts, k=1, factor 1.0 -> ceil(2.5) = 3
    assert D.capacity(10, 1, 4, 1.0) == 3


def _loads():
    rng = np.random.default_rng(3)
    loads = rng.poisson(384, size=(6, 64)).astype(np.float64)
    loads[1, :8] += 600.0
    return loads


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    patches, checks = MUTANTS[name]
    for mod, attr, fn in patches:
        monkeypatch.setattr(mod, attr, fn)
    caught = 0
    for check in checks:
        try:
            check()
        except AssertionError:
            caught += 1
    assert caught > 0, f"no pin caught the planted mistake: {name}"


def test_unmutated_oracle_passes_the_same_checks():
    for _, checks in MUTANTS.values():
        for check in checks:
            check()
