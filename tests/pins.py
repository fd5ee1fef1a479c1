"""Pins for the CPU oracle: checks against what the pages and the mathematics fix.

Each ``check_*`` takes the oracle module(s) as arguments and raises
AssertionError on a mismatch, so the same check can be run on the oracle
(``test_oracle_*.py``: must pass) and on copies of it with a planted mistake
(``test_oracle_mutants.py``: must fail).  None of these checks re-types the
oracle's own formula: each compares against an independent route (a library
routine, a brute force, a closed form, an invariant or a worked example from
the pages).
"""

from __future__ import annotations

import itertools
import json
import math
from pathlib import Path

import numpy as np

GOLDEN = Path(__file__).resolve().parent / "golden"


def golden(name: str) -> dict:
    return json.loads((GOLDEN / name).read_text())


# ----------------------------------------------------------------------------- router

def check_softmax_library(router) -> None:
    """softmax equals scipy.special.softmax and is shift invariant."""
    from scipy.special import softmax as sp_softmax
    rng = np.random.default_rng(11)
    z = rng.standard_normal((40, 13)) * 3.0
    p = router.softmax(z)
    np.testing.assert_allclose(p, sp_softmax(z, axis=1), rtol=1e-13, atol=0)
    np.testing.assert_allclose(router.softmax(z + 7.25), p, rtol=1e-12, atol=0)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=1e-14)


def _brute_topk_row(z: np.ndarray, k: int) -> list[int]:
    """The unique k-subset whose members all precede every non-member under
    (larger logit first, then lower index), listed in that order."""
    E = len(z)

    def before(i: int, j: int) -> bool:
        return z[i] > z[j] or (z[i] == z[j] and i < j)

    winners = [S for S in itertools.combinations(range(E), k)
               if all(before(i, j) for i in S for j in range(E) if j not in S)]
    assert len(winners) == 1
    return sorted(winners[0], key=lambda i: (-z[i], i))


def check_topk_bruteforce(router) -> None:
    """top_k equals brute-force enumeration of k-subsets, with many ties."""
    rng = np.random.default_rng(12)
    for E in range(1, 8):
        for k in range(1, min(E, 3) + 1):
            z = rng.integers(0, 3, size=(25, E)).astype(np.float64)   # ties everywhere
            z[:3] = rng.standard_normal((3, E))                        # and a few without
            got = router.top_k(z, k)
            for t in range(z.shape[0]):
                assert list(got[t]) == _brute_topk_row(z[t], k), (E, k, t, z[t], got[t])


def check_top1_argmax(router) -> None:
    """k = 1 reduces to numpy.argmax (first maximum on ties)."""
    rng = np.random.default_rng(13)
    z = rng.integers(0, 4, size=(200, 9)).astype(np.float64)
    np.testing.assert_array_equal(router.top_k(z, 1)[:, 0], np.argmax(z, axis=1))


def check_gate_hand_example(router) -> None:
    """z = [0, ln 3] gives p = [1/4, 3/4]: the top-1 gate is 3/4; a top-2
    renormalised gate is [3/4, 1/4] (the picks already hold all the mass)."""
    z = np.array([[0.0, math.log(3.0)]])
    p = router.softmax(z)
    idx1 = router.top_k(z, 1)
    assert idx1[0, 0] == 1
    np.testing.assert_allclose(router.gates(p, idx1, renorm=False), [[0.75]], rtol=1e-15)
    idx2 = router.top_k(z, 2)
    np.testing.assert_allclose(router.gates(p, idx2, renorm=True), [[0.75, 0.25]], rtol=1e-15)
    z3 = np.array([[math.log(2.0), 0.0, math.log(6.0)]])      # p = [2, 1, 6] / 9
    p3 = router.softmax(z3)
    np.testing.assert_allclose(router.gates(p3, router.top_k(z3, 2), renorm=True), [[0.75, 0.25]], rtol=1e-14)
    np.testing.assert_allclose(router.gates(p3, router.top_k(z3, 2), renorm=False), [[6 / 9, 2 / 9]], rtol=1e-14)


def check_counts_bruteforce(router) -> None:
    """bincount with minlength equals a plain loop; unused experts report 0."""
    rng = np.random.default_rng(14)
    idx = rng.integers(0, 5, size=(30, 2))
    E = 9
    want = [0] * E
    for e in idx.ravel():
        want[int(e)] += 1
    got = router.expert_counts(idx, E)
    assert list(got) == want and got[5:].sum() == 0


def check_fp_sums(router, synth) -> None:
    """sum_i f_i = 1 and sum_i P_i = 1 ([P1] §5.3) on every workload recipe."""
    for w in synth.ROUTER_WORKLOADS.values():
        small = w.with_tokens(257)
        out = router.router_forward(synth.router_logits(small), small.dtype, small.k, small.alpha,
                                    n_ranks=small.n_ranks)
        assert out["counts"].sum() == small.T * small.k
        assert abs(out["f"].sum() - 1.0) < 1e-12, out["f"].sum()
        assert abs(out["P"].sum() - 1.0) < 1e-12, out["P"].sum()


def check_balance_uniform_P(router) -> None:
    """Equal logits in every row: P_i = 1/N, so N * sum f_i P_i = 1 for any f ([P2] §2.2)."""
    rng = np.random.default_rng(15)
    T, E, k = 64, 6, 2
    z = np.repeat(rng.standard_normal((T, 1)), E, axis=1)
    out = router.router_forward(z.astype(np.float32), "fp32", k, alpha=0.01)
    np.testing.assert_allclose(out["P"], 1.0 / E, rtol=1e-14)
    assert abs(out["balance"] - 1.0) < 1e-13 and abs(out["l_aux"] - 0.01) < 1e-15


def check_balance_uniform_f(router) -> None:
    """Token t forced to expert t mod N (top-1): f_i = 1/N, so the balance is 1 for any P."""
    rng = np.random.default_rng(16)
    T, E = 96, 8
    z = rng.standard_normal((T, E))
    z[np.arange(T), np.arange(T) % E] += 20.0
    out = router.router_forward(z.astype(np.float32), "fp32", 1, alpha=0.5)
    np.testing.assert_allclose(out["f"], 1.0 / E, rtol=0)
    assert abs(out["balance"] - 1.0) < 1e-13 and abs(out["l_aux"] - 0.5) < 1e-13


def check_switch_hand_example(router) -> None:
    """Two tokens, two experts, top-1, worked by hand.

    z0 = [ln 3, 0] -> p0 = [3/4, 1/4], expert 0; z1 = [0, 0] -> p1 = [1/2, 1/2],
    a tie, expert 0.  counts = [2, 0], f = [1, 0], P = [5/8, 3/8];
    N * sum f P = 2 * 5/8 = 5/4; with alpha = 0.01, L_aux = 0.0125.
    """
    z = np.array([[math.log(3.0), 0.0], [0.0, 0.0]])
    out = router.router_forward(z, "fp32", 1, alpha=0.01)  # ln 3 rounds to fp32 first
    z32 = z.astype(np.float32).astype(np.float64)
    p00 = math.exp(z32[0, 0]) / (math.exp(z32[0, 0]) + 1.0)
    assert list(out["idx"][:, 0]) == [0, 0] and list(out["counts"]) == [2, 0]
    np.testing.assert_allclose(out["P"], [(p00 + 0.5) / 2, (1 - p00 + 0.5) / 2], rtol=1e-15)
    assert abs(out["balance"] - 2 * (p00 + 0.5) / 2) < 1e-15
    assert abs(out["balance"] - 1.25) < 1e-7 and abs(out["l_aux"] - 0.0125) < 1e-9


def check_cv_closed_forms(router) -> None:
    """Population CV on crafted load vectors."""
    assert router.load_cv(np.array([1, 3])) == 0.5                       # mean 2, std 1
    assert router.load_cv(np.array([4, 4, 4, 4])) == 0.0
    assert abs(router.load_cv(np.array([0, 0, 0, 4])) - math.sqrt(3.0)) < 1e-15   # mean 1, var 3
    assert abs(router.load_cv(np.array([2, 4, 4, 4, 5, 5, 7, 9])) - 2.0 / 5.0) < 1e-15  # std 2, mean 5


def check_log_example(router) -> None:
    """[P1] §5.3's log line: 8192 tokens over 8 experts, expert 3 receiving
    4320 and expert 7 receiving 312; [P1] §5.4 calls max/mean above 2
    imbalanced.  The oracle's batch statistics of a count vector with those
    entries (top-1, the other six experts sharing the rest) must give the
    printed max/mean and 312 over the mean of 1024 as min/mean."""
    g = golden("p1_s5_3_tokens_per_expert_log.json")
    E, T = g["num_experts"], g["total_tokens"]
    counts = np.zeros(E, dtype=np.int64)
    counts[3], counts[7] = g["max_expert_tokens"], g["min_expert_tokens_shown"]
    rest = T - counts[3] - counts[7]
    others = [e for e in range(E) if e not in (3, 7)]
    for i, e in enumerate(others):                    # 593 or 594 each: all above 312, below 4320
        counts[e] = rest // len(others) + (1 if i < rest % len(others) else 0)
    assert counts.sum() == T
    out = router.batch_statistics(counts, np.full(E, 1.0 / E), T, 1, 0.01)
    assert out["max_over_mean"] == g["max_over_mean"], out["max_over_mean"]
    assert out["min_over_mean"] == g["min_expert_tokens_shown"] / (T / E), out["min_over_mean"]
    assert router.is_ratio_imbalanced(out["max_over_mean"])
    assert not router.is_ratio_imbalanced(1.9)


def check_rank_loads_contiguous(router) -> None:
    """A rank's load is the tokens routed to the experts it hosts ([P4]
    introduction), the experts laid out contiguously: with 12 experts on 4
    ranks, rank 0 hosts experts 0-2, rank 1 experts 3-5, and so on.  Worked
    by hand for counts 1..12: 1+2+3, 4+5+6, 7+8+9, 10+11+12.  One expert per
    rank gives the counts back, one rank gives the total."""
    counts = np.arange(1, 13, dtype=np.int64)
    assert list(router.rank_loads(counts, 4)) == [6, 15, 24, 33]
    assert list(router.rank_loads(counts, 2)) == [21, 57]
    assert list(router.rank_loads(counts, 12)) == list(counts)
    assert list(router.rank_loads(counts, 1)) == [78]


def check_batch_scalars_hand(router) -> None:
    """The scalars of batch_statistics on a case worked by hand.

    T = 6 tokens, top-2, E = 4 experts, counts [6, 3, 2, 1] (12 = T*k
    assignments, mean 3 per expert): max/mean = 6/3 = 2, min/mean = 1/3
    ([P3] §5.1: max load over mean load), CV = pop-std / mean with
    std = sqrt(((6-3)^2 + 0 + 1 + 4) / 4) = sqrt(14)/2.  On 2 EP ranks the
    loads are [9, 3] (experts 0-1, 2-3), mean 6: rank max/mean = 1.5 and
    rank CV = 3/6 = 0.5 (population std 3).  With P uniform the balance is
    E * sum f/E = 1 and L_aux = alpha.
    """
    counts = np.array([6, 3, 2, 1], dtype=np.int64)
    out = router.batch_statistics(counts, np.full(4, 0.25), 6, 2, alpha=0.5, n_ranks=2)
    assert out["max_over_mean"] == 2.0, out["max_over_mean"]
    assert abs(out["min_over_mean"] - 1.0 / 3.0) < 1e-15, out["min_over_mean"]
    assert abs(out["cv"] - math.sqrt(14.0) / 2.0 / 3.0) < 1e-15, out["cv"]
    assert list(out["rank_load"]) == [9, 3]
    assert out["rank_max_over_mean"] == 1.5, out["rank_max_over_mean"]
    assert abs(out["rank_cv"] - 0.5) < 1e-15, out["rank_cv"]
    assert abs(out["balance"] - 1.0) < 1e-15 and abs(out["l_aux"] - 0.5) < 1e-15
    np.testing.assert_array_equal(out["f"], counts / 12.0)
    # no ranks: the rank outputs stay empty / zero
    out0 = router.batch_statistics(counts, np.full(4, 0.25), 6, 2, alpha=0.5, n_ranks=0)
    assert len(out0["rank_load"]) == 0 and out0["rank_cv"] == 0.0 and out0["rank_max_over_mean"] == 0.0


def check_cv_grades(router) -> None:
    """The CV bands of [P3] §5.1."""
    g = golden("p3_s5_1_cv_bands.json")
    for cv, label in g["cases"]:
        assert router.cv_grade(cv) == label, (cv, label)


def check_grad_finite_difference(router) -> None:
    """Central differences of g * L_aux(z) with f frozen match the closed form."""
    rng = np.random.default_rng(17)
    T, E, alpha, g = 5, 6, 0.3, 1.7
    z32 = rng.standard_normal((T, E)).astype(np.float32)
    z = z32.astype(np.float64)
    f = rng.random(E)
    f /= f.sum()
    grad = router.aux_loss_grad(z32, "fp32", f, alpha, grad_scale=g)
    h = 1e-6
    fd = np.zeros_like(z)
    for t in range(T):
        for j in range(E):
            zp, zm = z.copy(), z.copy()
            zp[t, j] += h
            zm[t, j] -= h
            fd[t, j] = (router.aux_loss_of_logits(zp, f, alpha, g) - router.aux_loss_of_logits(zm, f, alpha, g)) / (2 * h)
    scale = np.abs(grad).max()
    assert np.abs(grad - fd).max() <= 1e-7 * scale, np.abs(grad - fd).max() / scale


def check_grad_structure(router) -> None:
    """Rows of dL/dz sum to 0 (softmax shift invariance); equal logits give
    g * (alpha / T) * (f_j - 1/N)."""
    rng = np.random.default_rng(18)
    T, E, alpha = 7, 5, 0.2
    z = rng.standard_normal((T, E)).astype(np.float32)
    f = rng.random(E)
    f /= f.sum()
    grad = router.aux_loss_grad(z, "fp32", f, alpha)
    assert np.abs(grad.sum(axis=1)).max() < 1e-15
    zu = np.zeros((T, E), dtype=np.float32)
    gu = router.aux_loss_grad(zu, "fp32", f, alpha, grad_scale=3.0)
    np.testing.assert_allclose(gu, np.broadcast_to(3.0 * (alpha / T) * (f - 1.0 / E), (T, E)), rtol=1e-12, atol=1e-17)


# ----------------------------------------------------------------------------- dispatch

def check_capacity_example(dispatch) -> None:
    """[P1] §4.5: 1024 tokens, 8 experts, capacity factor 1.25 -> 160 tokens per expert."""
    g = golden("p1_s4_5_capacity_example.json")
    assert dispatch.capacity(g["tokens"], 1, g["num_experts"], g["capacity_factor"]) == g["capacity"]


def _brute_dispatch(idx: np.ndarray, E: int, C: int):
    flat = [int(e) for e in np.asarray(idx).ravel()]
    n = len(flat)
    rank = [sum(1 for b in range(a) if flat[b] == flat[a]) for a in range(n)]
    counts = [flat.count(e) for e in range(E)]
    offsets = [sum(counts[:e]) for e in range(E + 1)]
    perm = [-1] * n
    for a in range(n):
        perm[offsets[flat[a]] + rank[a]] = a
    slot = [r if r < C else -1 for r in rank]
    kept = [min(c, C) for c in counts]
    return perm, slot, offsets, counts, kept, n - sum(kept)


def check_dispatch_bruteforce(dispatch, router) -> None:
    """The stable dispatch equals an O((T*k)^2) count of earlier same-expert assignments."""
    rng = np.random.default_rng(19)
    for trial in range(30):
        T = int(rng.integers(1, 30))
        E = int(rng.integers(1, 7))
        k = int(rng.integers(1, min(E, 3) + 1))
        z = rng.integers(0, 3, size=(T, E)).astype(np.float64)
        idx = router.top_k(z, k)
        C = int(rng.integers(0, T + 2))
        got = dispatch.dispatch(idx, E, C)
        perm, slot, offsets, counts, kept, nd = _brute_dispatch(idx, E, C)
        assert list(got["perm"]) == perm, trial
        assert list(got["slot"]) == slot, trial
        assert list(got["offsets"]) == offsets and list(got["counts"]) == counts
        assert list(got["kept"]) == kept and got["n_dropped"] == nd


def check_dispatch_identities(dispatch, router, synth) -> None:
    """Counting identities on a workload-shaped batch with drops."""
    w = synth.ROUTER_WORKLOADS["zipf-hot-top8-T131072-E256"].with_tokens(2048)
    z = router.widen(synth.router_logits(w), w.dtype)
    idx = router.top_k(z, w.k)
    C = dispatch.capacity(w.T, w.k, w.E, w.capacity_factor)
    d = dispatch.dispatch(idx, w.E, C)
    n = w.T * w.k
    assert d["offsets"][-1] == n and d["kept"].sum() + d["n_dropped"] == n
    assert d["n_dropped"] > 0                                  # capacity factor 1.0 with hot experts drops
    assert sorted(d["perm"]) == list(range(n))
    flat = idx.ravel()
    for e in range(w.E):
        seg = d["perm"][d["offsets"][e]:d["offsets"][e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)
        assert np.all(d["slot"][seg[:d["kept"][e]]] == np.arange(d["kept"][e]))
        assert np.all(d["slot"][seg[d["kept"][e]:]] == -1)


# ----------------------------------------------------------------------------- Sinkhorn

def check_sinkhorn_two_rank(sinkhorn) -> None:
    """Two ranks, one overloaded: all the mass flows 0 -> 1, whatever the cost."""
    out = sinkhorn.taot_phase1(np.array([[3.0, 1.0]]), ranks_per_node=1, lam=10.0, iters=5)
    np.testing.assert_allclose(out["plan"][0], [[0.0, 1.0], [0.0, 0.0]], atol=1e-15)
    assert out["status"][0] == 0


def check_sinkhorn_dual(sinkhorn) -> None:
    """On a small non-symmetric problem, Sinkhorn-Knopp matches an independent
    solve of the entropic transport dual (scipy L-BFGS):
    max_{f,g} <f,a> + <g,b> - eps * sum_ij exp((f_i + g_j - W_ij)/eps)."""
    from scipy.optimize import minimize
    rng = np.random.default_rng(20)
    R, S, eps = 5, 5, 0.7
    W = rng.random((R, S)) * 2.0                  # not symmetric
    a = rng.random(R) + 0.1
    a /= a.sum()
    b = rng.random(S) + 0.1
    b /= b.sum()
    M = np.exp(-W / eps)

    def negdual(x):
        f, g = x[:R], x[R:]
        Tm = np.exp((f[:, None] + g[None, :] - W) / eps)
        val = f @ a + g @ b - eps * Tm.sum()
        grad = np.concatenate([a - Tm.sum(axis=1), b - Tm.sum(axis=0)])
        return -val, -grad

    res = minimize(negdual, np.zeros(R + S), jac=True, method="L-BFGS-B",
                   options={"gtol": 1e-14, "ftol": 1e-16, "maxiter": 10000})
    f, g = res.x[:R], res.x[R:]
    plan_dual = np.exp((f[:, None] + g[None, :] - W) / eps)
    u, v = sinkhorn.sinkhorn_knopp(a, b, M, 3000)
    plan = sinkhorn.transport_plan(u, M, v)
    np.testing.assert_allclose(plan, plan_dual, rtol=1e-6, atol=1e-9)


def check_sinkhorn_marginals(sinkhorn, loads: np.ndarray) -> None:
    """Column sums equal b after every v update; row sums reach a in 50 iterations;
    the plan has the diag(u) M diag(v) form and no negative entry."""
    out = sinkhorn.taot_phase1(loads, ranks_per_node=8, lam=10.0, iters=50)
    for m in range(loads.shape[0]):
        over = loads[m] - loads[m].mean()            # overload (+) / idle capacity (-)
        ok = (over > 0).any()
        a = np.clip(over, 0, None) / max(np.clip(over, 0, None).sum(), 1e-300)
        b = np.clip(-over, 0, None) / max(np.clip(-over, 0, None).sum(), 1e-300)
        if not ok:
            assert out["status"][m] == 1 and not out["plan"][m].any()
            continue
        plan = out["plan"][m]
        assert (plan >= 0).all()
        np.testing.assert_allclose(plan.sum(axis=0), b, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(plan.sum(axis=1), a, rtol=1e-9, atol=1e-15)
        np.testing.assert_allclose(plan, out["u"][m][:, None] * out["M"] * out["v"][m][None, :], rtol=1e-14)


def check_sinkhorn_topology_kernel(sinkhorn) -> None:
    """With eps = lambda = 10 the intra-node / cross-node kernel ratio is
    exp(-1/10) / exp(-10/10) = e^0.9 > 1 ([P4] §2, soft topology preference)."""
    W = sinkhorn.topology_cost(16, 8, 10.0)
    M = sinkhorn.gibbs_kernel(W, 10.0)
    assert M[0, 0] == 1.0 and abs(M[0, 1] / M[0, 8] - math.exp(0.9)) < 1e-14
    assert (W == W.T).all() and W[3, 3] == 0 and W[3, 5] == 1 and W[3, 12] == 10


# ----------------------------------------------------------------------------- next steps (bias, masked P, full backward)

def check_biased_topk_bruteforce(ext) -> None:
    """top_k_biased equals brute force over k-subsets of z + b (integer values:
    the fp32 sum is exact, ties everywhere); a zero bias gives plain top-k."""
    rng = np.random.default_rng(31)
    for E in range(1, 8):
        for k in range(1, min(E, 3) + 1):
            z = rng.integers(-2, 3, size=(20, E)).astype(np.float32)
            b = rng.integers(-2, 3, size=E).astype(np.float32)
            got = ext.top_k_biased(z, "fp32", b, k)
            s = z.astype(np.float64) + b.astype(np.float64)[None, :]
            for t in range(z.shape[0]):
                assert list(got[t]) == _brute_topk_row(s[t], k), (E, k, t, s[t], got[t])
            zero = ext.top_k_biased(z, "fp32", np.zeros(E, np.float32), k)
            for t in range(z.shape[0]):
                assert list(zero[t]) == _brute_topk_row(z[t].astype(np.float64), k)


def check_biased_topk_dominant(ext) -> None:
    """A bias far above the logits' spread puts its expert first in every row,
    and the rest of each row's picks are that row's plain top-(k-1) of the others."""
    rng = np.random.default_rng(32)
    T, E, k, hot = 50, 9, 3, 6
    z = rng.standard_normal((T, E)).astype(np.float32)
    b = np.zeros(E, np.float32)
    b[hot] = 100.0
    got = ext.top_k_biased(z, "fp32", b, k)
    assert (got[:, 0] == hot).all()
    others = [e for e in range(E) if e != hot]
    for t in range(T):
        rest = sorted(others, key=lambda e: (-float(z[t, e]), e))[:k - 1]
        assert list(got[t, 1:]) == rest


def check_biased_sum_is_fp32(ext) -> None:
    """The selection score is the fp32 sum: 1 + 2^-24 rounds to 1 in fp32, so
    a logit of 1 with bias 2^-24 ties a logit of 1 with bias 0 and the lower
    index wins; in float64 the first would win."""
    z = np.array([[1.0, 1.0]], np.float32)
    b = np.array([0.0, 2.0 ** -24], np.float32)
    assert list(ext.top_k_biased(z, "fp32", b, 1)[0]) == [0]
    b2 = np.array([0.0, 2.0 ** -23], np.float32)       # representable: expert 1 wins
    assert list(ext.top_k_biased(z, "fp32", b2, 1)[0]) == [1]


def check_bias_update_hand(ext) -> None:
    """T*k = 12 assignments over E = 4 experts (mean 3): counts [5, 3, 0, 4]
    move the biases by [-g, 0, +g, -g]; with T*k = 10 (mean 2.5, not an
    integer) no expert sits at the mean."""
    g = 0.125
    b = np.array([0.5, -0.25, 0.0, 1.0], np.float32)
    out = ext.bias_update(b, np.array([5, 3, 0, 4]), T=6, k=2, gamma=g)
    np.testing.assert_array_equal(out, np.array([0.375, -0.25, 0.125, 0.875], np.float32))
    assert out.dtype == np.float32
    out2 = ext.bias_update(np.zeros(4, np.float32), np.array([3, 2, 3, 2]), T=5, k=2, gamma=g)
    np.testing.assert_array_equal(out2, np.array([-g, g, -g, g], np.float32))


def check_bias_update_balances(ext, router) -> None:
    """Bias routing does what [P1] §4.3 says it is for: on a batch with a
    strongly preferred expert set, repeated selection + update lowers the load
    CV (the gate and aux loss are not involved)."""
    rng = np.random.default_rng(33)
    T, E, k = 2000, 16, 2
    z = (rng.standard_normal((T, E)) + np.linspace(2.0, -2.0, E)[None, :]).astype(np.float32)
    b = np.zeros(E, np.float32)
    cv0 = router.load_cv(router.expert_counts(ext.top_k_biased(z, "fp32", b, k), E))
    for _ in range(300):
        counts = router.expert_counts(ext.top_k_biased(z, "fp32", b, k), E)
        b = ext.bias_update(b, counts, T, k, gamma=0.02)
    cv1 = router.load_cv(router.expert_counts(ext.top_k_biased(z, "fp32", b, k), E))
    assert cv0 > 0.5 and cv1 < 0.1 * cv0, (cv0, cv1)
    assert b[0] < 0 < b[-1]          # the favoured expert is pushed down, the shunned one up


def check_masked_p_closed_forms(ext, router) -> None:
    """k = E picks every expert, so masked P = unmasked P / k; a per-token loop
    gives the masked mean for k < E."""
    rng = np.random.default_rng(34)
    T, E = 30, 5
    z = rng.standard_normal((T, E))
    p = router.softmax(z)
    idx_all = router.top_k(z, E)
    np.testing.assert_allclose(ext.mean_router_prob_masked(p, idx_all, E), router.mean_router_prob(p) / E,
                               rtol=1e-14, atol=0)
    k = 2
    idx = router.top_k(z, k)
    want = np.zeros(E)
    for t in range(T):
        for j in range(k):
            want[idx[t, j]] += p[t, idx[t, j]]
    want /= T * k
    np.testing.assert_allclose(ext.mean_router_prob_masked(p, idx, k), want, rtol=1e-14, atol=0)


def _full_grad_case(ext, router, renorm: bool, masked: bool, k: int, with_dgate: bool, seed: int):
    rng = np.random.default_rng(seed)
    T, E, alpha, g = 4, 6, 0.3, 1.7
    z32 = rng.standard_normal((T, E)).astype(np.float32)
    z = z32.astype(np.float64)
    idx = router.top_k(z, k)
    f = rng.random(E)
    f /= f.sum()
    dgate = rng.standard_normal((T, k)) if with_dgate else None
    grad = ext.router_backward_full(z32, "fp32", f, alpha, g, idx, dgate, renorm, masked)
    h = 1e-6
    fd = np.zeros_like(z)
    for t in range(T):
        for j in range(E):
            zp, zm = z.copy(), z.copy()
            zp[t, j] += h
            zm[t, j] -= h
            fd[t, j] = (ext.full_loss_of_logits(zp, f, alpha, g, idx, dgate, renorm, masked)
                        - ext.full_loss_of_logits(zm, f, alpha, g, idx, dgate, renorm, masked)) / (2 * h)
    return grad, fd, idx


def check_full_grad_finite_difference(ext, router) -> None:
    """Central differences of the main-loss gate term plus g * L_aux (picks and
    f frozen) match router_backward_full, for every combination of
    renormalised gates, masked P, k and the presence of dgate."""
    seed = 40
    for renorm in (False, True):
        for masked in (False, True):
            for k in (1, 2, 3):
                for with_dgate in (False, True):
                    seed += 1
                    grad, fd, _ = _full_grad_case(ext, router, renorm, masked, k, with_dgate, seed)
                    scale = max(np.abs(grad).max(), 1e-12)
                    err = np.abs(grad - fd).max() / scale
                    assert err <= 1e-7, (renorm, masked, k, with_dgate, err)


def check_full_grad_structure(ext, router) -> None:
    """Rows sum to zero; no dgate and unmasked P reduce to router.aux_loss_grad;
    with renormalised gates and no aux loss, the unpicked experts get no gradient
    (the renormalised gates depend only on the picked logits)."""
    rng = np.random.default_rng(50)
    T, E, k, alpha = 6, 7, 3, 0.2
    z = rng.standard_normal((T, E)).astype(np.float32)
    idx = router.top_k(z.astype(np.float64), k)
    f = rng.random(E)
    f /= f.sum()
    dgate = rng.standard_normal((T, k))
    g = ext.router_backward_full(z, "fp32", f, alpha, 1.3, idx, dgate, True, False)
    assert np.abs(g.sum(axis=1)).max() < 1e-14
    np.testing.assert_allclose(ext.router_backward_full(z, "fp32", f, alpha, 1.3, idx, None, True, False),
                               router.aux_loss_grad(z, "fp32", f, alpha, grad_scale=1.3), rtol=1e-12, atol=1e-18)
    gate_only = ext.router_backward_full(z, "fp32", f, 0.0, 1.0, idx, dgate, True, False)
    mask = ext.pick_mask(idx, E)
    # zero up to the rounding of sum_i p_i dp_i, which cancels exactly in real arithmetic
    assert np.abs(gate_only * (1.0 - mask)).max() <= 1e-14 * np.abs(gate_only).max()
    assert np.abs(gate_only * mask).max() > 1e-3


# ----------------------------------------------------------------------------- EPLB (replication, packing)

def check_packing_worked_example(eplb) -> None:
    """The page's example: [9, 7, 5, 3] onto 2 nodes of 2 groups -> {9, 3} / {7, 5}, 12 / 12,
    placed in the order 9, 7, 5, 3 (so 5 lands second on node 1 and 3 second on node 0)."""
    g = golden("p3_s4_1_2_balanced_packing_example.json")
    bins, pos, totals = eplb.balanced_packing(g["weights"], g["num_bins"])
    assert list(bins) == g["bin_of_item"], bins
    assert list(pos) == [0, 0, 1, 1], pos
    assert list(totals) == g["bin_totals"], totals


def check_packing_equal_weights_round_robin(eplb) -> None:
    """Equal weights: the lightest non-full bin is always the next one in turn,
    so item i goes to bin i mod G at position i // G."""
    for N, G in ((12, 4), (8, 8), (6, 1), (64, 16)):
        bins, pos, totals = eplb.balanced_packing([2.5] * N, G)
        assert list(bins) == [i % G for i in range(N)]
        assert list(pos) == [i // G for i in range(N)]
        assert np.all(totals == 2.5 * (N // G))


def check_packing_cardinality_and_mass(eplb) -> None:
    """Every bin takes exactly N / G items, and the bins' totals hold all the weight;
    a dominant item fills its bin with the lightest items only once the others are full."""
    bins, pos, totals = eplb.balanced_packing([10.0, 1.0, 1.0, 1.0], 2)
    assert list(bins) == [0, 1, 1, 0] and list(totals) == [11.0, 2.0]
    rng = np.random.default_rng(60)
    for N, G in ((48, 8), (30, 5), (7, 7), (24, 4)):
        w = rng.random(N) * 10
        if N == 24:
            w[:3] *= 50                          # a few dominant items: the capacity binds
        bins, pos, totals = eplb.balanced_packing(w, G)
        assert np.all(np.bincount(bins, minlength=G) == N // G)
        for b in range(G):
            assert sorted(pos[bins == b]) == list(range(N // G))
        assert abs(totals.sum(dtype=np.float64) - w.sum()) < 1e-4 * w.sum()


def check_replication_bruteforce(eplb) -> None:
    """The greedy replication reaches the smallest possible per-replica peak
    max_e w_e / c_e over all count vectors with sum c = num_phys and c >= 1
    (brute force on tiny cases)."""
    rng = np.random.default_rng(61)

    def compositions(total, parts):
        if parts == 1:
            yield (total,)
            return
        for first in range(1, total - parts + 2):
            for rest in compositions(total - first, parts - 1):
                yield (first,) + rest

    for _ in range(40):
        E = int(rng.integers(1, 5))
        w = rng.integers(0, 30, size=E)
        num_phys = E + int(rng.integers(0, 6))
        _, count = eplb.replicate_experts(w, num_phys)
        assert count.sum() == num_phys and count.min() >= 1
        best = min(max(w[e] / c[e] for e in range(E)) for c in compositions(num_phys, E))
        got = max(w[e] / count[e] for e in range(E))
        assert abs(got - best) < 1e-12, (w, num_phys, count, got, best)


def check_replication_hand_case(eplb) -> None:
    """w = [6, 2, 1], three extra replicas: 6/1 -> expert 0 (c = 2); 3 > 2 -> expert 0
    (c = 3); 6/3 = 2/1 ties -> the lower index, expert 0 (c = 4).  num_phys = E: identity."""
    p2l, c = eplb.replicate_experts([6, 2, 1], 6)
    assert list(c) == [4, 1, 1] and list(p2l) == [0, 1, 2, 0, 0, 0]
    p2l, c = eplb.replicate_experts([5, 9, 1, 3], 4)
    assert list(c) == [1, 1, 1, 1] and list(p2l) == [0, 1, 2, 3]


def check_plan_invariants(eplb) -> None:
    """Both policies: every GPU holds S slots; each expert's copies equal its count;
    the GPU loads add up to the total load; the hierarchical policy keeps every
    copy of an expert on the node its group was packed to."""
    rng = np.random.default_rng(62)
    E, num_phys, num_gpus, num_nodes, num_groups = 48, 64, 16, 4, 8
    w = rng.integers(0, 500, size=E)
    for groups in (0, num_groups):
        out = eplb.plan(w, num_phys, num_gpus, num_nodes, groups)
        assert out["hierarchical"] == (groups > 0)
        p2l, cnt = out["phy2log"], out["log_count"]
        assert np.array_equal(np.bincount(p2l, minlength=E), cnt) and cnt.sum() == num_phys
        assert abs(out["gpu_load"].sum(dtype=np.float64) - w.sum()) < 1e-5 * w.sum()
        S = num_phys // num_gpus
        loads = [sum(w[e] / cnt[e] for e in p2l[g * S:(g + 1) * S]) for g in range(num_gpus)]
        np.testing.assert_allclose(loads, out["gpu_load"], rtol=1e-5)
        if groups:
            gsize, slots_per_node = E // groups, num_phys // num_nodes
            for n in range(num_nodes):
                on_node = set(p2l[n * slots_per_node:(n + 1) * slots_per_node] // gsize)
                assert len(on_node) == groups // num_nodes
    out = eplb.plan(w, num_phys, num_gpus, 3, 8)            # 3 nodes do not divide 8 groups: global
    assert not out["hierarchical"]


# ----------------------------------------------------------------------------- TAOT Phase 2 (column-first matching)

def check_match_hand_single(match) -> None:
    """Two ranks on one node, experts [5, 3 | 1, 1]: rank loads 8 / 2, mean 5.  The cold
    rank can take min(w, floor(8 - 5), floor(5 - 2)) = 3 tokens of expert 0 or 1: the tie
    goes to expert 0; then both ranks sit at the mean and nothing else moves."""
    out = match.match([5, 3, 1, 1], np.zeros((2, 2), np.float32), R=2, ranks_per_node=2, K=2)
    assert out["slot_expert"].tolist() == [[-1, -1], [0, -1]]
    assert out["slot_tokens"].tolist() == [[0, 0], [3, 0]]
    assert out["rank_load"].tolist() == [5, 5] and out["moved"] == 3


def check_match_hand_arbitration(match) -> None:
    """Four ranks, two per node, one expert each.
    (a) Loads [10, 2, 2, 2], mean 4: every cold rank wants expert 0 (2 tokens each); rank 1
        shares rank 0's node and wins round 1, then the larger flow (rank 3), then rank 2:
        all end at the mean, whatever K >= 1.
    (b) Loads [2, 6, 8, 8], mean 6, K = 1: cold rank 0 can take 2 tokens of expert 2 or of
        expert 3, both across nodes: the flow decides (plan[3, 0] > plan[2, 0]: expert 3).
    (c) Loads [8, 4, 4, 8], mean 6, K = 1: cold rank 1 takes rank 0's expert (same node)
        and cold rank 2 rank 3's, although the flow prefers the cross-node pairs."""
    plan = np.zeros((4, 4), np.float32)
    plan[0, 2], plan[0, 3] = 0.25, 0.5
    for K in (1, 3):
        out = match.match([10, 2, 2, 2], plan, R=4, ranks_per_node=2, K=K)
        assert out["slot_expert"][:, 0].tolist() == [-1, 0, 0, 0]
        assert out["slot_tokens"][:, 0].tolist() == [0, 2, 2, 2]
        assert out["rank_load"].tolist() == [4, 4, 4, 4]
    pb = np.zeros((4, 4), np.float32)
    pb[2, 0], pb[3, 0] = 0.25, 0.5
    out = match.match([2, 6, 8, 8], pb, R=4, ranks_per_node=2, K=1)
    assert out["slot_expert"][:, 0].tolist() == [3, -1, -1, -1] and out["rank_load"].tolist() == [4, 6, 8, 6]
    pb[2, 0], pb[3, 0] = 0.5, 0.25
    out = match.match([2, 6, 8, 8], pb, R=4, ranks_per_node=2, K=1)
    assert out["slot_expert"][:, 0].tolist() == [2, -1, -1, -1] and out["rank_load"].tolist() == [4, 6, 6, 8]
    pc = np.zeros((4, 4), np.float32)
    pc[0, 1], pc[3, 1], pc[0, 2], pc[3, 2] = 0.1, 0.9, 0.9, 0.1
    out = match.match([8, 4, 4, 8], pc, R=4, ranks_per_node=2, K=1)
    assert out["slot_expert"][:, 0].tolist() == [-1, 0, 3, -1] and out["rank_load"].tolist() == [6, 6, 6, 6]


def check_match_invariants(match) -> None:
    """On skewed random loads: the total is kept, no hot rank drops below the mean and
    no cold rank rises above it, a rank holds at most K replicas and an expert once,
    every slot moves tokens, and an expert never gives away more than its load."""
    rng = np.random.default_rng(70)
    for trial in range(30):
        R, rpn, per, K = (8, 4, 3, 2) if trial % 2 else (16, 8, 2, 3)
        E = R * per
        w = rng.multinomial(40 * E, (np.arange(E) + 1.0) ** -1.2 / ((np.arange(E) + 1.0) ** -1.2).sum())
        w = w[rng.permutation(E)]
        plan = rng.random((R, R)).astype(np.float32)
        out = match.match(w, plan, R, rpn, K)
        before = w.reshape(R, per).sum(axis=1)
        after = out["rank_load"]
        total = before.sum()
        assert after.sum() == total
        hot, cold = before * R > total, before * R < total
        assert np.all(after[hot] * R >= total) and np.all(after[cold] * R <= total)
        assert np.all(after[hot] <= before[hot]) and np.all(after[cold] >= before[cold])
        se, st = out["slot_expert"], out["slot_tokens"]
        assert np.all((se >= 0) == (st > 0))
        for c in range(R):
            got = [e for e in se[c] if e >= 0]
            assert len(got) == len(set(got)) <= K
        given = np.zeros(E, np.int64)
        for c in range(R):
            for e, x in zip(se[c], st[c]):
                if e >= 0:
                    given[e] += x
        assert np.all(given <= w)
        assert out["moved"] == int(st.sum())
    none = match.match(w, plan, R, rpn, 0)
    assert none["moved"] == 0 and np.array_equal(none["rank_load"], before)


def check_plan_hand_cases(eplb) -> None:
    """Worked by hand from the page's rules.
    Hierarchical: the page's groups [9, 7, 5, 3] (one expert each) on 2 nodes of one GPU
    with 3 slots: node 0 takes groups {9, 3}, replicates expert 0 (9 > 3) and packs
    4.5, 4.5, 3 -> slots [0, 0, 3]; node 1 takes {7, 5}, replicates expert 1 and packs
    5, 3.5, 3.5 -> slots [2, 1, 1]; both GPUs carry 12.
    Global: loads [6, 2, 1, 3] onto 6 slots of 2 GPUs: expert 0 gets two more copies
    (6 > 3, then 6/2 ties 3/1 and the lower index wins); copies weigh 3, 2, 2, 2, 2, 1
    (items 3, 0, 1, 4, 5, 2) and land 3 -> GPU 0, 2 -> GPU 1, 2 -> GPU 1, 2 -> GPU 0,
    2 -> GPU 1 (the lighter), 1 -> GPU 0 (the only open one): 6 / 6."""
    h = eplb.plan([9, 7, 5, 3], 6, 2, 2, 4)
    assert h["hierarchical"] and h["phy2log"].tolist() == [0, 0, 3, 2, 1, 1]
    assert h["log_count"].tolist() == [2, 2, 1, 1] and h["gpu_load"].tolist() == [12.0, 12.0]
    g = eplb.plan([6, 2, 1, 3], 6, 2, 1, 0)
    assert not g["hierarchical"] and g["phy2log"].tolist() == [3, 0, 2, 0, 1, 0]
    assert g["log_count"].tolist() == [3, 1, 1, 1] and g["gpu_load"].tolist() == [6.0, 6.0]


def check_masked_p_hand(ext, router) -> None:
    """Two tokens, three experts, top-1, by hand: z = [0, ln 2, 0] gives p = [1/4, 1/2, 1/4]
    and picks expert 1; z = [ln 3, 0, 0] gives p = [3/5, 1/5, 1/5] and picks expert 0.
    Masked P = [3/5, 1/2, 0] / 2 = [0.3, 0.25, 0], balance 3 * (0.5*0.3 + 0.5*0.25) = 0.825;
    unmasked P = [0.425, 0.35, 0.225], balance 1.1625."""
    z = np.array([[0.0, math.log(2.0), 0.0], [math.log(3.0), 0.0, 0.0]])
    m = ext.router_forward_ex(z.astype(np.float32), "fp32", 1, 1.0, masked_p=True)
    u = ext.router_forward_ex(z.astype(np.float32), "fp32", 1, 1.0, masked_p=False)
    assert m["idx"][:, 0].tolist() == [1, 0]
    np.testing.assert_allclose(m["P"], [0.3, 0.25, 0.0], rtol=1e-7, atol=1e-9)
    np.testing.assert_allclose(u["P"], [0.425, 0.35, 0.225], rtol=1e-7)
    assert abs(m["balance"] - 0.825) < 1e-7 and abs(u["balance"] - 1.1625) < 1e-7


def _row_first_match(w, plan, R, rpn, K):
    """An expert-major greedy for comparison (the "row-first" order the TAOT page
    argues against): hot experts heaviest first, each placing replicas on the
    best-scoring cold ranks until its home rank or the cold ranks are spent."""
    w = [int(x) for x in w]
    E = len(w)
    per = E // R
    load = [sum(w[r * per:(r + 1) * per]) for r in range(R)]
    total = sum(load)
    w_rem, used, n_slots = list(w), set(), [0] * R
    P = np.asarray(plan, np.float32)
    for e in sorted(range(E), key=lambda e: (-w[e], e)):
        h = e // per
        while load[h] * R > total and w_rem[e] > 0:
            best = None
            for c in range(R):
                if n_slots[c] >= K or load[c] * R >= total or (c, e) in used:
                    continue
                x = min(w_rem[e], (load[h] * R - total) // R, (total - load[c] * R) // R)
                if x > 0:
                    s = (x, 1 if h // rpn == c // rpn else 0, float(P[h, c]), -c)
                    if best is None or s > best[0]:
                        best = (s, c, x)
            if best is None:
                break
            _, c, x = best
            load[h] -= x
            load[c] += x
            w_rem[e] -= x
            used.add((c, e))
            n_slots[c] += 1
    return np.asarray(load)


def check_match_column_first_claim(match, sinkhorn) -> None:
    """[P4] §2: the column-first matching leaves less residual imbalance than a
    row-first (expert-major) order, 1-2 % against 7-10 % on the page's loads.  On
    seeded Zipf loads (s 0.6-1.0, 16-64 ranks, K 2-4) the column-first plan's mean
    residual is below the expert-major greedy's and below 5 %."""
    rng = np.random.default_rng(80)
    col, row = [], []
    for s_exp, R, per, K in ((0.6, 16, 4, 2), (0.8, 32, 6, 2), (0.5, 64, 6, 4), (1.0, 16, 4, 3)):
        for _ in range(8):
            E = R * per
            p = (np.arange(E) + 1.0) ** -s_exp
            w = rng.multinomial(200 * E, p[rng.permutation(E)] / p.sum())
            rl = w.reshape(R, per).sum(axis=1).astype(np.float64)
            plan = np.asarray(sinkhorn.taot_phase1(rl[None, :], 8, 10.0, None, 50)["plan"][0], np.float32)
            col.append(match.residual_imbalance(match.match(w, plan, R, 8, K)["rank_load"]))
            row.append(match.residual_imbalance(_row_first_match(w, plan, R, 8, K)))
    assert np.mean(col) < np.mean(row), (np.mean(col), np.mean(row))
    assert np.mean(col) < 0.05, np.mean(col)


# ----------------------------------------------------------------------------- conversions, helpers, measures

def check_widen_library(router) -> None:
    """bf16 bit patterns widen to the values torch's own bfloat16 -> float32
    conversion gives, for every finite pattern (subnormals and -0.0 included),
    and fp32 logits pass through unchanged.  By hand: 0x3F80 is 1.0, 0xC040 is
    -3.0, 0x0001 is 2^-133, 0x7F7F is (2 - 2^-7) * 2^127."""
    import torch

    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):                     # the NaN patterns, left out below
        want = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy().astype(np.float64)
        got = router.widen(bits.reshape(256, 256), "bf16").ravel()
    fin = np.isfinite(want)
    assert fin.sum() == (1 << 16) - 2 * 128                   # 2 infinities and 254 NaNs left out
    np.testing.assert_array_equal(got[fin], want[fin])
    assert np.array_equal(np.signbit(got[fin]), np.signbit(want[fin]))
    hand = router.widen(np.array([[0x3F80, 0xC040, 0x0001, 0x7F7F]], dtype=np.uint16), "bf16")[0]
    assert list(hand) == [1.0, -3.0, 2.0 ** -133, (2.0 - 2.0 ** -7) * 2.0 ** 127]
    x = np.random.default_rng(19).standard_normal((3, 5)).astype(np.float32)
    np.testing.assert_array_equal(router.widen(x, "fp32"), x.astype(np.float64))


def check_balance_degree_hand(router) -> None:
    """[P3] §5.1's balance degree 1 - (max - mean) / mean: 1 when the peak is the
    mean, 0 when it is twice the mean, 0.25 at 1.75; [P1] §5.4's ratio flag is
    strictly above 2."""
    assert router.balance_degree(1.0) == 1.0
    assert router.balance_degree(2.0) == 0.0
    assert router.balance_degree(1.75) == 0.25
    assert router.balance_degree(4.21875) == -2.21875         # the [P1] §5.3 log line's max/mean
    assert not router.is_ratio_imbalanced(2.0) and router.is_ratio_imbalanced(2.0 + 2.0 ** -40)


def check_softmax_backward_autograd(ext) -> None:
    """The softmax Jacobian-vector product equals torch's autograd through
    torch.softmax in float64, on random rows and on a saturated row."""
    import torch

    rng = np.random.default_rng(21)
    z = rng.standard_normal((6, 7)) * 3.0
    z[0, 2] = 60.0                                            # one dominant logit
    dp = rng.standard_normal((6, 7))
    zt = torch.tensor(z, dtype=torch.float64, requires_grad=True)
    torch.softmax(zt, dim=1).backward(torch.tensor(dp, dtype=torch.float64))
    p = np.exp(z - z.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(ext.softmax_backward(p, dp), zt.grad.numpy(), rtol=1e-12, atol=1e-15)


def check_grad_wrt_probs_finite_difference(ext, router) -> None:
    """dL/dp of L(p) = sum dgate * gate(p) + g * alpha * E * sum_i f_i P_i(p), picks
    fixed, against central differences of that loss evaluated through
    router.gates and the (masked or unmasked) P, p treated as free variables."""
    rng = np.random.default_rng(22)
    T, E, k, alpha, g = 4, 5, 3, 0.3, 1.3
    p = rng.random((T, E)) + 0.1
    idx = np.array([rng.permutation(E)[:k] for _ in range(T)])
    f = rng.random(E)
    f /= f.sum()
    dgate = rng.standard_normal((T, k))

    def loss(q, renorm, masked):
        P = ext.mean_router_prob_masked(q, idx, k) if masked else router.mean_router_prob(q)
        return float((dgate * router.gates(q, idx, renorm)).sum()) + g * alpha * E * float((f * P).sum())

    h = 1e-6
    for renorm in (False, True):
        for masked in (False, True):
            got = ext.grad_wrt_probs(p, idx, f, alpha, g, T, k, dgate, renorm, masked)
            fd = np.zeros_like(p)
            for t in range(T):
                for i in range(E):
                    qp, qm = p.copy(), p.copy()
                    qp[t, i] += h
                    qm[t, i] -= h
                    fd[t, i] = (loss(qp, renorm, masked) - loss(qm, renorm, masked)) / (2 * h)
            np.testing.assert_allclose(got, fd, rtol=1e-7, atol=1e-8)


def check_supply_demand_hand(sinkhorn) -> None:
    """loads [3, 1, 1, 3]: mean 2, supply [1, 0, 0, 1] / 2, demand [0, 1, 1, 0] / 2;
    [5, 1, 0, 2]: mean 2, supply [3, 0, 0, 0] / 3, demand [0, 1, 2, 0] / 3; equal
    loads have no mass."""
    a, b, ok = sinkhorn.supply_demand(np.array([3.0, 1.0, 1.0, 3.0]))
    assert ok and list(a) == [0.5, 0.0, 0.0, 0.5] and list(b) == [0.0, 0.5, 0.5, 0.0]
    a, b, ok = sinkhorn.supply_demand(np.array([5.0, 1.0, 0.0, 2.0]))
    assert ok and list(a) == [1.0, 0.0, 0.0, 0.0]
    np.testing.assert_allclose(b, [0.0, 1.0 / 3.0, 2.0 / 3.0, 0.0], rtol=1e-15)
    _, _, ok = sinkhorn.supply_demand(np.full(5, 7.0))
    assert not ok


def check_topology_cost_hand(sinkhorn) -> None:
    """Four ranks, two per node, lambda = 10: W written out by hand; its Gibbs
    kernel at eps = 2 is exp(-W / 2) element by element."""
    W = sinkhorn.topology_cost(4, 2, 10.0)
    want = np.array([[0, 1, 10, 10], [1, 0, 10, 10], [10, 10, 0, 1], [10, 10, 1, 0]], dtype=np.float64)
    np.testing.assert_array_equal(W, want)
    M = sinkhorn.gibbs_kernel(W, 2.0)
    assert M[0, 0] == 1.0 and M[0, 1] == math.exp(-0.5) and M[1, 3] == math.exp(-5.0)


def check_residual_imbalance_hand(match) -> None:
    """(max - mean) / mean: [6, 4, 5, 5] -> 0.2, equal loads -> 0, [9, 1] -> 0.8."""
    assert abs(match.residual_imbalance([6, 4, 5, 5]) - 0.2) < 1e-15
    assert match.residual_imbalance([3, 3, 3]) == 0.0
    assert abs(match.residual_imbalance([9, 1]) - 0.8) < 1e-15


def check_forward_ex_reductions(ext, router) -> None:
    """router_forward_ex reduces to the plain forward: with a zero bias and
    unmasked P every output equals router.router_forward's.  With a bias only
    the choice of experts moves ([P1] §4.3): P stays the plain mean of the
    unbiased softmax, and each gate is the unbiased p of its pick (k = 1), or
    those p renormalised over the picks (k > 1)."""
    rng = np.random.default_rng(35)
    T, E = 40, 7
    z = rng.standard_normal((T, E)).astype(np.float32)
    for k in (1, 3):
        plain = router.router_forward(z, "fp32", k, 0.1, n_ranks=7)
        ex = ext.router_forward_ex(z, "fp32", k, 0.1, n_ranks=7, bias=np.zeros(E, np.float32))
        for key in ("idx", "gate", "counts", "f", "P", "rank_load"):
            np.testing.assert_array_equal(ex[key], plain[key], err_msg=key)
        for key in ("l_aux", "balance", "cv", "max_over_mean", "rank_cv"):
            assert ex[key] == plain[key], key
        b = np.zeros(E, np.float32)
        b[2], b[5] = 3.0, -3.0
        biased = ext.router_forward_ex(z, "fp32", k, 0.1, bias=b)
        np.testing.assert_array_equal(biased["P"], plain["P"])
        assert (biased["idx"] != plain["idx"]).any()
        p = np.exp(z.astype(np.float64) - z.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        for t in range(T):
            picked = p[t, biased["idx"][t]]
            want = picked if k == 1 else picked / picked.sum()
            np.testing.assert_allclose(biased["gate"][t], want, rtol=1e-14)
