"""GPU parity of the router path through the C ABI against the CPU oracle.

Small sizes span many CTAs and a ragged tail; full sizes are the four router
workloads as benchmarked, compared on every element.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import (FLT_MIN, RTOL, assert_close, assert_equal, check_backward, check_dispatch, check_forward,
                    oracle_forward, to_device, workload_inputs)

pytestmark = pytest.mark.gpu

WORKLOADS = list(synth.ROUTER_WORKLOADS)
SMALL_T = {"switch-top1-T4096-E8": 1001, "zipf-top2-T65536-E64": 3001,
           "zipf-hot-top8-T131072-E256": 2999, "zipf-ep64-top6-T262144-E384": 3007}


@pytest.fixture(scope="module")
def mr(native_lib):
    import moe_expert_routing_router_gb300 as m
    return m


def _run_fwd(mr, w, logits):
    x = to_device(logits, w.dtype)
    got = mr.moe_router_fwd(x, w.k, w.alpha, renorm=int(w.renorm), n_ranks=w.n_ranks)
    torch.cuda.synchronize()
    return x, got


@pytest.mark.parametrize("name", WORKLOADS)
@pytest.mark.parametrize("size", ["small", "full"])
def test_forward_parity(mr, name, size):
    w, logits = workload_inputs(name, SMALL_T[name] if size == "small" else None)
    _, got = _run_fwd(mr, w, logits)
    want = oracle_forward(logits, w.dtype, w.k, w.alpha, w.renorm, w.n_ranks)
    check_forward(got, want, w.n_ranks)


@pytest.mark.parametrize("name", WORKLOADS)
@pytest.mark.parametrize("size", ["small", "full"])
def test_backward_parity(mr, name, size):
    w, logits = workload_inputs(name, SMALL_T[name] if size == "small" else None)
    x = to_device(logits, w.dtype)
    rng = np.random.default_rng(5)
    f = rng.random(w.E).astype(np.float32)
    f /= f.sum()
    dl = mr.moe_router_bwd(x, torch.from_numpy(f).cuda(), w.alpha, grad_scale=1.5)
    torch.cuda.synchronize()
    check_backward(dl, logits, w.dtype, f.astype(np.float64), w.alpha, 1.5)


@pytest.mark.parametrize("name", WORKLOADS)
@pytest.mark.parametrize("size", ["small", "full"])
def test_dispatch_parity(mr, name, size):
    w, logits = workload_inputs(name, SMALL_T[name] if size == "small" else None)
    z = logits
    idx = np.concatenate([oracle.router.top_k(oracle.router.widen(z[r:r + 16384], w.dtype), w.k)
                          for r in range(0, w.T, 16384)])
    C = oracle.dispatch.capacity(w.T, w.k, w.E, w.capacity_factor)
    got = mr.moe_dispatch(torch.from_numpy(idx.astype(np.int32)).cuda(), w.E, w.capacity_factor)
    torch.cuda.synchronize()
    assert got["capacity"] == C
    check_dispatch(got, idx, w.E, C)


@pytest.mark.parametrize("name", WORKLOADS)
@pytest.mark.parametrize("size", ["small", "full"])
def test_step_parity_and_equals_separate_calls(mr, name, size):
    w, logits = workload_inputs(name, SMALL_T[name] if size == "small" else None)
    x = to_device(logits, w.dtype)
    st = mr.moe_router_step(x, w.k, w.alpha, w.capacity_factor, renorm=int(w.renorm), n_ranks=w.n_ranks,
                            grad_scale=1.0)
    torch.cuda.synchronize()
    want = oracle_forward(logits, w.dtype, w.k, w.alpha, w.renorm, w.n_ranks)
    check_forward(st, want, w.n_ranks)
    C = oracle.dispatch.capacity(w.T, w.k, w.E, w.capacity_factor)
    check_dispatch(st, want["idx"], w.E, C)
    check_backward(st["dlogits"], logits, w.dtype, want["f"], w.alpha, 1.0)
    # the three separate calls give the same bits, except P and the two scalars
    # built from it, which a split step forms in its backward (exact fixed-point
    # totals of other partial sums): those agree to rounding
    fw = mr.moe_router_fwd(x, w.k, w.alpha, renorm=int(w.renorm), n_ranks=w.n_ranks)
    dp = mr.moe_dispatch(fw["idx"], w.E, w.capacity_factor)
    dl = mr.moe_router_bwd(x, fw["f"], w.alpha, 1.0)
    torch.cuda.synchronize()
    check_step_equals_separate(st, fw, dp, dl)


def check_step_equals_separate(st, fw, dp, dl):
    for key in ("idx", "gate", "counts", "f", "rank_load"):
        assert torch.equal(st[key], fw[key]), key
    assert torch.equal(st["scalars"][2:], fw["scalars"][2:])
    assert_close("P", st["P"].cpu().numpy(), fw["P"].double().cpu().numpy(), 2 * RTOL, FLT_MIN)
    assert_close("L_aux, balance", st["scalars"][:2].cpu().numpy(), fw["scalars"][:2].double().cpu().numpy(), 2 * RTOL)
    for key in ("perm", "slot", "offsets", "kept", "n_dropped"):
        assert torch.equal(st[key], dp[key]), key
    assert torch.equal(st["dlogits"], dl)


def test_repeated_calls_are_bit_identical(mr):
    w, logits = workload_inputs("zipf-ep64-top6-T262144-E384", 20011)
    x = to_device(logits, w.dtype)
    a = mr.moe_router_step(x, w.k, w.alpha, w.capacity_factor, n_ranks=w.n_ranks)
    b = mr.moe_router_step(x, w.k, w.alpha, w.capacity_factor, n_ranks=w.n_ranks)
    torch.cuda.synchronize()
    for key in a:
        if isinstance(a[key], torch.Tensor):
            assert torch.equal(a[key], b[key]), key


# ----------------------------------------------------------------------------- edge cases

EDGE = [
    # (T, E, k, dtype, renorm, n_ranks, cf, levels)   levels > 0: integer logits (ties)
    (1, 1, 1, "fp32", -1, 0, 1.0, 0),
    (1, 1, 1, "bf16", -1, 1, 1.0, 0),
    (5, 8, 8, "bf16", -1, 2, 1.0, 0),          # k = E
    (777, 64, 4, "bf16", -1, 8, 1.0, 3),       # heavy ties, vector path
    (513, 7, 3, "fp32", -1, 7, 0.5, 2),        # odd E, scalar path, ties, drops
    (1000, 33, 2, "bf16", 0, 0, 2.0, 0),       # odd E, raw gates for k = 2
    (300, 100, 1, "bf16", 1, 10, 1.0, 0),      # renormalised top-1 gate (= 1)
    (4099, 1024, 8, "bf16", -1, 64, 1.25, 0),  # largest E and k
    (2050, 1000, 5, "fp32", -1, 8, 1.0, 4),    # E not a multiple of the vector width
    (100003, 64, 2, "bf16", -1, 0, 1.25, 0),   # long ragged batch
    (4096, 8, 1, "fp32", -1, 0, 1.25, 0),      # Switch top-1, E = 8
    (3000, 384, 6, "fp32", -1, 64, 1.0, 0),    # fp32 vector path at E = 384
    (2000, 16, 2, "bf16", -1, 4, 0.25, 0),     # capacity below the mean: most tokens dropped
    (2048, 64, 8, "bf16", -1, 8, 1.0, 0),      # k = 8 at E = 64
    (1500, 48, 6, "bf16", 0, 0, 1.25, 2),      # raw gates, ties
    (999, 40, 5, "bf16", 1, 5, 1.0, 0),        # odd k, renormalised
    (30011, 384, 6, "bf16", -1, 64, 1.25, 3),  # 32 lanes per row: candidate path with heavy ties
    (30011, 200, 4, "bf16", -1, 8, 1.0, 0),    # candidate path, columns past E in the last lanes
    (20011, 512, 8, "bf16", -1, 64, 1.0, 0),   # candidate path at E = 512
    (20011, 256, 1, "bf16", 1, 0, 1.0, 0),     # candidate path, top-1 renormalised
    (20011, 384, 6, "bf16", 0, 0, 1.25, 0),    # raw gates: the step keeps the softmax in its forward
]


@pytest.mark.parametrize("T,E,k,dtype,renorm,n_ranks,cf,levels", EDGE)
def test_edge_cases(mr, T, E, k, dtype, renorm, n_ranks, cf, levels):
    logits = synth.random_logits(T, E, dtype, seed=T * 7 + E, scale=2.0, integer_levels=levels)
    x = to_device(logits, dtype)
    st = mr.moe_router_step(x, k, 0.01, cf, renorm=renorm, n_ranks=n_ranks, grad_scale=0.5)
    torch.cuda.synchronize()
    rn = None if renorm < 0 else bool(renorm)
    want = oracle_forward(logits, dtype, k, 0.01, rn, n_ranks)
    check_forward(st, want, n_ranks)
    check_dispatch(st, want["idx"], E, oracle.dispatch.capacity(T, k, E, cf))
    check_backward(st["dlogits"], logits, dtype, want["f"], 0.01, 0.5)


SATURATED = [
    # (T, E, k, dtype): staged bf16 at E = 64 and E = 384, fp32 at E = 64
    (3001, 64, 2, "bf16"), (3007, 384, 6, "bf16"), (2001, 64, 2, "fp32"),
]


def _saturated_logits(T, E, dtype, seed):
    """N(0, 1) logits where every third row has one logit raised to +100 (a
    spread above 87, so that the other probabilities of the row fall below the
    smallest normal fp32 number), every seventh row two such logits (a tie at
    the top), and every eleventh row one at +88 (p near 2^-126)."""
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((T, E)).astype(np.float32)
    cols = rng.integers(0, E, size=T)
    z[0::3][np.arange(len(z[0::3])), cols[0::3]] = 100.0
    r7 = np.arange(0, T, 7)
    z[r7, cols[r7]] = 100.0
    z[r7, (cols[r7] + 5) % E] = 100.0
    r11 = np.arange(5, T, 11)
    z[r11, cols[r11]] = 88.0
    return synth.f32_to_bf16_bits(z) if dtype == "bf16" else z


@pytest.mark.parametrize("T,E,k,dtype", SATURATED)
def test_saturated_rows(mr, T, E, k, dtype):
    """Rows whose logits spread by more than about 87: the kernels flush p
    below 2^-126 to zero, the oracle keeps it in fp64; everything else must
    match as usual (the parity rules admit FLT_MIN of absolute error)."""
    logits = _saturated_logits(T, E, dtype, seed=T + E)
    x = to_device(logits, dtype)
    st = mr.moe_router_step(x, k, 0.01, 1.25, n_ranks=8, grad_scale=1.0)
    fw = mr.moe_router_fwd(x, k, 0.01, n_ranks=8)
    torch.cuda.synchronize()
    want = oracle_forward(logits, dtype, k, 0.01, None, 8)
    check_forward(st, want, 8)
    check_forward(fw, want, 8)
    check_dispatch(st, want["idx"], E, oracle.dispatch.capacity(T, k, E, 1.25))
    check_backward(st["dlogits"], logits, dtype, want["f"], 0.01, 1.0)
    dl = mr.moe_router_bwd(x, st["f"], 0.01, 1.0)
    torch.cuda.synchronize()
    assert torch.equal(dl, st["dlogits"])


def test_candidate_path_when_the_hot_experts_change(mr):
    """The fast top-k path takes its candidates from each CTA's first rows.
    Here the first half of the batch favours one set of experts and the second
    half another, so the candidates go stale and rows fall back to the full
    path; unskewed rows at the end make the check fail outright.  Every result
    must still match the oracle."""
    T, E, k = 40000, 384, 6
    rng = np.random.default_rng(21)
    z = rng.standard_normal((T, E)).astype(np.float32)
    hot_a = rng.choice(E, 24, replace=False)
    hot_b = rng.choice(np.setdiff1d(np.arange(E), hot_a), 24, replace=False)
    z[: T // 2, hot_a] += 3.0
    z[T // 2: 3 * T // 4, hot_b] += 3.0
    logits = synth.f32_to_bf16_bits(z)
    x = to_device(logits, "bf16")
    st = mr.moe_router_step(x, k, 0.001, 1.25, n_ranks=64, grad_scale=1.0)
    fw = mr.moe_router_fwd(x, k, 0.001, n_ranks=64)
    torch.cuda.synchronize()
    want = oracle_forward(logits, "bf16", k, 0.001, None, 64)
    check_forward(st, want, 64)
    check_forward(fw, want, 64)
    check_dispatch(st, want["idx"], E, oracle.dispatch.capacity(T, k, E, 1.25))
    check_backward(st["dlogits"], logits, "bf16", want["f"], 0.001, 1.0)


def test_misaligned_views_take_the_scalar_path(mr):
    T, E, k = 1500, 64, 2
    base = synth.random_logits(T + 1, E, "bf16", seed=3)
    flat = to_device(base, "bf16").reshape(-1)
    x = flat[3:3 + T * E].view(T, E)             # 6-byte offset: not 16-byte aligned
    logits = base.reshape(-1)[3:3 + T * E].reshape(T, E)
    fw = mr.moe_router_fwd(x, k, 0.01)
    dl_buf = torch.empty(T * E + 1, dtype=torch.float32, device="cuda")
    dl = mr.moe_router_bwd(x, fw["f"], 0.01, 1.0, dlogits=dl_buf[1:].view(T, E))
    torch.cuda.synchronize()
    want = oracle_forward(logits, "bf16", k, 0.01, None, 0)
    check_forward(fw, want, 0)
    check_backward(dl, logits, "bf16", want["f"], 0.01, 1.0)


def test_dispatch_of_arbitrary_assignments(mr):
    # user-supplied idx may repeat an expert within a token; the sort stays stable
    rng = np.random.default_rng(9)
    T, k, E = 5000, 3, 37
    idx = rng.integers(0, E, size=(T, k)).astype(np.int32)
    idx[:50] = 5                                    # a burst on one expert
    got = mr.moe_dispatch(torch.from_numpy(idx).cuda(), E, 0.8)
    torch.cuda.synchronize()
    C = oracle.dispatch.capacity(T, k, E, 0.8)
    check_dispatch(got, idx, E, C)


def test_uniform_routing_gives_unit_balance(mr):
    # [P2] §2.2: uniform routing makes E * sum f P equal to 1
    T, E = 4096, 16
    z = np.zeros((T, E), dtype=np.float32)
    z[np.arange(T), np.arange(T) % E] = 5.0
    fw = mr.moe_router_fwd(to_device(z, "fp32"), 1, 0.01)
    torch.cuda.synchronize()
    assert_equal("counts", fw["counts"].cpu().numpy(), np.full(E, T // E))
    sc = fw["scalars"].cpu().numpy()
    want = oracle_forward(z, "fp32", 1, 0.01, None, 0)
    assert abs(sc[1] - want["balance"]) <= 1e-5 * want["balance"]
    assert sc[2] == 0.0                             # CV of equal counts


# ----------------------------------------------------------------------------- shared-memory fallbacks

# Token counts past what the fused step keeps in shared memory per CTA at 152
# CTAs: E = 256 / k = 8 with 2.4M assignments (over 12288 per CTA: the dispatch
# ranks go through global memory), and E = 64 / k = 2 with 700k tokens (over
# 4096 rows per CTA: the backward recomputes each row's max and sum).
FALLBACK_CASES = [("zipf-hot-top8-T131072-E256", 300_000), ("zipf-top2-T65536-E64", 700_000)]


@pytest.mark.slow
@pytest.mark.parametrize("name,T", FALLBACK_CASES)
def test_step_past_the_shared_memory_buffers(mr, name, T):
    w, logits = workload_inputs(name, T)
    x = to_device(logits, w.dtype)
    st = mr.moe_router_step(x, w.k, w.alpha, w.capacity_factor, renorm=int(w.renorm), n_ranks=w.n_ranks)
    torch.cuda.synchronize()
    want = oracle_forward(logits, w.dtype, w.k, w.alpha, w.renorm, w.n_ranks)
    check_forward(st, want, w.n_ranks)
    C = oracle.dispatch.capacity(w.T, w.k, w.E, w.capacity_factor)
    check_dispatch(st, want["idx"], w.E, C)
    check_backward(st["dlogits"], logits, w.dtype, want["f"], w.alpha, 1.0)


@pytest.mark.slow
def test_dispatch_past_the_shared_memory_buffer(mr):
    """Given assignments over 12288 per CTA: the ranks go through global memory."""
    rng = np.random.default_rng(11)
    T, E, k = 300_000, 256, 8
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)   # k distinct experts per token
    C = oracle.dispatch.capacity(T, k, E, 1.0)
    got = mr.moe_dispatch(torch.from_numpy(idx).cuda(), E, 1.0)
    torch.cuda.synchronize()
    assert got["capacity"] == C
    check_dispatch(got, idx, E, C)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("E,k", [(64, 2), (256, 8), (384, 6), (7, 3)])
def test_signed_zero_ties(mr, dtype, E, k):
    """-0.0 and +0.0 are equal logits: the lower column wins between them."""
    rng = np.random.default_rng(E * 10 + k)
    T = 1201
    z = rng.choice(np.array([-0.0, 0.0, -0.0, 0.0, -1.0, -2.5, 0.5]), size=(T, E)).astype(np.float32)
    z[::7] = rng.choice(np.array([-0.0, 0.0], dtype=np.float32), size=(len(z[::7]), E))   # rows of zeros only
    logits = z if dtype == "fp32" else synth.f32_to_bf16_bits(z)
    x = to_device(logits, dtype)
    st = mr.moe_router_step(x, k, 0.01, 1.0, n_ranks=0, grad_scale=1.0)
    torch.cuda.synchronize()
    want = oracle_forward(logits, dtype, k, 0.01, None, 0)
    check_forward(st, want, 0)
    check_dispatch(st, want["idx"], E, oracle.dispatch.capacity(T, k, E, 1.0))
    check_backward(st["dlogits"], logits, dtype, want["f"], 0.01, 1.0)


@pytest.mark.parametrize("E,k", [(64, 8), (64, 3), (56, 7)])
def test_small_expert_counts_equal_separate_calls(mr, E, k):
    """At E <= 64 (one or two vectors per lane) the separate calls give the fused step's bits."""
    logits = synth.random_logits(3001, E, "bf16", seed=E + k, scale=2.0)
    x = to_device(logits, "bf16")
    st = mr.moe_router_step(x, k, 0.01, 1.25, n_ranks=0, grad_scale=1.0)
    fw = mr.moe_router_fwd(x, k, 0.01, n_ranks=0)
    dp = mr.moe_dispatch(fw["idx"], E, 1.25)
    dl = mr.moe_router_bwd(x, fw["f"], 0.01, 1.0)
    torch.cuda.synchronize()
    want = oracle_forward(logits, "bf16", k, 0.01, None, 0)
    check_forward(st, want, 0)
    check_dispatch(st, want["idx"], E, oracle.dispatch.capacity(3001, k, E, 1.25))
    check_backward(st["dlogits"], logits, "bf16", want["f"], 0.01, 1.0)
    check_step_equals_separate(st, fw, dp, dl)


def test_back_to_back_calls_on_one_workspace(mr):
    """Launches queued without a host sync on one workspace (each may be scheduled
    while the previous one finishes): steps, forwards and dispatches of different
    sizes in turn, every result checked afterwards."""
    ws = mr.Workspace()
    ws.ensure(262144, 1024, 8)           # one buffer for every call below, whatever its E
    cases = [("zipf-top2-T65536-E64", 20001), ("zipf-hot-top8-T131072-E256", 9001), ("switch-top1-T4096-E8", 4096),
             ("zipf-ep64-top6-T262144-E384", 7001), ("zipf-top2-T65536-E64", 3001)]
    runs = []
    for name, T in cases:
        w, logits = workload_inputs(name, T)
        x = to_device(logits, w.dtype)
        st = mr.moe_router_step(x, w.k, w.alpha, w.capacity_factor, renorm=int(w.renorm), n_ranks=w.n_ranks, ws=ws)
        fw = mr.moe_router_fwd(x, w.k, w.alpha, renorm=int(w.renorm), n_ranks=w.n_ranks, ws=ws)
        dp = mr.moe_dispatch(fw["idx"], w.E, w.capacity_factor, ws=ws)
        runs.append((w, logits, st, fw, dp))
    torch.cuda.synchronize()
    assert mr.moe_get_device_status(ws) == 0
    for w, logits, st, fw, dp in runs:
        want = oracle_forward(logits, w.dtype, w.k, w.alpha, w.renorm, w.n_ranks)
        check_forward(st, want, w.n_ranks)
        check_forward(fw, want, w.n_ranks)
        C = oracle.dispatch.capacity(w.T, w.k, w.E, w.capacity_factor)
        check_dispatch(st, want["idx"], w.E, C)
        check_dispatch(dp, want["idx"], w.E, C)
        check_backward(st["dlogits"], logits, w.dtype, want["f"], w.alpha, 1.0)
