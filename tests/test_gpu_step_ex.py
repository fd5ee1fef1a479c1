"""GPU parity of the extended step (moe_router_step_ex: bias routing and its
update, masked P, dispatch, and the backward of the gates' upstream gradient
added to the aux loss's, in one launch) through the C ABI against the CPU
oracle: oracle.routing_ext's forward and full backward and oracle.dispatch on
the oracle's picks.

Tolerances are those of the separate calls' tests (test_gpu_router_ext.py):
idx, counts, rank loads, the updated bias and every dispatch output bit-exact;
gate, f, P and the scalars within 1e-5 relative; dlogits within
1e-5 * (|o| + p * (|dp| + sum_i p_i |dp_i|)).
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import RTOL, assert_close, assert_equal, to_device, workload_inputs
from test_gpu_router_ext import GAMMA, SMALL_T, check_backward_full, check_forward, oracle_forward_ex, seeded_bias

pytestmark = pytest.mark.gpu

WORKLOADS = list(synth.ROUTER_WORKLOADS)
G_SCALE = 1.5


@pytest.fixture(scope="module")
def mr(native_lib):
    import moe_expert_routing_router_gb300 as m
    return m


def run_step_ex(mr, logits, dtype, k, alpha, cf, renorm, n_ranks, bias, masked, dgate, gamma=GAMMA, ws=None):
    x = to_device(logits, dtype)
    bt = None if bias is None else torch.from_numpy(bias).cuda()
    dg = None if dgate is None else torch.from_numpy(dgate).cuda()
    got = mr.moe_router_step_ex(x, k, alpha, cf, renorm=int(renorm), n_ranks=n_ranks, grad_scale=G_SCALE, bias=bt,
                                bias_gamma=gamma, bias_out=True, masked_p=masked, dgate=dg, ws=ws)
    torch.cuda.synchronize()
    return got


def check_step_ex(got, logits, dtype, k, alpha, cf, renorm, n_ranks, bias, masked, dgate, gamma=GAMMA):
    T, E = logits.shape
    want = oracle_forward_ex(logits, dtype, k, alpha, renorm, n_ranks, bias, masked, gamma)
    check_forward(got, want, n_ranks)
    C = oracle.dispatch.capacity(T, k, E, cf)
    disp = oracle.dispatch.dispatch(want["idx"], E, C)
    for key in ("perm", "slot", "offsets", "kept"):
        assert_equal(key, got[key].cpu().numpy(), disp[key])
    assert int(got["n_dropped"].item()) == disp["n_dropped"]
    assert got["capacity"] == C
    f32 = want["f"].astype(np.float32).astype(np.float64)      # the f the kernel holds (fp32 of counts / (T*k))
    check_backward_full(got["dlogits"], logits, dtype, f32, alpha, G_SCALE, want["idx"], dgate, renorm, masked)


CASES = [(True, False, True), (False, True, True), (True, True, False), (True, True, True)]


@pytest.mark.parametrize("name", WORKLOADS)
@pytest.mark.parametrize("bias_on,masked,with_dgate", CASES)
def test_step_ex_parity_small(mr, name, bias_on, masked, with_dgate):
    """Every workload at a size the oracle runs in seconds (several row stages,
    a ragged tail), with and without bias, masked P and dgate."""
    w, logits = workload_inputs(name, SMALL_T[name])
    bias = seeded_bias(w.E) if bias_on else None
    dgate = np.random.default_rng(w.E).standard_normal((w.T, w.k)).astype(np.float32) if with_dgate else None
    got = run_step_ex(mr, logits, w.dtype, w.k, w.alpha, w.capacity_factor, w.renorm, w.n_ranks, bias, masked, dgate)
    check_step_ex(got, logits, w.dtype, w.k, w.alpha, w.capacity_factor, w.renorm, w.n_ranks, bias, masked, dgate)


@pytest.mark.parametrize("name", WORKLOADS)
def test_step_ex_parity_full(mr, name):
    """The full workload sizes, in the launch configuration the benchmark times
    (biased selection, unmasked P, the gates' upstream gradient)."""
    w, logits = workload_inputs(name)
    bias = seeded_bias(w.E)
    dgate = np.random.default_rng(5).standard_normal((w.T, w.k)).astype(np.float32)
    got = run_step_ex(mr, logits, w.dtype, w.k, w.alpha, w.capacity_factor, w.renorm, w.n_ranks, bias, False, dgate)
    check_step_ex(got, logits, w.dtype, w.k, w.alpha, w.capacity_factor, w.renorm, w.n_ranks, bias, False, dgate)


def test_step_ex_masked_full_e64(mr):
    w, logits = workload_inputs("zipf-top2-T65536-E64")
    bias = seeded_bias(w.E, 3)
    dgate = np.random.default_rng(6).standard_normal((w.T, w.k)).astype(np.float32)
    got = run_step_ex(mr, logits, w.dtype, w.k, w.alpha, w.capacity_factor, w.renorm, w.n_ranks, bias, True, dgate)
    check_step_ex(got, logits, w.dtype, w.k, w.alpha, w.capacity_factor, w.renorm, w.n_ranks, bias, True, dgate)


@pytest.mark.parametrize("name", WORKLOADS)
def test_step_ex_plain_matches_step(mr, name):
    """No bias, unmasked P and no dgate: the step of moe_router_step, integers
    bit for bit and the floats within rounding."""
    w, logits = workload_inputs(name, SMALL_T[name])
    x = to_device(logits, w.dtype)
    a = mr.moe_router_step_ex(x, w.k, w.alpha, w.capacity_factor, renorm=int(w.renorm), n_ranks=w.n_ranks,
                              grad_scale=G_SCALE)
    b = mr.moe_router_step(x, w.k, w.alpha, w.capacity_factor, renorm=int(w.renorm), n_ranks=w.n_ranks,
                           grad_scale=G_SCALE)
    torch.cuda.synchronize()
    for key in ("idx", "counts", "rank_load", "perm", "slot", "offsets", "kept", "n_dropped"):
        assert_equal(key, a[key].cpu().numpy(), b[key].cpu().numpy())
    for key in ("gate", "f", "P", "scalars"):
        assert_close(key, a[key].cpu().numpy(), b[key].cpu().numpy().astype(np.float64), 2 * RTOL)
    assert "bias_out" not in a


def test_step_ex_bias_in_place_over_steps(mr):
    """Four steps of the extended step with the bias updated in place follow
    the oracle's iteration bit for bit (picks and bias), and the load CV falls."""
    w, logits = workload_inputs("zipf-top2-T65536-E64", 4096)
    x = to_device(logits, w.dtype)
    gamma = 0.05
    bias_d = torch.zeros(w.E, dtype=torch.float32, device="cuda")
    b = np.zeros(w.E, np.float32)
    cvs = []
    for _ in range(4):
        got = mr.moe_router_step_ex(x, w.k, w.alpha, w.capacity_factor, renorm=1, bias=bias_d, bias_gamma=gamma,
                                    bias_out=bias_d)
        torch.cuda.synchronize()
        want = oracle_forward_ex(logits, w.dtype, w.k, w.alpha, True, 0, b, False, gamma)
        assert_equal("idx", got["idx"].cpu().numpy(), want["idx"])
        b = want["bias_out"]
        assert np.array_equal(bias_d.cpu().numpy().view(np.uint32), b.view(np.uint32))
        cvs.append(float(got["scalars"][2]))
    assert cvs[-1] < cvs[0]


@pytest.mark.parametrize("E,k,dtype", [(40, 3, "fp32"), (64, 2, "bf16"), (8, 8, "bf16"), (1, 1, "fp32"),
                                       (96, 5, "bf16"), (200, 8, "fp32"), (384, 6, "bf16"), (384, 8, "fp32"),
                                       (512, 4, "bf16"), (1000, 8, "fp32"), (1023, 7, "bf16")])
def test_step_ex_ties_and_edge_shapes(mr, E, k, dtype):
    """Integer logits and biases (the fp32 scores tie everywhere, so the
    lower-index rule decides most picks and many lanes hold more than two keys
    above the k-th pick), E off the vector width (the direct variants), k = E
    and E = 1, with masked P and dgate."""
    rng = np.random.default_rng(E * 10 + k)
    T = 777
    z = rng.integers(-3, 4, size=(T, E)).astype(np.float32)
    logits = synth.f32_to_bf16_bits(z) if dtype == "bf16" else z
    bias = rng.integers(-2, 3, size=E).astype(np.float32)
    dgate = rng.standard_normal((T, k)).astype(np.float32)
    for masked in (False, True):
        got = run_step_ex(mr, logits, dtype, k, 0.01, 1.25, k > 1, 0, bias, masked, dgate, gamma=0.25)
        check_step_ex(got, logits, dtype, k, 0.01, 1.25, k > 1, 0, bias, masked, dgate, gamma=0.25)


def test_step_ex_plain_gates_and_single_token(mr):
    """Plain gates (renorm = 0) with k > 1, and a batch of one token."""
    rng = np.random.default_rng(12)
    z = (rng.standard_normal((1500, 64)) * 2.0).astype(np.float32)
    bias = seeded_bias(64, 13)
    dgate = rng.standard_normal((1500, 4)).astype(np.float32)
    got = run_step_ex(mr, z, "fp32", 4, 0.02, 1.0, False, 8, bias, False, dgate)
    check_step_ex(got, z, "fp32", 4, 0.02, 1.0, False, 8, bias, False, dgate)
    one = np.array([[0.5, -1.0, 2.0, 2.0, 0.0, 1.5, -0.25, 3.0]], np.float32)
    b1 = np.array([0, 0, 0, 0, 0, 0, 0, -2.0], np.float32)
    dg1 = np.array([[0.3, -0.7]], np.float32)
    got = run_step_ex(mr, one, "fp32", 2, 0.01, 1.0, True, 0, b1, False, dg1, gamma=0.5)
    check_step_ex(got, one, "fp32", 2, 0.01, 1.0, True, 0, b1, False, dg1, gamma=0.5)
    assert got["idx"].cpu().tolist() == [[2, 3]]
