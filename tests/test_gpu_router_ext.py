"""GPU parity of the method's next steps through the C ABI against the CPU oracle:
bias routing and the bias update ([P1] §4.3), masked P ([P2] §3.1) and the full
router backward through the gates.

Tolerances are those of ``parity.py``: idx, counts, rank loads and the updated
bias bit-exact (the bias step is one fp32 addition on both sides); gate, f, P
and the scalars within 1e-5 relative; dlogits within
1e-5 * (|o| + p * (|dp| + sum_i p_i |dp_i|)) -- the gradient p * (dp - sum p dp)
is a difference that cancels, so 1e-5 relative is taken against the size of
its terms.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import FLT_MIN, RTOL, SCALARS, assert_close, assert_equal, to_device, workload_inputs

pytestmark = pytest.mark.gpu

R, X = oracle.router, oracle.routing_ext
WORKLOADS = list(synth.ROUTER_WORKLOADS)
SMALL_T = {"switch-top1-T4096-E8": 1001, "zipf-top2-T65536-E64": 3001,
           "zipf-hot-top8-T131072-E256": 2999, "zipf-ep64-top6-T262144-E384": 3007}
GAMMA = 0.001


@pytest.fixture(scope="module")
def mr(native_lib):
    import moe_expert_routing_router_gb300 as m
    return m


def seeded_bias(E: int, seed: int = 7) -> np.ndarray:
    """A bias of the size the update rule reaches after a few hundred steps."""
    return (np.random.default_rng(seed).standard_normal(E) * 0.5).astype(np.float32)


def oracle_forward_ex(logits, dtype, k, alpha, renorm, n_ranks, bias, masked, gamma, chunk=16384) -> dict:
    """The oracle's forward with bias selection / masked P, over row chunks."""
    T, E = logits.shape
    b = np.zeros(E, np.float32) if bias is None else bias
    idx = np.empty((T, k), dtype=np.int64)
    gate = np.empty((T, k))
    psum = np.zeros(E)
    for r0 in range(0, T, chunk):
        sl = logits[r0:r0 + chunk]
        p = R.softmax(R.widen(sl, dtype))
        i = X.top_k_biased(sl, dtype, b, k)
        idx[r0:r0 + chunk] = i
        gate[r0:r0 + chunk] = R.gates(p, i, renorm)
        psum += (X.mean_router_prob_masked(p, i, k) * (p.shape[0] * k) if masked else p.sum(axis=0))
    counts = R.expert_counts(idx, E)
    P = psum / (T * k) if masked else psum / T
    out = R.batch_statistics(counts, P, T, k, alpha, n_ranks)
    out["idx"], out["gate"] = idx, gate
    out["bias_out"] = X.bias_update(b, counts, T, k, gamma)
    return out


def check_forward(got: dict, want: dict, n_ranks: int) -> None:
    assert_equal("idx", got["idx"].cpu().numpy(), want["idx"])
    assert_close("gate", got["gate"].cpu().numpy(), want["gate"], RTOL, FLT_MIN)
    assert_equal("counts", got["counts"].cpu().numpy(), want["counts"])
    assert_close("f", got["f"].cpu().numpy(), want["f"], RTOL)
    assert_close("P", got["P"].cpu().numpy(), want["P"], RTOL, FLT_MIN)
    sc = got["scalars"].cpu().numpy()
    for j, name in enumerate(SCALARS):
        assert_close(f"scalar {name}", sc[j], want[name], RTOL)
    if n_ranks > 0:
        assert_equal("rank_load", got["rank_load"].cpu().numpy(), want["rank_load"])
    if "bias_out" in got:
        g = got["bias_out"].cpu().numpy()
        assert g.dtype == np.float32
        assert np.array_equal(g.view(np.uint32), want["bias_out"].view(np.uint32)), "bias_out not bit-exact"


def run_fwd_ex(mr, w, logits, bias, masked, gamma=GAMMA):
    x = to_device(logits, w.dtype)
    bt = None if bias is None else torch.from_numpy(bias).cuda()
    got = mr.moe_router_fwd_ex(x, w.k, w.alpha, renorm=int(w.renorm), n_ranks=w.n_ranks, bias=bt,
                               masked_p=masked, bias_gamma=gamma, bias_out=True)
    torch.cuda.synchronize()
    return x, got


@pytest.mark.parametrize("name", WORKLOADS)
@pytest.mark.parametrize("size", ["small", "full"])
def test_bias_routing_parity(mr, name, size):
    w, logits = workload_inputs(name, SMALL_T[name] if size == "small" else None)
    bias = seeded_bias(w.E)
    _, got = run_fwd_ex(mr, w, logits, bias, masked=False)
    want = oracle_forward_ex(logits, w.dtype, w.k, w.alpha, w.renorm, w.n_ranks, bias, False, GAMMA)
    check_forward(got, want, w.n_ranks)


@pytest.mark.parametrize("name", WORKLOADS)
@pytest.mark.parametrize("size", ["small", "full"])
def test_masked_p_parity(mr, name, size):
    w, logits = workload_inputs(name, SMALL_T[name] if size == "small" else None)
    _, got = run_fwd_ex(mr, w, logits, None, masked=True)
    want = oracle_forward_ex(logits, w.dtype, w.k, w.alpha, w.renorm, w.n_ranks, None, True, GAMMA)
    check_forward(got, want, w.n_ranks)


@pytest.mark.parametrize("name", WORKLOADS)
def test_zero_bias_unmasked_matches_moe_router_fwd(mr, name):
    w, logits = workload_inputs(name, SMALL_T[name])
    x, got = run_fwd_ex(mr, w, logits, np.zeros(w.E, np.float32), masked=False)
    ref = mr.moe_router_fwd(x, w.k, w.alpha, renorm=int(w.renorm), n_ranks=w.n_ranks)
    torch.cuda.synchronize()
    for key in ("idx", "counts", "rank_load"):
        assert_equal(key, got[key].cpu().numpy(), ref[key].cpu().numpy())
    for key in ("gate", "f", "P", "scalars"):
        assert_close(key, got[key].cpu().numpy(), ref[key].cpu().numpy().astype(np.float64), 2 * RTOL)


def test_bias_update_in_place_over_steps(mr):
    """Five steps of routing + in-place update on one batch follow the oracle's
    iteration bit for bit, and the load CV falls."""
    w, logits = workload_inputs("zipf-top2-T65536-E64", 4096)
    x = to_device(logits, w.dtype)
    gamma = 0.05
    bias_d = torch.zeros(w.E, dtype=torch.float32, device="cuda")
    b = np.zeros(w.E, np.float32)
    cvs = []
    for _ in range(5):
        got = mr.moe_router_fwd_ex(x, w.k, w.alpha, renorm=1, bias=bias_d, bias_gamma=gamma, bias_out=bias_d)
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
def test_ties_and_edge_shapes(mr, E, k, dtype):
    """Integer logits and integer biases: the fp32 sums tie everywhere, so the
    lower-index rule decides most picks (and the collision check hands many
    rows to the 64-bit keys); E not a multiple of the vector width, k = E and
    E = 1 are covered."""
    rng = np.random.default_rng(E * 10 + k)
    T = 777
    z = rng.integers(-3, 4, size=(T, E)).astype(np.float32)
    logits = synth.f32_to_bf16_bits(z) if dtype == "bf16" else z
    bias = rng.integers(-2, 3, size=E).astype(np.float32)
    x = to_device(logits, dtype)
    for masked in (False, True):
        got = mr.moe_router_fwd_ex(x, k, 0.01, renorm=-1, bias=torch.from_numpy(bias).cuda(), masked_p=masked,
                                   bias_gamma=0.25, bias_out=True)
        torch.cuda.synchronize()
        want = oracle_forward_ex(logits, dtype, k, 0.01, k > 1, 0, bias, masked, 0.25)
        check_forward(got, want, 0)


def test_single_token(mr):
    logits = np.array([[0.5, -1.0, 2.0, 2.0, 0.0, 1.5, -0.25, 3.0]], np.float32)
    bias = np.array([0, 0, 0, 0, 0, 0, 0, -2.0], np.float32)
    x = to_device(logits, "fp32")
    got = mr.moe_router_fwd_ex(x, 2, 0.01, bias=torch.from_numpy(bias).cuda(), bias_gamma=0.5, bias_out=True)
    torch.cuda.synchronize()
    want = oracle_forward_ex(logits, "fp32", 2, 0.01, True, 0, bias, False, 0.5)
    check_forward(got, want, 0)
    assert got["idx"].cpu().tolist() == [[2, 3]]


# ----------------------------------------------------------------------------- full backward

def check_backward_full(dl: torch.Tensor, logits, dtype, f, alpha, g, idx, dgate, renorm, masked,
                        chunk=16384) -> None:
    T, E = logits.shape
    k = idx.shape[1]
    got = dl.cpu().numpy()
    for r0 in range(0, T, chunk):
        sl = logits[r0:r0 + chunk]
        i = idx[r0:r0 + chunk]
        dg = None if dgate is None else dgate[r0:r0 + chunk].astype(np.float64)
        want = X.router_backward_full(sl, dtype, f, alpha, g, i, dg, renorm, masked, T=T)
        p = R.softmax(R.widen(sl, dtype))
        dp = X.grad_wrt_probs(p, i, f, alpha, g, T, k, dg, renorm, masked)
        scale = p * (np.abs(dp) + (p * np.abs(dp)).sum(axis=1, keepdims=True))
        assert_close(f"dlogits rows {r0}..", got[r0:r0 + chunk], want, RTOL, RTOL * scale + FLT_MIN)


def _picks(logits, dtype, k):
    return np.concatenate([R.top_k(R.widen(logits[r:r + 16384], dtype), k) for r in range(0, logits.shape[0], 16384)])


@pytest.mark.parametrize("name", WORKLOADS)
@pytest.mark.parametrize("size", ["small", "full"])
@pytest.mark.parametrize("masked", [False, True])
def test_backward_full_parity(mr, name, size, masked):
    w, logits = workload_inputs(name, SMALL_T[name] if size == "small" else None)
    if size == "full" and masked and w.E > 64:
        pytest.skip("masked full-size case covered at E <= 64; small sizes cover every E")
    x = to_device(logits, w.dtype)
    rng = np.random.default_rng(9)
    f = rng.random(w.E).astype(np.float32)
    f /= f.sum()
    idx = _picks(logits, w.dtype, w.k)
    dgate = rng.standard_normal((w.T, w.k)).astype(np.float32)
    dl = mr.moe_router_bwd_full(x, torch.from_numpy(f).cuda(), w.alpha, grad_scale=1.5,
                                idx=torch.from_numpy(idx.astype(np.int32)).cuda(),
                                dgate=torch.from_numpy(dgate).cuda(), renorm=int(w.renorm), masked_p=masked)
    torch.cuda.synchronize()
    check_backward_full(dl, logits, w.dtype, f.astype(np.float64), w.alpha, 1.5, idx, dgate, w.renorm, masked)


@pytest.mark.parametrize("renorm", [0, 1])
@pytest.mark.parametrize("E,k,dtype", [(40, 3, "fp32"), (8, 8, "bf16"), (1, 1, "fp32"), (384, 6, "bf16")])
def test_backward_full_gate_only_and_shapes(mr, renorm, E, k, dtype):
    """alpha = 0 leaves the gate term alone (with renormalised gates it is zero
    on the unpicked experts); ragged E, k = E and E = 1 are covered."""
    rng = np.random.default_rng(E + k + renorm)
    T = 513
    z = (rng.standard_normal((T, E)) * 2.0).astype(np.float32)
    logits = synth.f32_to_bf16_bits(z) if dtype == "bf16" else z
    x = to_device(logits, dtype)
    f = np.full(E, 1.0 / E, np.float32)
    idx = _picks(logits, dtype, k)
    dgate = rng.standard_normal((T, k)).astype(np.float32)
    dl = mr.moe_router_bwd_full(x, torch.from_numpy(f).cuda(), 0.0, idx=torch.from_numpy(idx.astype(np.int32)).cuda(),
                                dgate=torch.from_numpy(dgate).cuda(), renorm=renorm)
    torch.cuda.synchronize()
    check_backward_full(dl, logits, dtype, f.astype(np.float64), 0.0, 1.0, idx, dgate, bool(renorm), False)


@pytest.mark.parametrize("name", WORKLOADS)
def test_backward_full_without_dgate_matches_moe_router_bwd(mr, name):
    w, logits = workload_inputs(name, SMALL_T[name])
    x = to_device(logits, w.dtype)
    f = np.random.default_rng(3).random(w.E).astype(np.float32)
    f /= f.sum()
    ft = torch.from_numpy(f).cuda()
    a = mr.moe_router_bwd_full(x, ft, w.alpha, grad_scale=2.0, k=w.k)
    b = mr.moe_router_bwd(x, ft, w.alpha, grad_scale=2.0)
    torch.cuda.synchronize()
    check_backward_full(a, logits, w.dtype, f.astype(np.float64), w.alpha, 2.0,
                        np.zeros((w.T, w.k), np.int64), None, w.renorm, False)
    bb = b.cpu().numpy().astype(np.float64)
    p = R.softmax(R.widen(logits, w.dtype))
    c = 2.0 * w.alpha * w.E / w.T
    scale = c * p * (f[None, :] + (p * f[None, :]).sum(axis=1, keepdims=True))
    assert_close("bwd_full vs bwd", a.cpu().numpy(), bb, 0.0, 4 * RTOL * scale + 1e-30)


def test_interleaved_with_the_fused_step_on_one_workspace(mr):
    """The forward's accumulators share the workspace with the fused step's
    group sums: calls of both kinds and of different E follow each other on
    one workspace, without a host sync, and each stays exact."""
    ws = mr.Workspace()
    cases = []
    for name in ("zipf-top2-T65536-E64", "zipf-ep64-top6-T262144-E384"):
        w, logits = workload_inputs(name, 2047)
        cases.append((w, logits, to_device(logits, w.dtype), seeded_bias(w.E, 11)))
    outs = []
    for rep in range(2):
        for w, logits, x, bias in cases:
            st = mr.moe_router_step(x, w.k, w.alpha, w.capacity_factor, renorm=int(w.renorm), n_ranks=w.n_ranks, ws=ws)
            fx = mr.moe_router_fwd_ex(x, w.k, w.alpha, renorm=int(w.renorm), n_ranks=w.n_ranks,
                                      bias=torch.from_numpy(bias).cuda(), masked_p=bool(rep), bias_gamma=GAMMA,
                                      bias_out=True, ws=ws)
            outs.append((w, logits, bias, bool(rep), st, fx))
    torch.cuda.synchronize()
    for w, logits, bias, masked, st, fx in outs:
        plain = oracle_forward_ex(logits, w.dtype, w.k, w.alpha, w.renorm, w.n_ranks, None, False, GAMMA)
        assert_equal("step counts", st["counts"].cpu().numpy(), plain["counts"])
        assert_equal("step idx", st["idx"].cpu().numpy(), plain["idx"])
        want = oracle_forward_ex(logits, w.dtype, w.k, w.alpha, w.renorm, w.n_ranks, bias, masked, GAMMA)
        check_forward(fx, want, w.n_ranks)


@pytest.mark.parametrize("E,dtype", [(384, "fp32"), (512, "fp32"), (384, "bf16")])
def test_scores_equal_in_their_upper_bits(mr, E, dtype):
    """Scores that differ only below the upper 22 bits of their image (fp32
    logits 1.5 + j * 2^-20, or bf16 logits with biases of that size): the
    32-bit selection keys must see the collision and leave the row to the
    64-bit keys."""
    rng = np.random.default_rng(E)
    T, k = 517, 6
    if dtype == "fp32":
        z = (np.float32(1.5) + rng.integers(0, 3, size=(T, E)).astype(np.float32) * np.float32(2.0 ** -20))
        logits, bias = z.astype(np.float32), np.zeros(E, np.float32)
    else:
        logits = synth.f32_to_bf16_bits(np.full((T, E), 1.5, np.float32) + rng.integers(0, 2, size=(T, E)).astype(np.float32))
        bias = (rng.integers(0, 3, size=E) * 2.0 ** -19).astype(np.float32)
    x = to_device(logits, dtype)
    got = mr.moe_router_fwd_ex(x, k, 0.01, bias=torch.from_numpy(bias).cuda(), bias_gamma=0.5, bias_out=True)
    torch.cuda.synchronize()
    check_forward(got, oracle_forward_ex(logits, dtype, k, 0.01, True, 0, bias, False, 0.5), 0)


@pytest.mark.parametrize("name", ["zipf-top2-T65536-E64", "zipf-ep64-top6-T262144-E384"])
def test_repeated_calls_are_bit_identical(mr, name):
    """The per-expert sums are added in a fixed order (masked P included, whose
    picks from several rows of a warp may share an expert): two calls give the
    same bits in every output."""
    w, logits = workload_inputs(name, 20011)
    x = to_device(logits, w.dtype)
    bias = torch.from_numpy(seeded_bias(w.E)).cuda()
    for masked in (False, True):
        a = mr.moe_router_fwd_ex(x, w.k, w.alpha, renorm=int(w.renorm), n_ranks=w.n_ranks, bias=bias, masked_p=masked,
                                 bias_gamma=GAMMA, bias_out=True)
        b = mr.moe_router_fwd_ex(x, w.k, w.alpha, renorm=int(w.renorm), n_ranks=w.n_ranks, bias=bias, masked_p=masked,
                                 bias_gamma=GAMMA, bias_out=True)
        torch.cuda.synchronize()
        for key in ("idx", "gate", "counts", "f", "P", "scalars", "bias_out"):
            ta, tb = a[key].cpu(), b[key].cpu()
            assert torch.equal(ta.view(torch.int32) if ta.dtype == torch.float32 else ta,
                               tb.view(torch.int32) if tb.dtype == torch.float32 else tb), (key, masked)
