"""Data-parallel batch statistics, emulated on one GPU: the batch is split into
G shards routed by separate calls, moe_router_combine merges their counts and P,
and each shard's backward takes the batch's f.  The merged counts must equal
the unsharded call's and the oracle's bit for bit; f, P, the scalars and the
gradient must match the oracle's whole-batch values within the router's
tolerances (parity.py)."""

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import FLT_MIN, RTOL, SCALARS, assert_close, assert_equal, check_backward, oracle_forward, to_device, workload_inputs

pytestmark = pytest.mark.gpu

WORKLOADS = list(synth.ROUTER_WORKLOADS)


@pytest.fixture(scope="module")
def mr(native_lib):
    import moe_expert_routing_router_gb300 as m
    return m


@pytest.mark.parametrize("name", WORKLOADS)
@pytest.mark.parametrize("G", [2, 3, 8])
def test_sharded_statistics(mr, name, G):
    w, logits = workload_inputs(name, 20011 if large(name) else None)
    T = w.T
    cuts = np.linspace(0, T, G + 1).astype(int)
    cuts[1] -= 7                                          # shards of unequal size
    x = to_device(logits, w.dtype)
    counts, Ps, Ts = [], [], []
    for s in range(G):
        out = mr.moe_router_fwd(x[cuts[s]:cuts[s + 1]], w.k, w.alpha, renorm=int(w.renorm), n_ranks=w.n_ranks)
        counts.append(out["counts"])
        Ps.append(out["P"])
        Ts.append(int(cuts[s + 1] - cuts[s]))
    got = mr.moe_router_combine(torch.stack(counts), torch.stack(Ps), Ts, w.k, w.alpha, n_ranks=w.n_ranks)
    whole = mr.moe_router_fwd(x, w.k, w.alpha, renorm=int(w.renorm), n_ranks=w.n_ranks)
    torch.cuda.synchronize()
    want = oracle_forward(logits, w.dtype, w.k, w.alpha, w.renorm, w.n_ranks)
    assert_equal("counts", got["counts"].cpu().numpy(), want["counts"])
    assert_equal("counts vs unsharded", got["counts"].cpu().numpy(), whole["counts"].cpu().numpy())
    assert_close("f", got["f"].cpu().numpy(), want["f"], RTOL)
    assert_close("P", got["P"].cpu().numpy(), want["P"], RTOL, FLT_MIN)
    sc = got["scalars"].cpu().numpy()
    for j, nm in enumerate(SCALARS):
        assert_close(f"scalar {nm}", sc[j], want[nm], RTOL)
    if w.n_ranks:
        assert_equal("rank_load", got["rank_load"].cpu().numpy(), want["rank_load"])
    # each shard's backward with the batch's f and its coefficient rescaled to the batch's T
    from moe_expert_routing_router_gb300 import dp
    f32 = want["f"].astype(np.float32)
    parts = []
    for s in range(G):
        g = dp.shard_grad_scale(1.0, Ts[s], T)
        parts.append(mr.moe_router_bwd(x[cuts[s]:cuts[s + 1]], torch.from_numpy(f32).cuda(), w.alpha, g))
    dl = torch.cat(parts)
    torch.cuda.synchronize()
    check_backward(dl, logits, w.dtype, f32.astype(np.float64), w.alpha, 1.0)


def large(name: str) -> bool:
    """Workloads above 65536 tokens are split at 20011 tokens (the full sizes are
    covered by the unsharded parity tests)."""
    return synth.ROUTER_WORKLOADS[name].T > 65536


@pytest.mark.parametrize("masked", [False, True])
def test_sharded_masked_p_and_bias(mr, masked):
    """The combine takes the bias-routing forward's statistics too (masked P included)."""
    w, logits = workload_inputs("zipf-top2-T65536-E64", 12007)
    x = to_device(logits, w.dtype)
    bias = torch.from_numpy((np.random.default_rng(5).standard_normal(w.E) * 0.5).astype(np.float32)).cuda()
    cuts = [0, 5000, 12007]
    outs = [mr.moe_router_fwd_ex(x[a:b], w.k, w.alpha, bias=bias, masked_p=masked) for a, b in zip(cuts, cuts[1:])]
    got = mr.moe_router_combine(torch.stack([o["counts"] for o in outs]), torch.stack([o["P"] for o in outs]),
                                [b - a for a, b in zip(cuts, cuts[1:])], w.k, w.alpha, masked_p=masked)
    whole = mr.moe_router_fwd_ex(x, w.k, w.alpha, bias=bias, masked_p=masked)
    torch.cuda.synchronize()
    assert_equal("counts", got["counts"].cpu().numpy(), whole["counts"].cpu().numpy())
    for key in ("f", "P", "scalars"):
        assert_close(key, got[key].cpu().numpy(), whole[key].cpu().numpy().astype(np.float64), 2 * RTOL)
