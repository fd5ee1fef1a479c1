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


def _global_dispatch_case(mr, name: str, cuts, cf: float):
    """Routes the shards [cuts[s], cuts[s+1]) of one batch separately, takes each
    shard's cap_base from the stacked counts and dispatches it with the batch's
    capacity; checks everything against one oracle dispatch of the whole batch."""
    w, logits = workload_inputs(name, int(cuts[-1]))
    G = len(cuts) - 1
    x = to_device(logits, w.dtype)
    want = oracle_forward(logits, w.dtype, w.k, w.alpha, w.renorm, w.n_ranks)
    C = oracle.dispatch.capacity(w.T, w.k, w.E, cf)
    whole = oracle.dispatch.dispatch(want["idx"], w.E, C)
    outs = [mr.moe_router_fwd(x[cuts[s]:cuts[s + 1]], w.k, w.alpha, renorm=int(w.renorm)) for s in range(G)]
    stacked = torch.stack([o["counts"] for o in outs])
    for s in range(G):
        a, b = int(cuts[s]), int(cuts[s + 1])
        idx_ref = want["idx"][a:b]
        base = mr.moe_shard_capacity_base(stacked, s)
        got = mr.moe_dispatch_sharded(outs[s]["idx"], w.E, cf, w.T, base)
        torch.cuda.synchronize()
        assert_equal(f"shard {s} idx", outs[s]["idx"].cpu().numpy(), idx_ref)
        lower = np.bincount(want["idx"][:a].ravel(), minlength=w.E) if a > 0 else np.zeros(w.E, np.int64)
        assert_equal(f"shard {s} cap_base", base.cpu().numpy(), lower)
        local = oracle.dispatch.dispatch(idx_ref, w.E, C)
        assert_equal(f"shard {s} perm", got["perm"].cpu().numpy(), local["perm"])
        assert_equal(f"shard {s} offsets", got["offsets"].cpu().numpy(), local["offsets"])
        slot_ref = whole["slot"][a * w.k:b * w.k]
        assert_equal(f"shard {s} slot", got["slot"].cpu().numpy(), slot_ref)
        kept_ref = np.bincount(idx_ref.ravel()[slot_ref >= 0], minlength=w.E)
        assert_equal(f"shard {s} kept", got["kept"].cpu().numpy(), kept_ref)
        assert int(got["n_dropped"].item()) == int((slot_ref < 0).sum())
        assert got["capacity"] == C


@pytest.mark.parametrize("name", WORKLOADS)
@pytest.mark.parametrize("G", [2, 3, 8])
@pytest.mark.parametrize("cf", [0.5, 1.25])
def test_global_capacity_dispatch(mr, name, G, cf):
    """Dispatch with the capacity of the whole batch across G emulated ranks: the
    ranks' slots, concatenated in rank order, are one dispatch's slots of the
    whole batch, bit for bit; each rank's perm and offsets are its own."""
    T = 20011 if large(name) else synth.ROUTER_WORKLOADS[name].T
    cuts = np.linspace(0, T, G + 1).astype(int)
    cuts[1] -= 7                                          # ranks of unequal size
    _global_dispatch_case(mr, name, cuts, cf)


def test_global_capacity_dispatch_edges(mr):
    """A rank of one row; a second rank that finds most experts' buffers already
    filled by the first (a capacity of 7 per expert); a single rank."""
    name = "zipf-top2-T65536-E64"
    _global_dispatch_case(mr, name, [0, 1, 2, 5000], 1.0)
    _global_dispatch_case(mr, name, [0, 4000, 4100], 0.05)
    _global_dispatch_case(mr, name, [0, 3001], 1.25)


def test_data_parallel_step_single_rank(mr):
    """dp.data_parallel_step end to end in a one-rank gloo group: the exchange
    degenerates to the rank's own statistics, so routing, counts and the
    dispatch with cap_base = 0 must equal the oracle's whole-batch results bit
    for bit, and f, P, the scalars and the gradient match within tolerance."""
    import os
    import socket
    import torch.distributed as dist
    from moe_expert_routing_router_gb300 import dp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=0, world_size=1)
    try:
        w, logits = workload_inputs("zipf-top2-T65536-E64", 30011)
        x = to_device(logits, w.dtype)
        got = dp.data_parallel_step(x, w.k, w.alpha, w.capacity_factor, renorm=int(w.renorm), n_ranks=w.n_ranks)
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    want = oracle_forward(logits, w.dtype, w.k, w.alpha, w.renorm, w.n_ranks)
    C = oracle.dispatch.capacity(w.T, w.k, w.E, w.capacity_factor)
    disp = oracle.dispatch.dispatch(want["idx"], w.E, C)
    assert_equal("idx", got["idx"].cpu().numpy(), want["idx"])
    assert_equal("counts", got["counts"].cpu().numpy(), want["counts"])
    assert_equal("cap_base", got["cap_base"].cpu().numpy(), np.zeros(w.E, np.int64))
    for key in ("perm", "slot", "offsets", "kept"):
        assert_equal(key, got[key].cpu().numpy(), disp[key])
    assert int(got["n_dropped"].item()) == disp["n_dropped"]
    assert got["capacity"] == C
    assert_close("f", got["f"].cpu().numpy(), want["f"], RTOL)
    assert_close("P", got["P"].cpu().numpy(), want["P"], RTOL, FLT_MIN)
    check_backward(got["dlogits"], logits, w.dtype, want["f"].astype(np.float32).astype(np.float64), w.alpha, 1.0)
