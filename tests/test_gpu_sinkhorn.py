"""GPU parity of the batched topology-aware Sinkhorn plan (TAOT Phase 1)."""

from pathlib import Path

import numpy as np
import pytest
import torch

import oracle
from parity import SK_RTOL, assert_close, assert_equal

pytestmark = pytest.mark.gpu

LOADS = Path(__file__).resolve().parent / "golden" / "taot_sinkhorn_B1024_R64_loads.npy"


@pytest.fixture(scope="module")
def mr(native_lib):
    import moe_expert_routing_router_gb300 as m
    return m


def _check(got, want, loads):
    assert_equal("status", got["status"].cpu().numpy(), want["status"])
    u, v, plan = (got[x].cpu().numpy().astype(np.float64) for x in ("u", "v", "plan"))
    for m in range(loads.shape[0]):
        assert_close(f"u[{m}]", u[m], want["u"][m], SK_RTOL, SK_RTOL * np.abs(want["u"][m]).max())
        assert_close(f"v[{m}]", v[m], want["v"][m], SK_RTOL, SK_RTOL * np.abs(want["v"][m]).max())
        assert_close(f"plan[{m}]", plan[m], want["plan"][m], SK_RTOL, SK_RTOL * np.abs(want["plan"][m]).max())
        if want["status"][m] == 0:
            over = loads[m] - loads[m].mean()
            a = np.clip(over, 0, None) / np.clip(over, 0, None).sum()
            b = np.clip(-over, 0, None) / np.clip(-over, 0, None).sum()
            assert_close(f"row marginal[{m}]", plan[m].sum(axis=1), a, SK_RTOL, SK_RTOL * a.max())
            assert_close(f"column marginal[{m}]", plan[m].sum(axis=0), b, SK_RTOL, SK_RTOL * b.max())


def test_sinkhorn_parity_on_the_ep64_microbatches(mr):
    loads = np.load(LOADS).astype(np.float64)
    got = mr.taot_sinkhorn_batched(torch.from_numpy(loads.astype(np.float32)).cuda(), 8, 10.0, 0.0, 50)
    torch.cuda.synchronize()
    want = oracle.sinkhorn.taot_phase1(loads, 8, 10.0, None, 50)
    _check(got, want, loads)


@pytest.mark.parametrize("R,rpn,lam,eps,iters", [(2, 1, 10.0, 0.0, 5), (16, 4, 3.0, 1.5, 50),
                                                  (37, 37, 10.0, 0.0, 20), (64, 8, 10.0, 0.0, 0),
                                                  (64, 2, 25.0, 5.0, 200), (1, 1, 10.0, 0.0, 50),
                                                  (48, 6, 10.0, 0.0, 50), (64, 32, 10.0, 0.0, 50),
                                                  (64, 64, 4.0, 0.0, 30)])
def test_sinkhorn_shapes_and_edges(mr, R, rpn, lam, eps, iters):
    rng = np.random.default_rng(R * 31 + iters)
    B = 33
    loads = rng.poisson(200, size=(B, R)).astype(np.float64)
    loads[0] = 100.0                                         # nothing to move
    if R >= 4:
        loads[1, : R // 4] += 500.0                         # one hot quarter
    got = mr.taot_sinkhorn_batched(torch.from_numpy(loads.astype(np.float32)).cuda(), rpn, lam, eps, iters)
    torch.cuda.synchronize()
    want = oracle.sinkhorn.taot_phase1(loads, rpn, lam, eps if eps > 0 else None, iters)
    if iters == 0:
        # no update yet: u = 0 and v = 1 on the planned microbatches, an empty plan
        assert_equal("status", got["status"].cpu().numpy(), want["status"])
        assert not got["plan"].any() and not got["u"].any()
        return
    _check(got, want, loads)


def test_sinkhorn_without_plan_output(mr):
    loads = np.load(LOADS)[:64].astype(np.float32)
    a = mr.taot_sinkhorn_batched(torch.from_numpy(loads).cuda(), 8, 10.0, with_plan=False)
    b = mr.taot_sinkhorn_batched(torch.from_numpy(loads).cuda(), 8, 10.0, with_plan=True)
    torch.cuda.synchronize()
    assert a["plan"] is None and torch.equal(a["u"], b["u"]) and torch.equal(a["v"], b["v"])


def test_sinkhorn_plan_into_a_misaligned_view(mr):
    """A plan pointer that is only 4-byte aligned takes the scalar stores."""
    loads = np.load(LOADS)[:16].astype(np.float32)
    B, R = loads.shape
    x = torch.from_numpy(loads).cuda()
    backing = torch.zeros(B * R * R + 1, dtype=torch.float32, device="cuda")
    view = backing[1:].view(B, R, R)
    assert view.data_ptr() % 16 != 0
    out = {"u": torch.empty_like(x), "v": torch.empty_like(x), "plan": view,
           "status": torch.empty(B, dtype=torch.int32, device="cuda")}
    a = mr.taot_sinkhorn_batched(x, 8, 10.0, out=out)
    b = mr.taot_sinkhorn_batched(x, 8, 10.0)
    torch.cuda.synchronize()
    assert torch.equal(a["plan"], b["plan"]) and backing[0].item() == 0.0
