"""moe_router_step_static: the step for callers that cannot allocate device scratch.

Such callers (code that must not allocate, plugins with a fixed memory budget,
runtimes that keep all device memory in their own pool) pass only inputs and
outputs; the library's scratch is a fixed array in its image.  This checks,
through the C ABI, that two calls in a row give the same results as the
workspace-taking moe_router_step, and that sizes beyond the array are refused.
It is collected last so that a failure here leaves every other test run.
"""

import numpy as np
import pytest
import torch

import synth
from parity import RTOL, assert_close, to_device

pytestmark = pytest.mark.gpu

FIELDS_EXACT = ("idx", "counts", "rank_load", "perm", "slot", "offsets", "kept", "n_dropped")
FIELDS_FLOAT = ("gate", "f", "P", "scalars", "dlogits")


@pytest.fixture(scope="module")
def mr(native_lib):
    import moe_expert_routing_router_gb300 as m
    return m


@pytest.mark.parametrize("name,T", [("zipf-top2-T65536-E64", 20011), ("zipf-ep64-top6-T262144-E384", 6007),
                                    ("zipf-hot-top8-T131072-E256", 131072)])
def test_static_step_matches_workspace_step_twice(mr, name, T):
    w = synth.ROUTER_WORKLOADS[name]
    w = w if T == w.T else w.with_tokens(T)
    x = to_device(synth.router_logits(w), w.dtype)
    ref = mr.moe_router_step(x, w.k, w.alpha, w.capacity_factor, n_ranks=w.n_ranks, grad_scale=0.75)
    for _ in range(2):
        got = mr.moe_router_step_static(x, w.k, w.alpha, w.capacity_factor, n_ranks=w.n_ranks, grad_scale=0.75)
        torch.cuda.synchronize()
        for key in FIELDS_EXACT:
            assert torch.equal(got[key], ref[key]), key
        for key in FIELDS_FLOAT:
            want = ref[key].double().cpu().numpy()
            assert_close(key, got[key].double().cpu().numpy(), want, RTOL, RTOL * np.abs(want).max())


def test_static_step_refuses_too_many_experts(mr, native_lib):
    x = to_device(synth.random_logits(64, 600, "bf16", seed=2), "bf16")
    with pytest.raises(mr.api._native.MoeRouterError) as err:
        mr.moe_router_step_static(x, 2, 0.01, 1.25)
    assert err.value.status == 1 and b"512" in native_lib.moe_last_error()
