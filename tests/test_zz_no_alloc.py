"""moe_router_step_static: the step for callers that cannot allocate device scratch.

Such callers (code that must not allocate, plugins with a fixed memory budget,
runtimes that keep all device memory in their own pool) pass only inputs and
outputs; the library's scratch is a fixed array in its image.  These tests
check, through the C ABI, that two calls in a row give bit for bit the results
of the workspace-taking moe_router_step without any device memory being
allocated, that sizes beyond the array are refused, and that an expired device
wait is reported through moe_get_device_status(NULL).  The file is collected
last so that a failure here leaves every other test run.
"""

import pytest
import torch

import synth
from parity import to_device

pytestmark = pytest.mark.gpu

FIELDS = ("idx", "gate", "counts", "f", "P", "scalars", "rank_load", "perm", "slot", "offsets", "kept", "n_dropped",
          "dlogits")
AFTER_BARRIER = ("counts", "f", "P", "scalars", "perm", "offsets", "kept", "n_dropped", "dlogits")


@pytest.fixture(scope="module")
def mr(native_lib):
    import moe_expert_routing_router_gb300 as m
    return m


def _outputs(T, E, k, n_ranks):
    i32, f32 = torch.int32, torch.float32
    return {"idx": torch.empty((T, k), dtype=i32, device="cuda"), "gate": torch.empty((T, k), dtype=f32, device="cuda"),
            "counts": torch.empty(E, dtype=i32, device="cuda"), "f": torch.empty(E, dtype=f32, device="cuda"),
            "P": torch.empty(E, dtype=f32, device="cuda"), "scalars": torch.empty(7, dtype=f32, device="cuda"),
            "rank_load": torch.empty(max(n_ranks, 0), dtype=i32, device="cuda"),
            "perm": torch.empty(T * k, dtype=i32, device="cuda"), "slot": torch.empty(T * k, dtype=i32, device="cuda"),
            "offsets": torch.empty(E + 1, dtype=i32, device="cuda"), "kept": torch.empty(E, dtype=i32, device="cuda"),
            "n_dropped": torch.empty(1, dtype=i32, device="cuda"),
            "dlogits": torch.empty((T, E), dtype=f32, device="cuda")}


CASES = [("zipf-top2-T65536-E64", 20011, None), ("zipf-ep64-top6-T262144-E384", 6007, None),
         ("zipf-hot-top8-T131072-E256", 131072, None), ("random-E512-top8", 4099, (512, 8))]


@pytest.mark.parametrize("name,T,shape", CASES)
def test_static_step_matches_workspace_step_twice(mr, name, T, shape):
    if shape is None:
        w = synth.ROUTER_WORKLOADS[name]
        w = w if T == w.T else w.with_tokens(T)
        x = to_device(synth.router_logits(w), w.dtype)
        k, alpha, cf, n_ranks = w.k, w.alpha, w.capacity_factor, w.n_ranks
    else:                                  # E = 512, the largest this entry point serves
        E, k = shape
        x = to_device(synth.random_logits(T, E, "bf16", seed=3), "bf16")
        alpha, cf, n_ranks = 0.01, 1.0, 64
    E = x.shape[1]
    ref = mr.moe_router_step(x, k, alpha, cf, n_ranks=n_ranks, grad_scale=0.75)
    outs = [_outputs(T, E, k, n_ranks) for _ in range(2)]
    # set-up: the first use on a device looks up the array's address (which
    # loads the library's module holding it, if that has not happened yet)
    assert mr.moe_get_device_status(None) == 0
    torch.cuda.synchronize()
    held = torch.cuda.memory_allocated()
    free_before = torch.cuda.mem_get_info()[0]
    for o in outs:                          # two calls in a row on the shared array
        mr.moe_router_step_static(x, k, alpha, cf, n_ranks=n_ranks, grad_scale=0.75, out=o)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == held
    assert torch.cuda.mem_get_info()[0] == free_before
    assert mr.moe_get_device_status(None) == 0
    for o in outs:
        for key in FIELDS:
            assert torch.equal(o[key], ref[key]), key


def test_static_step_refuses_too_many_experts(mr, native_lib):
    x = to_device(synth.random_logits(64, 600, "bf16", seed=2), "bf16")
    with pytest.raises(mr.api._native.MoeRouterError) as err:
        mr.moe_router_step_static(x, 2, 0.01, 1.25)
    assert err.value.status == 1 and b"512" in native_lib.moe_last_error()


def test_static_step_reports_an_expired_wait(mr, native_lib):
    """A grid-barrier wait made to expire (1 ms limit, one CTA more than the
    grid has) is reported by moe_get_device_status(NULL); a call made before
    that read writes none of the outputs that follow the barrier; after the
    read the next call is correct again."""
    w = synth.ROUTER_WORKLOADS["zipf-top2-T65536-E64"]
    x = to_device(synth.router_logits(w), w.dtype)
    E, k = w.E, w.k
    ref = mr.moe_router_step(x, k, w.alpha, w.capacity_factor, grad_scale=1.0)
    torch.cuda.synchronize()
    native_lib.moe_set_wait_timeout_ns(1_000_000)
    native_lib.moe_set_unreachable_barriers(1)
    try:
        mr.moe_router_step_static(x, k, w.alpha, w.capacity_factor, grad_scale=1.0)
        torch.cuda.synchronize()
    finally:
        native_lib.moe_set_unreachable_barriers(0)
        native_lib.moe_set_wait_timeout_ns(0)
    o = _outputs(w.T, E, k, 0)
    for key in AFTER_BARRIER:
        o[key].fill_(-7)
    mr.moe_router_step_static(x, k, w.alpha, w.capacity_factor, grad_scale=1.0, out=o)
    torch.cuda.synchronize()
    for key in AFTER_BARRIER:
        assert bool((o[key] == -7).all()), f"{key} was written while the error bits were set"
    flags = mr.moe_get_device_status(None)
    assert flags & 1, f"expected an expired grid-barrier wait, got flags {flags}"
    assert mr.moe_get_device_status(None) == 0
    got = mr.moe_router_step_static(x, k, w.alpha, w.capacity_factor, grad_scale=1.0)
    torch.cuda.synchronize()
    assert mr.moe_get_device_status(None) == 0
    for key in FIELDS:
        if key != "rank_load":
            assert torch.equal(got[key], ref[key]), key
