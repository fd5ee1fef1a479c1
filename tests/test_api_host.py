"""The binding has no CPU path.  Every entry point refuses host tensors before
it reaches the library (so nothing is computed on the host, and nothing is
handed to a kernel with a host pointer), and a library that is not built is an
error, not a fallback.  Runs without a GPU: no call gets as far as the library."""

import pytest
import torch

import moe_expert_routing_router_gb300 as mr
from moe_expert_routing_router_gb300 import _native, api

T, E, k, B, R = 8, 16, 2, 3, 8
x = torch.zeros(T, E, dtype=torch.bfloat16)
f = torch.full((E,), 1.0 / E)
idx = torch.zeros(T, k, dtype=torch.int32)
dgate = torch.zeros(T, k)
bias = torch.zeros(E)
counts = torch.zeros(2, E, dtype=torch.int32)
P = torch.zeros(2, E)
loads = torch.ones(B, R)
iloads = torch.ones(B, E, dtype=torch.int32)
plan = torch.zeros(B, R, R)

CALLS = {
    "moe_router_fwd": lambda: mr.moe_router_fwd(x, k, 0.01),
    "moe_router_bwd": lambda: mr.moe_router_bwd(x, f, 0.01),
    "moe_router_fwd_ex": lambda: mr.moe_router_fwd_ex(x, k, 0.01, bias=bias, bias_gamma=1e-3, bias_out=True),
    "moe_router_bwd_full": lambda: mr.moe_router_bwd_full(x, f, 0.01, idx=idx, dgate=dgate),
    "moe_dispatch": lambda: mr.moe_dispatch(idx, E, 1.25),
    "moe_shard_capacity_base": lambda: mr.moe_shard_capacity_base(counts, 0),
    "moe_dispatch_sharded": lambda: mr.moe_dispatch_sharded(idx, E, 1.25, 2 * T, torch.zeros(E, dtype=torch.int32)),
    "moe_router_step": lambda: mr.moe_router_step(x, k, 0.01, 1.25),
    "moe_router_step_ex": lambda: mr.moe_router_step_ex(x, k, 0.01, 1.25, bias=bias, dgate=dgate),
    "moe_router_step_static": lambda: mr.moe_router_step_static(x, k, 0.01, 1.25),
    "moe_router_combine": lambda: mr.moe_router_combine(counts, P, [T, T], k, 0.01),
    "taot_sinkhorn_batched": lambda: mr.taot_sinkhorn_batched(loads, 4, 10.0),
    "moe_eplb_plan": lambda: mr.moe_eplb_plan(iloads, 24, 4),
    "taot_match_batched": lambda: mr.taot_match_batched(torch.ones(B, 4 * R, dtype=torch.int32), plan, 4, 2),
}


def _library_reached(*a, **kw):
    raise AssertionError("a call with host tensors reached the library")


@pytest.mark.parametrize("name", sorted(CALLS))
def test_host_tensors_are_refused_before_the_library(name, monkeypatch):
    monkeypatch.setattr(api, "lib", _library_reached)
    with pytest.raises(ValueError, match="CUDA tensor"):
        CALLS[name]()


def test_every_public_entry_point_is_covered():
    """Every device entry point the package exports is in the table above (the
    host-buffer step and the size queries take no device tensors)."""
    host_side = {"Workspace", "moe_dispatch_capacity", "moe_get_device_status", "SCALAR_NAMES",
                 "moe_router_step_host", "moe_router_step_host_device_size", "host_step_outputs"}
    exported = {n for n in api.__all__ if n not in host_side}
    assert exported == set(CALLS), exported ^ set(CALLS)


def test_a_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(_native, "LIB_PATH", tmp_path / "libmoerouter.so")
    monkeypatch.setattr(_native, "_lib", None)
    with pytest.raises(RuntimeError, match="is not built"):
        _native.lib()


class _FakeStream:
    pass


def _recording_stream_ctx(monkeypatch):
    import contextlib
    entered = []

    @contextlib.contextmanager
    def fake(stream):
        entered.append(stream)
        yield

    monkeypatch.setattr(torch.cuda, "stream", fake)
    monkeypatch.setattr(api, "lib", _library_reached)
    return entered


def test_a_given_stream_is_current_while_the_call_allocates(monkeypatch):
    """With a stream given (by keyword or by position), the call runs with it as
    torch's current stream, so that what it allocates belongs to the stream its
    kernels write on; with none given, the current stream is left alone."""
    entered = _recording_stream_ctx(monkeypatch)
    s = _FakeStream()
    with pytest.raises(ValueError):
        mr.moe_router_step(x, k, 0.01, 1.25, stream=s)
    with pytest.raises(ValueError):
        mr.moe_router_bwd(x, f, 0.01, 1.0, None, s)                 # stream by position
    with pytest.raises(ValueError):
        mr.moe_router_fwd(x, k, 0.01)
    assert entered == [s, s]


def test_every_device_entry_point_takes_its_stream():
    """Every device entry point (and the host-buffer step) is wrapped so."""
    for name in sorted(CALLS) + ["moe_router_step_host"]:
        fn = getattr(mr, name)
        assert hasattr(fn, "__wrapped__") and "stream" in fn.__wrapped__.__code__.co_varnames, name
