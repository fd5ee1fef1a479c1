"""moe_router_step_host: the step on host logits, every output copied back.

Through the C ABI, the host arrays must hold bit for bit what the device step
writes for the same logits, on two router workloads at a size that spans many
CTAs, and on consecutive calls that reuse one staging buffer.
"""

import pytest
import torch

import synth
from parity import to_device

pytestmark = pytest.mark.gpu

FIELDS = ("idx", "gate", "counts", "f", "P", "scalars", "rank_load", "perm", "slot", "offsets", "kept", "n_dropped",
          "dlogits")


@pytest.fixture(scope="module")
def mr(native_lib):
    import moe_expert_routing_router_gb300 as m
    return m


@pytest.mark.parametrize("name,T", [("zipf-top2-T65536-E64", 30011), ("zipf-ep64-top6-T262144-E384", 20011),
                                    ("switch-top1-T4096-E8", 4096)])
def test_host_step_equals_device_step(mr, name, T):
    w = synth.ROUTER_WORKLOADS[name]
    w = w if T == w.T else w.with_tokens(T)
    logits = synth.router_logits(w)
    x_dev = to_device(logits, w.dtype)
    x_host = x_dev.cpu().pin_memory()
    ref = mr.moe_router_step(x_dev, w.k, w.alpha, w.capacity_factor, renorm=int(w.renorm), n_ranks=w.n_ranks,
                             grad_scale=0.5)
    dev = torch.empty(mr.moe_router_step_host_device_size(x_host.dtype, w.T, w.E, w.k, w.n_ranks),
                      dtype=torch.uint8, device="cuda")
    for _ in range(2):
        out = mr.host_step_outputs(w.T, w.E, w.k, w.n_ranks)
        mr.moe_router_step_host(x_host, w.k, w.alpha, w.capacity_factor, renorm=int(w.renorm), n_ranks=w.n_ranks,
                                grad_scale=0.5, dev=dev, out=out)
        torch.cuda.synchronize()
        for key in FIELDS:
            assert torch.equal(out[key], ref[key].cpu()), key
