"""Bounded device waits: an expired grid-barrier wait is reported, not hung on.

A test hook makes every grid barrier wait for one CTA more than the grid has (a
release that nothing performs) and the wait limit is cut to 1 ms.  Every CTA's
wait then runs out; the kernel stops writing and returns, and the host reads
MOE_ERR_TIMEOUT.  Nothing faults or hangs: every wait has a limit, a CTA lets
its own bulk copies land before it exits, and after an expired wait no CTA
writes outside the outputs.  The workspace is then reset and reused.
"""

import pytest
import torch

import synth
from parity import check_forward, oracle_forward, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mr(native_lib):
    import moe_expert_routing_router_gb300 as m
    return m


@pytest.mark.parametrize("E,dtype", [(64, "bf16"), (7, "fp32")])   # staged and direct variants
def test_expired_barrier_wait_is_reported_and_recoverable(mr, native_lib, E, dtype):
    T, k = 65536, 2
    logits = synth.random_logits(T, E, dtype, seed=1)
    x = to_device(logits, dtype)
    ws = mr.Workspace()
    native_lib.moe_set_wait_timeout_ns(1_000_000)
    native_lib.moe_set_unreachable_barriers(1)
    try:
        mr.moe_router_step(x, k, 0.01, 1.25, ws=ws)
        flags = mr.moe_get_device_status(ws)
    finally:
        native_lib.moe_set_unreachable_barriers(0)
        native_lib.moe_set_wait_timeout_ns(0)
    assert flags & 1, f"expected an expired grid-barrier wait, got flags {flags}"
    # the status read reset the workspace: the next calls are correct
    got = mr.moe_router_fwd(x, k, 0.01, ws=ws)
    assert mr.moe_get_device_status(ws) == 0
    check_forward(got, oracle_forward(logits, dtype, k, 0.01, None, 0), 0)
    st = mr.moe_router_step(x, k, 0.01, 1.25, ws=ws)
    assert mr.moe_get_device_status(ws) == 0
    torch.cuda.synchronize()
    assert torch.equal(st["idx"], got["idx"])
