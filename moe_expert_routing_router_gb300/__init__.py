"""GB300-native (sm_103a) MoE expert routing with equal-cost load balancing.

The library is a C ABI (include/moe_router.h) over hand-written CUDA kernels;
this package builds it in-tree and binds it with ctypes.  The native library
is loaded lazily on the first call and there is no non-CUDA fallback.
"""

from .api import (  # noqa: F401
    SCALAR_NAMES,
    Workspace,
    moe_dispatch,
    moe_dispatch_capacity,
    moe_dispatch_sharded,
    moe_eplb_plan,
    moe_get_device_status,
    moe_router_bwd,
    moe_router_combine,
    moe_router_fwd,
    moe_router_fwd_ex,
    moe_router_bwd_full,
    moe_router_step,
    moe_router_step_ex,
    moe_router_step_host,
    moe_router_step_host_device_size,
    moe_router_step_static,
    moe_shard_capacity_base,
    host_step_outputs,
    taot_match_batched,
    taot_sinkhorn_batched,
)

__all__ = [
    "SCALAR_NAMES", "Workspace", "moe_dispatch", "moe_dispatch_capacity", "moe_dispatch_sharded", "moe_eplb_plan", "moe_get_device_status",
    "moe_router_bwd", "moe_router_bwd_full", "moe_router_combine", "moe_router_fwd", "moe_router_fwd_ex", "moe_router_step", "moe_router_step_ex", "moe_router_step_host", "moe_router_step_host_device_size", "host_step_outputs", "moe_router_step_static", "moe_shard_capacity_base", "taot_match_batched", "taot_sinkhorn_batched",
]
