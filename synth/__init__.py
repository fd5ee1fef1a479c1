"""Seeded synthetic inputs for the router path, the topology-aware Sinkhorn plan
and the EPLB replication / packing planner.

Both the CPU oracle and the CUDA tests/benchmark take their inputs from here, so
the two sides always see the same bits.  The module only draws random numbers
and encodes them (fp64 -> fp32 -> bf16 round-to-nearest-even); it holds none of
the routing, loss, dispatch, transport or placement arithmetic.
"""

from .workloads import (  # noqa: F401
    RouterWorkload,
    EplbWorkload,
    EPLB_WORKLOADS,
    eplb_loads,
    SinkhornWorkload,
    ROUTER_WORKLOADS,
    SINKHORN_WORKLOADS,
    router_logits,
    sinkhorn_microbatch_logits,
    random_logits,
    f32_to_bf16_bits,
    bf16_bits_to_f32,
)
