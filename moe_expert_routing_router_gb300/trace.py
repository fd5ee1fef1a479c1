"""Phase timeline of the persistent router kernel (device timestamps per CTA).

``phase_timeline`` runs the fused step (or the extended step with a seeded
bias and upstream gradient of the gates, or the forward, or the dispatch of
the forward's picks) on logits the caller supplies, with the library's phase
tracing on (moe_set_trace_buffer), and returns for each CTA the time of each
phase boundary since the first CTA started.  ``summary`` turns that into the
median / min / max over CTAs per boundary.  Uses only the public ABI.
"""

from __future__ import annotations

import numpy as np
import torch

from . import _native
from .api import Workspace, moe_dispatch, moe_router_fwd, moe_router_step, moe_router_step_ex

POINTS = ("entry", "first forward stage landed", "forward rows done (warp 0)", "per-CTA partials published",
          "grid barrier passed", "totals, bases, offsets in smem", "(unused)", "first backward stage",
          "backward rows done (warp 0)", "dispatch + E-sized outputs done", "all warps joined", "exit",
          "in-CTA dispatch ranks done", "SM id", "forward rows done (all warps)", "backward rows done (all warps)")
SM_ID = 13
TRACE_POINTS = 16
MAX_CTAS = 2048


def phase_timeline(x: torch.Tensor, k: int, alpha: float, capacity_factor: float, renorm: int = -1,
                   n_ranks: int = 0, mode: str = "step", reps: int = 3,
                   cold: bool = False) -> tuple[int, np.ndarray]:
    """Returns (CTAs, times [CTAs, points] in microseconds since the first CTA's entry; NaN = not passed).

    x: router logits [T, E] (bf16 or fp32) on the current CUDA device.
    cold: before each traced launch, write a buffer of three times the L2 size so
    that the launch finds its inputs in HBM, as in the benchmark's rotation."""
    E = x.shape[1]
    ws = Workspace()
    if mode == "step":
        def run():
            moe_router_step(x, k, alpha, capacity_factor, renorm=renorm, n_ranks=n_ranks, ws=ws)
    elif mode == "step_ex":
        T = x.shape[0]
        gen = torch.Generator(device=x.device).manual_seed(7)
        bias = torch.randn(E, generator=gen, device=x.device) * 0.5
        dgate = torch.randn(T, k, generator=gen, device=x.device)

        def run():
            moe_router_step_ex(x, k, alpha, capacity_factor, renorm=renorm, n_ranks=n_ranks, bias=bias,
                               dgate=dgate, ws=ws)
    elif mode == "fwd":
        def run():
            moe_router_fwd(x, k, alpha, renorm=renorm, n_ranks=n_ranks, ws=ws)
    else:                                          # dispatch of the forward's picks
        idx = moe_router_fwd(x, k, alpha, renorm=renorm, n_ranks=n_ranks, ws=ws)["idx"]

        def run():
            moe_dispatch(idx, E, capacity_factor, ws=ws)
    for _ in range(3):
        run()
    torch.cuda.synchronize()
    buf = torch.zeros(MAX_CTAS * TRACE_POINTS, dtype=torch.int64, device="cuda")
    flush = torch.empty(3 * 129 * 2**20, dtype=torch.uint8, device="cuda") if cold else None
    lib = _native.lib()
    lib.moe_set_trace_buffer(buf.data_ptr(), MAX_CTAS)
    try:
        for _ in range(reps):
            buf.zero_()
            if flush is not None:
                flush.fill_(1)
            run()
            torch.cuda.synchronize()
    finally:
        lib.moe_set_trace_buffer(None, 0)
    t = buf.view(-1, TRACE_POINTS).cpu().numpy().astype(np.int64)[:, :len(POINTS)]
    t = t[t[:, 0] > 0]
    rel = np.where(t > 0, (t - t[:, 0].min()) / 1000.0, np.nan)
    rel[:, SM_ID] = t[:, SM_ID]
    return t.shape[0], rel


def summary(rel: np.ndarray) -> dict:
    """Per phase boundary (by name): median, min and max over CTAs in microseconds."""
    out = {}
    for i in range(1, len(POINTS)):
        col = rel[:, i]
        if i == SM_ID or np.all(np.isnan(col)):
            continue
        out[POINTS[i]] = {"median": float(np.nanmedian(col)), "min": float(np.nanmin(col)),
                          "max": float(np.nanmax(col))}
    return out
