"""Phase timeline of the persistent router kernel (device timestamps per CTA).

    python -m moe_expert_routing_router_gb300.trace [--mode step|fwd|dispatch] [--cold] WORKLOAD...

Runs the fused step (or the forward, or the dispatch of the forward's picks) on a synthetic workload with the
library's phase tracing on (moe_set_trace_buffer) and prints, for each phase
boundary, the median / min / max over CTAs of the time since the first CTA
started.  Uses only the public ABI.
"""

from __future__ import annotations

import argparse
import sys
from pathlib import Path

import numpy as np
import torch

from . import _native
from .api import Workspace, moe_dispatch, moe_router_fwd, moe_router_step

POINTS = ("entry", "first forward stage landed", "forward rows done (warp 0)", "per-CTA partials published",
          "grid barrier passed", "totals, bases, offsets in smem", "(unused)", "first backward stage",
          "backward rows done (warp 0)", "dispatch + E-sized outputs done", "all warps joined", "exit",
          "in-CTA dispatch ranks done", "SM id", "forward rows done (all warps)", "backward rows done (all warps)")
SM_ID = 13
TRACE_POINTS = 16
MAX_CTAS = 2048


def _device_logits(w, seed: int = 0) -> torch.Tensor:
    sys.path.insert(0, str(Path(__file__).resolve().parents[1]))
    import synth
    z = synth.router_logits(w, seed)
    if w.dtype == "bf16":
        return torch.from_numpy(z.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(z).cuda()


def phase_timeline(w, mode: str = "step", reps: int = 3, cold: bool = False) -> tuple[int, np.ndarray]:
    """Returns (CTAs, times [CTAs, points] in microseconds since the first CTA's entry; NaN = not passed).

    cold: before each traced launch, write a buffer of three times the L2 size so
    that the launch finds its inputs in HBM, as in the benchmark's rotation."""
    x = _device_logits(w)
    ws = Workspace()
    if mode == "step":
        def run():
            moe_router_step(x, w.k, w.alpha, w.capacity_factor, renorm=int(w.renorm), n_ranks=w.n_ranks, ws=ws)
    elif mode == "fwd":
        def run():
            moe_router_fwd(x, w.k, w.alpha, renorm=int(w.renorm), n_ranks=w.n_ranks, ws=ws)
    else:                                          # dispatch of the forward's picks
        idx = moe_router_fwd(x, w.k, w.alpha, renorm=int(w.renorm), n_ranks=w.n_ranks, ws=ws)["idx"]

        def run():
            moe_dispatch(idx, w.E, w.capacity_factor, ws=ws)
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


def main() -> int:
    sys.path.insert(0, str(Path(__file__).resolve().parents[1]))
    import synth
    ap = argparse.ArgumentParser()
    ap.add_argument("--mode", choices=("step", "fwd", "dispatch"), default="step")
    ap.add_argument("--cold", action="store_true", help="flush L2 before each traced launch")
    ap.add_argument("workloads", nargs="*", default=list(synth.ROUTER_WORKLOADS))
    args = ap.parse_args()
    for name in args.workloads:
        w = synth.ROUTER_WORKLOADS[name]
        G, rel = phase_timeline(w, args.mode, cold=args.cold)
        print(f"{args.mode} {name}: {G} CTAs, last exit {np.nanmax(rel[:, 11]):.2f} us")
        for i in range(1, len(POINTS)):
            if i == SM_ID:
                continue
            col = rel[:, i]
            if np.all(np.isnan(col)):
                continue
            print(f"   {POINTS[i]:>34}: median {np.nanmedian(col):8.2f}  min {np.nanmin(col):8.2f}  "
                  f"max {np.nanmax(col):8.2f} us")
    return 0


if __name__ == "__main__":
    sys.exit(main())
