"""Writes the per-rank loads of the batched Sinkhorn workload (1024 microbatches, 64 ranks).

Microbatch m is the 384-expert top-6 router workload re-seeded with seed m at
4096 tokens; its loads are the pre-drop token counts of the 64 simulated
expert-parallel ranks (6 contiguous experts each).  Only ``synth`` and the
oracle are called, so the stored loads never come from the CUDA path.

    python tests/golden/make_taot_loads.py
"""

import sys
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parents[2]
sys.path.insert(0, str(ROOT))

import oracle  # noqa: E402
import synth  # noqa: E402

OUT = Path(__file__).resolve().parent / "taot_sinkhorn_B1024_R64_loads.npy"


def microbatch_loads(s: "synth.SinkhornWorkload", m: int) -> np.ndarray:
    src = synth.ROUTER_WORKLOADS[s.source]
    z = oracle.router.widen(synth.sinkhorn_microbatch_logits(s, m), src.dtype)
    counts = oracle.router.expert_counts(oracle.router.top_k(z, src.k), src.E)
    return oracle.router.rank_loads(counts, s.R)


def main() -> None:
    s = synth.SINKHORN_WORKLOADS["taot-sinkhorn-B1024-R64"]
    loads = np.stack([microbatch_loads(s, m) for m in range(s.B)]).astype(np.int32)
    np.save(OUT, loads)
    print(OUT, loads.shape, loads.sum(axis=1)[:4])


if __name__ == "__main__":
    main()
