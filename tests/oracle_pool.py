"""The oracle over many independent problems in a process pool (spawned
workers, so that no worker inherits a CUDA context).  Test infrastructure."""

from __future__ import annotations

import multiprocessing as mp
import os
import sys
from concurrent.futures import ProcessPoolExecutor
from pathlib import Path

ROOT = str(Path(__file__).resolve().parents[1])


def _match_one(args):
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    from oracle import taot_match
    loads, plan, R, rpn, K = args
    out = taot_match.match(loads, plan, R, rpn, K)
    return out["slot_expert"], out["slot_tokens"], out["rank_load"]


def match_all(loads, plans, R: int, rpn: int, K: int) -> list:
    """oracle.taot_match.match for every microbatch b of loads[b], plans[b]."""
    jobs = [(loads[b], plans[b], R, rpn, K) for b in range(len(loads))]
    with ProcessPoolExecutor(max_workers=max(1, os.cpu_count() or 1), mp_context=mp.get_context("spawn")) as ex:
        return list(ex.map(_match_one, jobs, chunksize=8))
