"""Benchmark of the MoE router hot path on GB300: one step = router forward +
dispatch + backward over one batch (one launch of moe_router_step).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-extra] [--parallelism auto|dp|replicas]
                    [--section step|next_steps|step_ex|eplb|taot_match [--tokens T]]

Prints one JSON line on rank 0.  With --gpus N > 1 (under torchrun) the ranks
hold one batch of N * T rows, T per rank (weak scaling), and run the
data-parallel step: each routes its rows, the ranks all-gather their counts
and P, combine them, dispatch with the whole batch's capacity and run the
backward of the batch's loss (--parallelism replicas instead runs the fused
single-launch step on every rank independently).  The timed region is
bracketed by a barrier and the slowest rank's time is reported.  Unless
--no-extra, the line also carries the other router workloads (`also`), the
separate calls, the Sinkhorn plan, the bias-routing forward / full backward /
bias-routed step (`next_steps`), the EPLB planner (`eplb`) and TAOT Phase 2
(`taot_match`); --section prints one of those parts alone.

`--impl reference` times the CPU oracle (fp64 numpy, the only other use of
``oracle/`` outside the tests) on a bounded sample of the same workload.
"""

from __future__ import annotations

import os

for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import json  # noqa: E402
import math  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import threading  # noqa: E402
import time  # noqa: E402
from pathlib import Path  # noqa: E402

import numpy as np  # noqa: E402

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import synth  # noqa: E402

METRIC = "router fwd+bwd+dispatch tokens/s; achieved HBM GB/s vs GB300 peak"
DEFAULT_WORKLOAD = "zipf-ep64-top6-T262144-E384"
EXTRA_WORKLOADS = ("zipf-top2-T65536-E64", "zipf-hot-top8-T131072-E256")
DETAIL_WORKLOADS = ("zipf-top2-T65536-E64", "zipf-ep64-top6-T262144-E384")   # separate calls, next steps
SINKHORN_WORKLOAD = "taot-sinkhorn-B1024-R64"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ----------------------------------------------------------------------------- sizes

def algorithmic_bytes(w: synth.RouterWorkload) -> int:
    """Bytes the step must move: logits read once, dlogits written in fp32, and
    idx, gate, perm, slot (4 bytes each) per assignment."""
    esize = 2 if w.dtype == "bf16" else 4
    return w.T * (w.E * (esize + 4) + 16 * w.k)


STEP_KERNEL_SOURCES = ("router_kernels.cuh", "device_common.cuh", "router_instances.cuh", "router_table.h",
                       "router_bf16_staged.cu", "router_bf16_direct.cu", "router_fp32_staged.cu",
                       "router_fp32_direct.cu", "router_dispatch.cu")


def kernel_source_hash() -> str:
    """Hash of the sources of the router step kernel and its launch: the files
    that build router_persistent_kernel, and the part of abi.cu that lays out
    the workspace, picks the variant, sizes and launches the grid, plus the
    moe_router_step entry point.  It changes whenever that kernel or its launch
    does, and not when other entry points of the library do."""
    import hashlib
    h = hashlib.sha256()
    csrc = ROOT / "moe_expert_routing_router_gb300" / "csrc"
    for name in STEP_KERNEL_SOURCES:
        h.update(name.encode())
        h.update((csrc / name).read_bytes())
    abi = (csrc / "abi.cu").read_text()
    a = abi.index("moe_status moe_router_step(")
    part = abi[:abi.index("moe_status check_fwd_outputs(")] + abi[a:abi.index("\n}\n", a) + 3]
    h.update(b"abi.cu")
    h.update(part.encode())
    return h.hexdigest()[:16]


def measured_traffic(workload: str) -> dict | None:
    """DRAM bytes per launch of the step kernel from the committed ncu summary,
    only while the kernel sources are the ones that summary was taken with."""
    p = ROOT / "profiles" / "router_step_dram_traffic.txt"
    if not p.exists():
        return None
    cur = kernel_source_hash()
    for ln in p.read_text().splitlines():
        f = ln.split()
        if len(f) >= 8 and f[0] == "workload" and f[1] == workload and f[6] == "source_hash" and f[7] == cur:
            return {"read": int(f[3]), "write": int(f[5])}
    return None


def peaks() -> dict:
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured (MEASURED_PEAKS.json hbm_gbs)"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "source": "fallback 6.8 TB/s"}


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling in the background."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- GPU arm

def to_device(logits: np.ndarray, dtype: str, torch, device):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(logits).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).to(device)


def out_buffers(w, torch, device) -> dict:
    T, E, k = w.T, w.E, w.k
    i32, f32 = torch.int32, torch.float32
    return {
        "idx": torch.empty((T, k), dtype=i32, device=device), "gate": torch.empty((T, k), dtype=f32, device=device),
        "counts": torch.empty(E, dtype=i32, device=device), "f": torch.empty(E, dtype=f32, device=device),
        "P": torch.empty(E, dtype=f32, device=device), "scalars": torch.empty(7, dtype=f32, device=device),
        "rank_load": torch.empty(max(w.n_ranks, 0), dtype=i32, device=device),
        "perm": torch.empty(T * k, dtype=i32, device=device), "slot": torch.empty(T * k, dtype=i32, device=device),
        "offsets": torch.empty(E + 1, dtype=i32, device=device), "kept": torch.empty(E, dtype=i32, device=device),
        "n_dropped": torch.empty(1, dtype=i32, device=device),
        "dlogits": torch.empty((T, E), dtype=f32, device=device),
    }


def replay_plan(steps: int, n_min: int) -> tuple[int, int, int]:
    """(steps per graph S, replays R, buffer sets) for K = steps timed steps:
    R * S = K with R >= 10 where K allows, and the buffer sets (at least
    n_min) dividing S, so that every replay rotates through them the same way.
    When no divisor of S reaches n_min, one graph of all K steps is replayed
    once."""
    S = 1
    for d in range(max(1, steps // 10), 0, -1):
        if steps % d == 0:
            S = d
            break
    for n in range(n_min, S + 1):
        if S % n == 0:
            return S, steps // S, n
    return steps, 1, n_min


def percentile(xs: list[float], q: float) -> float:
    ys = sorted(xs)
    if len(ys) == 1:
        return ys[0]
    pos = q * (len(ys) - 1)
    lo = int(math.floor(pos))
    hi = min(lo + 1, len(ys) - 1)
    return ys[lo] + (ys[hi] - ys[lo]) * (pos - lo)


def time_router(w, steps: int, warmup: int, torch, device, dist_ctx, soak_s: float = 0.0, sampler=None) -> dict:
    """Device-timed steps of moe_router_step: K steps as R replays of one CUDA
    graph of S steps (R >= 10 where K allows), each replay between two CUDA
    events on the launching stream; buffers rotated so that a set is reused
    only after at least 3x the L2 of other traffic."""
    import moe_expert_routing_router_gb300 as mr
    logits = synth.router_logits(w)
    step_bytes = algorithmic_bytes(w)
    S, R, n_sets = replay_plan(steps, max(2, math.ceil(3 * L2_BYTES / step_bytes)))
    x0 = to_device(logits, w.dtype, torch, device)
    xs = [x0] + [x0.clone() for _ in range(n_sets - 1)]
    outs = [out_buffers(w, torch, device) for _ in range(n_sets)]
    ws = mr.Workspace(device)
    stream = torch.cuda.current_stream(device)

    def step(i):
        mr.moe_router_step(xs[i % n_sets], w.k, w.alpha, w.capacity_factor, renorm=int(w.renorm),
                           n_ranks=w.n_ranks, grad_scale=1.0, ws=ws, out=outs[i % n_sets])

    for i in range(max(warmup, 3)):
        step(i)
    torch.cuda.synchronize(device)
    # S steps captured once into a CUDA graph, so that the device time is
    # measured, not the Python-side launch rate.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(S):
            step(i)
    graph.replay()
    torch.cuda.synchronize(device)
    if sampler is not None:
        sampler.start()
    t_end = time.time() + soak_s
    while time.time() < t_end:                      # loaded window for the clock samples
        graph.replay()
        torch.cuda.synchronize(device)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(R + 1)]
    dist_ctx.barrier()
    torch.cuda.synchronize(device)
    ev[0].record(stream)
    for r in range(R):
        graph.replay()
        ev[r + 1].record(stream)
    torch.cuda.synchronize(device)
    dist_ctx.barrier()
    clocks = sampler.stop() if sampler is not None else None
    total_ms = ev[0].elapsed_time(ev[R])
    per_step = [ev[r].elapsed_time(ev[r + 1]) / S for r in range(R)]
    flags = mr.moe_get_device_status(ws)
    if flags:
        raise RuntimeError(f"device wait expired during the benchmark (flags {flags})")
    # one kernel per step: the mean step time is its mean launch duration
    return {"total_ms": dist_ctx.max(total_ms), "launch_ms_mean": total_ms / steps, "n_sets": n_sets,
            "clocks": clocks, "step_bytes": step_bytes,
            "spread": {"replays": R, "steps_per_replay": S, "ms_per_step_median": statistics.median(per_step),
                       "ms_per_step_p10": percentile(per_step, 0.1), "ms_per_step_p90": percentile(per_step, 0.9)},
            "timing": f"{R} replays of a CUDA graph of {S} steps, each between two CUDA events on the launching stream"}


def time_e2e(w, steps: int, warmup: int, torch, device, dist_ctx) -> dict:
    """The step through the C ABI on HOST buffers (moe_router_step_host):
    every step copies its logits from pinned host memory into device staging,
    runs the step, and copies every output back to pinned host memory (idx,
    gate, counts, f, P, scalars, rank loads, perm, slot, offsets, kept,
    n_dropped, dlogits).  Consecutive steps alternate between two streams,
    each with its own staging buffer, workspace and host outputs, so that one
    step's copies overlap the other's kernel; the kernels run one after the
    other (each waits for the previous step's kernel_done event)."""
    import moe_expert_routing_router_gb300 as mr
    logits = synth.router_logits(w)
    host_x = to_device(logits, w.dtype, torch, "cpu").pin_memory()
    streams = [torch.cuda.Stream(device) for _ in range(2)]
    wss = [mr.Workspace(device) for _ in range(2)]
    dev_bytes = mr.moe_router_step_host_device_size(host_x.dtype, w.T, w.E, w.k, w.n_ranks)
    devs = [torch.empty(dev_bytes, dtype=torch.uint8, device=device) for _ in range(2)]
    outs = [mr.host_step_outputs(w.T, w.E, w.k, w.n_ranks) for _ in range(2)]
    h2d = host_x.numel() * host_x.element_size()
    d2h = sum(t.numel() * t.element_size() for t in outs[0].values())

    compute = torch.cuda.current_stream(device)
    done = [torch.cuda.Event() for _ in range(2)]
    for e in done:                                   # creates the events' CUDA handles
        e.record(compute)

    def run(n):
        for i in range(n):
            b = i & 1
            mr.moe_router_step_host(host_x, w.k, w.alpha, w.capacity_factor, renorm=int(w.renorm),
                                    n_ranks=w.n_ranks, grad_scale=1.0, ws=wss[b], dev=devs[b], out=outs[b],
                                    stream=streams[b], device=device, kernel_after=done[b ^ 1],
                                    kernel_done=done[b])

    run(max(warmup, 3))
    torch.cuda.synchronize(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    dist_ctx.barrier()
    t0.record(compute)
    for s in streams:
        s.wait_event(t0)
    run(steps)
    for s in streams:
        compute.wait_stream(s)
    t1.record(compute)
    torch.cuda.synchronize(device)
    dist_ctx.barrier()
    ms = dist_ctx.max(t0.elapsed_time(t1)) / steps
    for b in range(2):
        if mr.moe_get_device_status(wss[b]):
            raise RuntimeError("device wait expired during the end-to-end benchmark")
    return {"ms_per_step": ms, "h2d": h2d, "d2h": d2h, "steps": steps}


def time_dp(w, steps: int, warmup: int, torch, device, dist_ctx, e2e: bool = False, sampler=None) -> dict:
    """Device-timed data-parallel steps (dp.data_parallel_step): each rank routes
    its own w.T rows of a batch of world * w.T rows (its logits a row rotation
    of the workload's by the rank), exchanges counts and P in one all-gather,
    combines them, dispatches with the whole batch's capacity and runs the
    backward of the batch's loss.  Five library launches and one collective per
    step, issued eagerly; the logits (201 MB at E = 384) exceed the L2.  With
    e2e, every step also copies its logits from pinned host memory and every
    output of the rank (idx, gate, perm, slot, offsets, kept, n_dropped,
    dlogits and the batch's counts, f, P, scalars, rank loads) back to pinned
    host memory."""
    import moe_expert_routing_router_gb300 as mr
    from moe_expert_routing_router_gb300 import dp
    logits = np.roll(synth.router_logits(w), dist_ctx.rank * 97, axis=0)
    x = to_device(logits, w.dtype, torch, device)
    host_x = to_device(logits, w.dtype, torch, "cpu").pin_memory() if e2e else None
    ws = mr.Workspace(device)
    T_shard = [w.T] * dist_ctx.world
    keys = ("idx", "gate", "perm", "slot", "offsets", "kept", "n_dropped", "dlogits", "counts", "f", "P",
            "scalars", "rank_load")
    host_out: dict = {}
    stream = torch.cuda.current_stream(device)

    def step():
        if e2e:
            x.copy_(host_x, non_blocking=True)
        o = dp.data_parallel_step(x, w.k, w.alpha, w.capacity_factor, renorm=int(w.renorm), n_ranks=w.n_ranks,
                                  ws=ws, T_shard=T_shard)
        if e2e:
            for k in keys:
                if k not in host_out:
                    host_out[k] = torch.empty(o[k].shape, dtype=o[k].dtype, pin_memory=True)
                host_out[k].copy_(o[k], non_blocking=True)
        return o

    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize(device)
    if sampler is not None:
        sampler.start()
    dist_ctx.barrier()
    torch.cuda.synchronize(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize(device)
    dist_ctx.barrier()
    clocks = sampler.stop() if sampler is not None else None
    ms = dist_ctx.max(t0.elapsed_time(t1)) / steps
    if mr.moe_get_device_status(ws):
        raise RuntimeError("device wait expired during the data-parallel benchmark")
    h2d = host_x.numel() * host_x.element_size() if e2e else 0
    d2h = sum(t.numel() * t.element_size() for t in host_out.values()) if e2e else 0
    return {"ms_per_step": ms, "h2d": h2d, "d2h": d2h, "steps": steps, "clocks": clocks}


def time_calls(w, torch, device, hbm_gbs: float, reps: int = 20) -> dict:
    """The forward, backward and dispatch as separate C-ABI calls (moe_router_fwd,
    moe_router_bwd, moe_dispatch), each a CUDA graph of `reps` calls over buffer
    sets rotated at least 3x L2 apart, with its algorithmic bytes per call."""
    import moe_expert_routing_router_gb300 as mr
    esize = 2 if w.dtype == "bf16" else 4
    T, E, k = w.T, w.E, w.k
    nbytes = {"moe_router_fwd": T * E * esize + T * k * 8,          # logits in; idx, gate out
              "moe_router_bwd": T * E * (esize + 4),                # logits in; dlogits out
              "moe_dispatch": T * k * 12}                           # idx in; perm, slot out
    x0 = to_device(synth.router_logits(w), w.dtype, torch, device)
    ws = mr.Workspace(device)
    ref = mr.moe_router_fwd(x0, w.k, w.alpha, renorm=int(w.renorm), n_ranks=w.n_ranks, ws=ws)
    out = {}
    for name, b in nbytes.items():
        n_sets = max(2, math.ceil(3 * L2_BYTES / b))
        xs = [x0] + [x0.clone() for _ in range(n_sets - 1)] if name != "moe_dispatch" else None
        idxs = [ref["idx"].clone() for _ in range(n_sets)] if name == "moe_dispatch" else None
        bufs = [out_buffers(w, torch, device) for _ in range(n_sets)]
        fo = lambda i: {kk: bufs[i][kk] for kk in ("idx", "gate", "counts", "f", "P", "scalars", "rank_load")}
        def call(i):
            j = i % n_sets
            if name == "moe_router_fwd":
                mr.moe_router_fwd(xs[j], w.k, w.alpha, renorm=int(w.renorm), n_ranks=w.n_ranks, ws=ws, out=fo(j))
            elif name == "moe_router_bwd":
                mr.moe_router_bwd(xs[j], ref["f"], w.alpha, 1.0, dlogits=bufs[j]["dlogits"])
            else:
                mr.moe_dispatch(idxs[j], w.E, w.capacity_factor, ws=ws,
                                out={kk: bufs[j][kk] for kk in ("perm", "slot", "offsets", "kept", "n_dropped")})
        for i in range(3):
            call(i)
        torch.cuda.synchronize(device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(reps):
                call(i)
        stream = torch.cuda.current_stream(device)
        g.replay()
        torch.cuda.synchronize(device)
        a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b2.record(stream)
        torch.cuda.synchronize(device)
        us = a.elapsed_time(b2) / reps * 1e3
        gbs = b / (us * 1e-6) / 1e9
        out[name] = {"us_per_call": round(us, 2), "algorithmic_bytes": b, "achieved_gbs": round(gbs, 1),
                     "frac_of_hbm_peak": round(gbs / hbm_gbs, 4)}
        del xs, idxs, bufs, g
    return out


def _graph_us(torch, device, call, reps: int) -> float:
    """Mean time of `call(i)` for i in 0..reps-1, as one CUDA graph replayed
    between two CUDA events (after three eager warm-up calls and one replay)."""
    for i in range(3):
        call(i)
    torch.cuda.synchronize(device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(reps):
            call(i)
    stream = torch.cuda.current_stream(device)
    g.replay()
    torch.cuda.synchronize(device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    g.replay()
    b.record(stream)
    torch.cuda.synchronize(device)
    return a.elapsed_time(b) / reps * 1e3


def time_next_steps(w, torch, device, hbm_gbs: float, reps: int = 20) -> dict:
    """The method's next steps through the C ABI: the forward with bias routing
    and the in-place bias update, the forward with masked P, the full backward
    through the gates, and a bias-routed training step, as three calls (fwd_ex
    + dispatch + bwd_full) and as one launch (moe_router_step_ex).  Each is a CUDA graph of `reps` calls over buffer sets rotated
    at least 3x L2 apart, with its algorithmic bytes per call."""
    import moe_expert_routing_router_gb300 as mr
    esize = 2 if w.dtype == "bf16" else 4
    T, E, k = w.T, w.E, w.k
    fwd_b = T * E * esize + T * k * 8                     # logits in; idx, gate out
    bwd_b = T * E * (esize + 4) + T * k * 8               # logits, idx, dgate in; dlogits out
    step_b = T * E * (esize + 4) + T * k * 20             # + perm, slot out
    x0 = to_device(synth.router_logits(w), w.dtype, torch, device)
    ws = mr.Workspace(device)
    rng = np.random.default_rng(1)
    bias = torch.from_numpy((rng.standard_normal(E) * 0.5).astype(np.float32)).to(device)
    ref = mr.moe_router_fwd_ex(x0, k, w.alpha, renorm=int(w.renorm), n_ranks=w.n_ranks, bias=bias, ws=ws)
    n_sets = max(2, math.ceil(3 * L2_BYTES / fwd_b))
    xs = [x0] + [x0.clone() for _ in range(n_sets - 1)]
    bufs = [out_buffers(w, torch, device) for _ in range(n_sets)]
    idxs = [ref["idx"].clone() for _ in range(n_sets)]
    dgates = [torch.randn(T, k, device=device) for _ in range(n_sets)]
    fo = lambda j: {kk: bufs[j][kk] for kk in ("idx", "gate", "counts", "f", "P", "scalars", "rank_load")}
    do = lambda j: {kk: bufs[j][kk] for kk in ("perm", "slot", "offsets", "kept", "n_dropped")}

    def fwd_bias(i):
        j = i % n_sets
        mr.moe_router_fwd_ex(xs[j], k, w.alpha, renorm=int(w.renorm), n_ranks=w.n_ranks, bias=bias,
                             bias_gamma=1e-3, bias_out=bias, ws=ws, out=fo(j))

    def fwd_masked(i):
        j = i % n_sets
        mr.moe_router_fwd_ex(xs[j], k, w.alpha, renorm=int(w.renorm), n_ranks=w.n_ranks, masked_p=True,
                             ws=ws, out=fo(j))

    def bwd_full(i):
        j = i % n_sets
        mr.moe_router_bwd_full(xs[j], ref["f"], w.alpha, 1.0, idx=idxs[j], dgate=dgates[j],
                               renorm=int(w.renorm), dlogits=bufs[j]["dlogits"])

    def step(i):
        j = i % n_sets
        o = fo(j)
        mr.moe_router_fwd_ex(xs[j], k, w.alpha, renorm=int(w.renorm), n_ranks=w.n_ranks, bias=bias,
                             bias_gamma=1e-3, bias_out=bias, ws=ws, out=o)
        mr.moe_dispatch(o["idx"], E, w.capacity_factor, ws=ws, out=do(j))
        mr.moe_router_bwd_full(xs[j], o["f"], w.alpha, 1.0, idx=o["idx"], dgate=dgates[j],
                               renorm=int(w.renorm), dlogits=bufs[j]["dlogits"])

    def step_one(i):
        j = i % n_sets
        mr.moe_router_step_ex(xs[j], k, w.alpha, w.capacity_factor, renorm=int(w.renorm), n_ranks=w.n_ranks,
                              bias=bias, bias_gamma=1e-3, bias_out=bias, dgate=dgates[j], ws=ws,
                              out={**fo(j), **do(j), "dlogits": bufs[j]["dlogits"]})

    out = {"workload": w.name}
    for name, fn, b in (("moe_router_fwd_ex (bias routing + update)", fwd_bias, fwd_b),
                        ("moe_router_fwd_ex (masked P)", fwd_masked, fwd_b),
                        ("moe_router_bwd_full (gates + aux)", bwd_full, bwd_b),
                        ("bias-routed step (fwd_ex + dispatch + bwd_full)", step, step_b),
                        ("bias-routed step in one launch (moe_router_step_ex)", step_one, step_b)):
        us = _graph_us(torch, device, fn, reps)
        gbs = b / (us * 1e-6) / 1e9
        out[name] = {"us_per_call": round(us, 2), "tokens_per_s": round(T / (us * 1e-6), 1),
                     "algorithmic_bytes": b, "achieved_gbs": round(gbs, 1), "frac_of_hbm_peak": round(gbs / hbm_gbs, 4)}
    del xs, bufs, idxs, dgates
    return out


def time_step(w, torch, device, hbm_gbs: float, reps: int = 20) -> dict:
    """The fused step alone (moe_router_step: forward, dispatch and the aux-loss
    backward in one launch), as a CUDA graph of `reps` calls over buffer sets
    rotated at least 3x L2 apart; the first three calls run eagerly.  With
    --tokens this is a smaller case of the same kernel instantiation."""
    import moe_expert_routing_router_gb300 as mr
    step_b = algorithmic_bytes(w)
    x0 = to_device(synth.router_logits(w), w.dtype, torch, device)
    n_sets = max(2, math.ceil(3 * L2_BYTES / step_b))
    xs = [x0] + [x0.clone() for _ in range(n_sets - 1)]
    bufs = [out_buffers(w, torch, device) for _ in range(n_sets)]
    ws = mr.Workspace(device)

    def call(i):
        j = i % n_sets
        mr.moe_router_step(xs[j], w.k, w.alpha, w.capacity_factor, renorm=int(w.renorm), n_ranks=w.n_ranks,
                           grad_scale=1.0, ws=ws, out=bufs[j])

    us = _graph_us(torch, device, call, reps)
    flags = mr.moe_get_device_status(ws)
    if flags:
        raise RuntimeError(f"device wait expired during the benchmark (flags {flags})")
    gbs = step_b / (us * 1e-6) / 1e9
    return {"workload": w.name, "T": w.T, "n_sets": n_sets, "us_per_call": round(us, 2),
            "tokens_per_s": round(w.T / (us * 1e-6), 1), "algorithmic_bytes": step_b,
            "achieved_gbs": round(gbs, 1), "frac_of_hbm_peak": round(gbs / hbm_gbs, 4)}


def time_step_ex(w, torch, device, hbm_gbs: float, reps: int = 20) -> dict:
    """The bias-routed step in one launch alone (moe_router_step_ex: bias routing
    with the bias updated in place, dispatch, and the backward of a seeded
    upstream gradient of the gates), as a CUDA graph of `reps` calls over buffer
    sets rotated at least 3x L2 apart; the first three calls run eagerly."""
    import moe_expert_routing_router_gb300 as mr
    esize = 2 if w.dtype == "bf16" else 4
    step_b = w.T * w.E * (esize + 4) + w.T * w.k * 20
    x0 = to_device(synth.router_logits(w), w.dtype, torch, device)
    n_sets = max(2, math.ceil(3 * L2_BYTES / (w.T * w.E * esize)))
    xs = [x0] + [x0.clone() for _ in range(n_sets - 1)]
    bufs = [out_buffers(w, torch, device) for _ in range(n_sets)]
    rng = np.random.default_rng(1)
    bias = torch.from_numpy((rng.standard_normal(w.E) * 0.5).astype(np.float32)).to(device)
    dgates = [torch.from_numpy(rng.standard_normal((w.T, w.k)).astype(np.float32)).to(device) for _ in range(n_sets)]
    ws = mr.Workspace(device)

    def call(i):
        j = i % n_sets
        mr.moe_router_step_ex(xs[j], w.k, w.alpha, w.capacity_factor, renorm=int(w.renorm), n_ranks=w.n_ranks,
                              bias=bias, bias_gamma=1e-3, bias_out=bias, dgate=dgates[j], ws=ws, out=bufs[j])

    us = _graph_us(torch, device, call, reps)
    gbs = step_b / (us * 1e-6) / 1e9
    return {"workload": w.name, "T": w.T, "us_per_call": round(us, 2), "tokens_per_s": round(w.T / (us * 1e-6), 1),
            "algorithmic_bytes": step_b, "achieved_gbs": round(gbs, 1), "frac_of_hbm_peak": round(gbs / hbm_gbs, 4)}


def time_eplb(torch, device, hbm_gbs: float, reps: int = 10) -> dict:
    """The batched EPLB planner (moe_eplb_plan) on 1024 problems of 384 experts,
    both policies, each a CUDA graph of `reps` calls; with the load balance it
    reaches (CV of the GPU loads against the CV of the expert loads)."""
    import moe_expert_routing_router_gb300 as mr
    w = synth.EPLB_WORKLOADS["eplb-zipf-E384-B1024"]
    loads_np = synth.eplb_loads(w)
    loads = torch.from_numpy(loads_np.astype(np.int32)).to(device)
    nbytes = w.B * (w.E * 4 + w.num_phys * 4 + w.E * 4 + w.num_gpus * 4)
    out = {"workload": w.name, "B": w.B, "E": w.E, "num_phys": w.num_phys, "num_gpus": w.num_gpus,
           "num_nodes": w.num_nodes, "bound": "latency (two sequential greedy loops per problem, one warp each)",
           "expert_load_cv_mean": round(float((loads_np.std(axis=1) / loads_np.mean(axis=1)).mean()), 4)}
    for policy, groups in (("global", 0), ("hierarchical", w.num_groups)):
        o = mr.moe_eplb_plan(loads, w.num_phys, w.num_gpus, w.num_nodes, groups)
        us = _graph_us(torch, device, lambda i: mr.moe_eplb_plan(loads, w.num_phys, w.num_gpus, w.num_nodes, groups,
                                                                  out=o), reps)
        gl = o["gpu_load"].double()
        cv = float((gl.std(dim=1, unbiased=False) / gl.mean(dim=1)).mean())
        out[policy] = {"num_groups": groups, "us_per_call": round(us, 2), "problems_per_s": round(w.B / (us * 1e-6), 1),
                       "gpu_load_cv_mean": round(cv, 4), "algorithmic_bytes": nbytes,
                       "frac_of_hbm_peak": round(nbytes / (us * 1e-6) / 1e9 / hbm_gbs, 5)}
    return out


def time_taot_match(torch, device, hbm_gbs: float, reps: int = 10, K: int = 4) -> dict:
    """TAOT Phase 2 (taot_match_batched) on 1024 microbatches of 384 experts over
    64 ranks in 8 nodes, up to K = 4 replicas per cold rank, fed by the Phase 1
    plan of taot_sinkhorn_batched; a CUDA graph of `reps` calls of Phase 1 +
    Phase 2 and of Phase 2 alone, with the residual imbalance (max - mean) / mean
    of the rank loads before and after."""
    import moe_expert_routing_router_gb300 as mr
    w = synth.EPLB_WORKLOADS["eplb-zipf-E384-B1024"]
    R, rpn = 64, 8
    loads = torch.from_numpy(synth.eplb_loads(w).astype(np.int32)).to(device)
    rank = loads.view(w.B, R, -1).sum(dim=2).float().contiguous()
    sk = mr.taot_sinkhorn_batched(rank, rpn, 10.0, 0.0, 50)
    o = mr.taot_match_batched(loads, sk["plan"], rpn, K)

    def both(i):
        mr.taot_sinkhorn_batched(rank, rpn, 10.0, 0.0, 50, out=sk)
        mr.taot_match_batched(loads, sk["plan"], rpn, K, out=o)

    us_both = _graph_us(torch, device, both, reps)
    us_match = _graph_us(torch, device, lambda i: mr.taot_match_batched(loads, sk["plan"], rpn, K, out=o), reps)
    before, after = rank.double(), o["rank_load"].double()
    imb = lambda x: float(((x.max(dim=1).values - x.mean(dim=1)) / x.mean(dim=1)).mean())
    nbytes = w.B * (w.E * 4 + R * R * 4 + 2 * R * K * 4 + R * 4)
    return {"workload": w.name, "B": w.B, "E": w.E, "R": R, "ranks_per_node": rpn, "K": K,
            "bound": "latency (dependent rounds of score, arbitration and commit per microbatch, until no cold rank matches)",
            "us_per_call_phase2": round(us_match, 2), "us_per_call_phase1_and_2": round(us_both, 2),
            "microbatches_per_s": round(w.B / (us_match * 1e-6), 1), "algorithmic_bytes_phase2": nbytes,
            "frac_of_hbm_peak": round(nbytes / (us_match * 1e-6) / 1e9 / hbm_gbs, 5),
            "residual_imbalance_before": round(imb(before), 4), "residual_imbalance_after": round(imb(after), 4)}


def time_sinkhorn(torch, device, hbm_gbs: float, reps: int = 20) -> dict:
    """The batched TAOT Sinkhorn call, timed as a CUDA graph of `reps` calls on
    the 1024-microbatch workload.  Its bound is the HBM write of the plan."""
    import moe_expert_routing_router_gb300 as mr
    s = synth.SINKHORN_WORKLOADS[SINKHORN_WORKLOAD]
    loads_path = ROOT / "tests" / "golden" / "taot_sinkhorn_B1024_R64_loads.npy"
    loads = torch.from_numpy(np.load(loads_path).astype(np.float32)).to(device)
    out = {"u": torch.empty_like(loads), "v": torch.empty_like(loads),
           "plan": torch.empty((s.B, s.R, s.R), dtype=torch.float32, device=device),
           "status": torch.empty(s.B, dtype=torch.int32, device=device)}
    call = lambda: mr.taot_sinkhorn_batched(loads, s.ranks_per_node, s.lam, s.eps, s.iters, out=out)
    for _ in range(3):
        call()
    torch.cuda.synchronize(device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):                  # captured on torch's side stream
        for _ in range(reps):
            call()
    stream = torch.cuda.current_stream(device)  # replay() runs on the current stream
    g.replay()
    torch.cuda.synchronize(device)
    ms = []
    for _ in range(5):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize(device)
        ms.append(a.elapsed_time(b) / reps)
    us = statistics.median(ms) * 1e3
    nbytes = 4 * (3 * s.B * s.R + s.B * s.R * s.R + s.B)   # loads in; u, v, plan, status out
    flops = s.B * s.iters * 2 * 2 * s.R * s.R              # the dense GEMV form, for reference
    gbs = nbytes / (us * 1e-6) / 1e9
    # Each microbatch is 2 * iters dependent O(R) sweeps (warp shuffles and a
    # reciprocal each): the call is bound by that chain's latency; the HBM
    # fraction of its bytes is reported beside it.
    return {"workload": SINKHORN_WORKLOAD, "us_per_call": round(us, 2), "bound": "latency",
            "algorithmic_bytes_per_call": nbytes, "achieved_gbs": round(gbs, 1), "peak_gbs": hbm_gbs,
            "frac_of_hbm_peak": round(gbs / hbm_gbs, 4),
            "dense_form_gflop_per_call": round(flops / 1e9, 4),
            "dense_form_equivalent_tflops": round(flops / (us * 1e-6) / 1e12, 2),
            "timing": f"CUDA graph of {reps} calls, median of 5 replays"}


# ----------------------------------------------------------------------------- CPU oracle

def oracle_step(w, logits: np.ndarray) -> None:
    """One pass of the oracle over a batch: forward, dispatch, backward."""
    import oracle
    fw = oracle.router.router_forward(logits, w.dtype, w.k, w.alpha, w.renorm, w.n_ranks)
    T = logits.shape[0]
    oracle.dispatch.dispatch(fw["idx"], w.E, oracle.dispatch.capacity(T, w.k, w.E, w.capacity_factor))
    oracle.router.aux_loss_grad(logits, w.dtype, fw["f"], w.alpha, 1.0)


def time_oracle(w, budget_s: float, min_steps: int = 1, rows: int | None = None) -> dict:
    """The oracle on a sample of `rows` tokens of the workload (default: sized
    so that about `budget_s` seconds of CPU work are done)."""
    if rows is None:
        probe = w.with_tokens(min(w.T, 2048))
        lg = synth.router_logits(probe)
        t0 = time.perf_counter()
        oracle_step(probe, lg)
        per_row = (time.perf_counter() - t0) / probe.T
        rows = int(min(w.T, max(256, budget_s / max(min_steps, 1) / per_row)))
    sample = w if rows == w.T else w.with_tokens(rows)
    lg = synth.router_logits(sample)
    times = []
    t_end = time.perf_counter() + budget_s
    while len(times) < min_steps or time.perf_counter() < t_end:
        t0 = time.perf_counter()
        oracle_step(sample, lg)
        times.append(time.perf_counter() - t0)
    sec = statistics.median(times)
    return {"value": rows / sec, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{rows} of {w.T} tokens of {w.name} (same E, k, recipe); median of {len(times)} "
                      f"oracle steps (fwd + dispatch + bwd, fp64 numpy, single thread; host nproc {os.cpu_count()})",
            "sec_per_step": sec, "rows": rows}


# ----------------------------------------------------------------------------- distributed

class DistCtx:
    def __init__(self, torch):
        self.torch = torch
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend=backend)
            self.dist = dist
            self.backend = backend

    def barrier(self):
        if self.world > 1:
            self.dist.barrier()

    def max(self, x: float) -> float:
        if self.world == 1:
            return x
        dev = f"cuda:{self.local}" if self.backend == "nccl" else "cpu"
        t = self.torch.tensor([x], dtype=self.torch.float64, device=dev)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.world > 1:
            self.dist.destroy_process_group()


# ----------------------------------------------------------------------------- main

def config_of(w, extra: dict | None = None) -> dict:
    c = {"workload": w.name, "T": w.T, "E": w.E, "k": w.k, "logits": w.dtype, "alpha": w.alpha,
         "capacity_factor": w.capacity_factor, "gate_renorm": w.renorm}
    if w.n_ranks:
        c["ep_ranks"] = w.n_ranks
        c["ranks_per_node"] = w.ranks_per_node
    if extra:
        c.update(extra)
    return c


def run_reference(args) -> dict:
    w = synth.ROUTER_WORKLOADS[args.workload]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if int(os.environ.get("RANK", "0")) != 0:
        return {}
    budget = 120.0 / max(args.steps + args.warmup, 1)       # whole run within ~2 minutes
    probe = time_oracle(w, budget_s=0.0, min_steps=1, rows=min(w.T, 2048))
    per_row = 1.0 / probe["value"]
    rows = int(min(w.T, max(256, budget / per_row)))
    sample = w if rows == w.T else w.with_tokens(rows)
    lg = synth.router_logits(sample)
    for _ in range(args.warmup):
        oracle_step(sample, lg)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(sample, lg)
    sec = (time.perf_counter() - t0) / args.steps
    value = rows / sec
    desc = (f"{rows} of {w.T} tokens of {w.name} per step; oracle fwd + dispatch + bwd "
            f"(fp64 numpy, single thread; host nproc {os.cpu_count()})")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, {"sample_tokens": rows}),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_dp(args, torch, dist_ctx, device, pk, w) -> dict:
    """The data-parallel partition of one batch over the ranks (weak scaling: w.T
    rows per rank), timed as dp.data_parallel_step."""
    sampler = ClockSampler(dist_ctx.local)
    r = time_dp(w, args.steps, args.warmup, torch, device, dist_ctx, sampler=sampler)
    e = time_dp(w, max(5, min(args.steps, 50)), args.warmup, torch, device, dist_ctx, e2e=True)
    ms = r["ms_per_step"]
    step_bytes = algorithmic_bytes(w)
    achieved = step_bytes / (ms * 1e-3) / 1e9
    kernels = ("moe_router_fwd", "moe_router_combine", "moe_shard_capacity_base", "moe_dispatch_sharded",
               "moe_router_bwd")
    line = {
        "metric": METRIC, "value": dist_ctx.world * w.T / (ms * 1e-3), "unit": "tokens/s",
        "n_gpus": dist_ctx.world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config_of(w, {"parallelism": f"dp{dist_ctx.world}", "global_batch": dist_ctx.world * w.T,
                                "l2": "each rank's logits exceed the 129 MB L2",
                                "timing": f"{args.steps} eager data-parallel steps between two CUDA events, "
                                          f"barrier and synchronize on both sides, slowest rank"}),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / pk["hbm_gbs"], 4), "traffic": None,
                     "kernel": "the whole step per rank: " + ", ".join(kernels) + " and one all-gather",
                     "algorithmic_bytes_per_launch": step_bytes, "peak_source": pk["source"]},
        "e2e": {"value": dist_ctx.world * w.T / (e["ms_per_step"] * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"], "ms_per_step": e["ms_per_step"],
                "steps": e["steps"],
                "timing": "the data-parallel step on pinned host buffers: logits copied in and every output "
                          "of the rank copied out each step"},
        "gpu_launches": len(kernels) * args.steps,
        "clocks": r["clocks"],
    }
    if dist_ctx.rank == 0:
        cb = time_oracle(w, budget_s=args.cpu_seconds, min_steps=2)
        line["cpu_baseline"] = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")}
    return line


def parallelism_of(choice: str, world: int) -> str:
    """dp (one batch split over the ranks) by default with several ranks,
    replicas (the fused step on every rank, or the single GPU) otherwise."""
    par = choice if choice != "auto" else ("dp" if world > 1 else "replicas")
    if par == "dp" and world < 2:
        raise SystemExit("--parallelism dp needs at least two ranks (torchrun)")
    return par


def run_ours(args) -> dict:
    import torch
    dist_ctx = DistCtx(torch)
    device = torch.device("cuda", dist_ctx.local)
    torch.cuda.set_device(device)
    pk = peaks()
    w = synth.ROUTER_WORKLOADS[args.workload]
    if parallelism_of(args.parallelism, dist_ctx.world) == "dp":
        line = run_dp(args, torch, dist_ctx, device, pk, w)
        dist_ctx.close()
        return line if dist_ctx.rank == 0 else {}
    sampler = ClockSampler(dist_ctx.local)
    r = time_router(w, args.steps, args.warmup, torch, device, dist_ctx, soak_s=args.soak_seconds, sampler=sampler)
    ms_step = r["total_ms"] / args.steps
    value = dist_ctx.world * w.T / (ms_step * 1e-3)
    achieved = r["step_bytes"] / (r["launch_ms_mean"] * 1e-3) / 1e9
    e2e = time_e2e(w, max(5, min(args.steps, 50)), args.warmup, torch, device, dist_ctx)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": dist_ctx.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config_of(w, {"l2": f"inputs and outputs rotated over {r['n_sets']} buffer sets "
                                      f"(>= 3x the 129 MB L2 between reuses)",
                                "parallelism": f"replicas x{dist_ctx.world}", "timing": r["timing"]}),
        "spread": r["spread"],
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / pk["hbm_gbs"], 4),
                     "traffic": (lambda t: None if t is None else t["read"] + t["write"])(measured_traffic(w.name)),
                     "kernel": "router_persistent_kernel (moe_router_step, one launch per step)",
                     "algorithmic_bytes_per_launch": r["step_bytes"],
                     "launch_us_mean": round(r["launch_ms_mean"] * 1e3, 2), "peak_source": pk["source"]},
        "e2e": {"value": dist_ctx.world * w.T / (e2e["ms_per_step"] * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "ms_per_step": e2e["ms_per_step"], "steps": e2e["steps"],
                "read_back": "every output of the step: idx, gate, counts, f, P, scalars, rank_load, perm, slot, "
                             "offsets, kept, n_dropped, dlogits",
                "timing": "C-ABI moe_router_step_host calls issued eagerly, alternating over two streams (each "
                          "with its own staging buffer and workspace; kernels ordered one after the other); the "
                          "logits copied from pinned host memory and every output copied back to pinned host "
                          "memory each step; CUDA events around all K steps"},
        "gpu_launches": args.steps,
        "clocks": r["clocks"],
    }
    if dist_ctx.rank == 0 and not args.no_extra:
        also = {}
        for name in EXTRA_WORKLOADS:
            wx = synth.ROUTER_WORKLOADS[name]
            kx = max(args.steps, 10)
            rx = time_router(wx, kx, args.warmup, torch, device, _Solo())
            msx = rx["total_ms"] / kx
            ach = rx["step_bytes"] / (rx["launch_ms_mean"] * 1e-3) / 1e9
            also[name] = {"value": wx.T / (msx * 1e-3), "unit": "tokens/s", "ms_per_step": msx,
                          "launch_us_mean": round(rx["launch_ms_mean"] * 1e3, 2),
                          "roofline_frac": round(ach / pk["hbm_gbs"], 4), "achieved_gbs": round(ach, 1),
                          "algorithmic_bytes_per_launch": rx["step_bytes"], "spread": rx["spread"],
                          "traffic": (lambda t: None if t is None else t["read"] + t["write"])(
                              measured_traffic(wx.name))}
        line["also"] = also
        line["separate_calls"] = {name: time_calls(synth.ROUTER_WORKLOADS[name], torch, device, pk["hbm_gbs"])
                                  for name in DETAIL_WORKLOADS}
        line["sinkhorn"] = time_sinkhorn(torch, device, pk["hbm_gbs"])
        line["eplb"] = time_eplb(torch, device, pk["hbm_gbs"])
        line["taot_match"] = time_taot_match(torch, device, pk["hbm_gbs"])
        line["next_steps"] = {name: time_next_steps(synth.ROUTER_WORKLOADS[name], torch, device, pk["hbm_gbs"])
                              for name in DETAIL_WORKLOADS}
    if dist_ctx.rank == 0:
        cb = time_oracle(w, budget_s=args.cpu_seconds, min_steps=2)
        line["cpu_baseline"] = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")}
    dist_ctx.close()
    return line if dist_ctx.rank == 0 else {}


class _Solo:
    def barrier(self):
        pass

    def max(self, x):
        return x


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(synth.ROUTER_WORKLOADS))
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads and the Sinkhorn line")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--soak-seconds", type=float, default=1.0,
                    help="loaded window before the timed region, for the clock samples")
    ap.add_argument("--parallelism", choices=("auto", "dp", "replicas"), default="auto",
                    help="with N > 1 ranks: dp (default) splits one batch over the ranks (dp.data_parallel_step); "
                         "replicas runs the fused step independently on every rank")
    ap.add_argument("--tokens", type=int, default=None,
                    help="with --section step, next_steps or step_ex: the workload cut to this many rows")
    ap.add_argument("--section", choices=("step", "next_steps", "step_ex", "eplb", "taot_match"), default=None,
                    help="print only this part of the extra lines (for --workload), as JSON; no bench line")
    args = ap.parse_args()
    if args.warmup < 3:
        log("warmup raised to 3")
        args.warmup = 3
    if args.section is not None:
        import torch
        device = torch.device("cuda", 0)
        torch.cuda.set_device(device)
        hbm = peaks()["hbm_gbs"]
        wsec = synth.ROUTER_WORKLOADS[args.workload]
        if args.tokens is not None and args.tokens != wsec.T:
            wsec = wsec.with_tokens(args.tokens)
        part = (time_step(wsec, torch, device, hbm) if args.section == "step" else
                time_next_steps(wsec, torch, device, hbm)
                if args.section == "next_steps" else
                time_step_ex(wsec, torch, device, hbm) if args.section == "step_ex" else
                time_eplb(torch, device, hbm) if args.section == "eplb" else time_taot_match(torch, device, hbm))
        print(json.dumps(part), flush=True)
        return 0
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
