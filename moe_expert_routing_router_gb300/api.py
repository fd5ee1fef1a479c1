"""Python binding of the C ABI (include/moe_router.h): argument marshalling only.

Every function takes CUDA tensors, allocates outputs with torch (device memory
is the only thing torch provides here), passes raw pointers and the current
torch stream to the library, and checks the returned status.  All arithmetic
runs in the library's CUDA kernels; nothing here computes on the host.
"""

from __future__ import annotations

import contextlib
import ctypes as C
import functools
import inspect

import torch

from . import _native
from ._native import MOE_DTYPE_BF16, MOE_DTYPE_FP32, MOE_NUM_SCALARS, SCALAR_NAMES, check, lib

__all__ = [
    "Workspace", "moe_router_fwd", "moe_router_bwd", "moe_dispatch", "moe_dispatch_capacity",
    "moe_shard_capacity_base", "moe_dispatch_sharded", "moe_router_step_ex",
    "moe_router_step", "moe_router_step_static", "moe_router_fwd_ex", "moe_router_bwd_full", "moe_eplb_plan", "taot_match_batched", "moe_router_combine", "taot_sinkhorn_batched", "moe_get_device_status", "SCALAR_NAMES",
]

_DTYPES = {torch.float32: MOE_DTYPE_FP32, torch.bfloat16: MOE_DTYPE_BF16}


def _stream_handle(stream: torch.cuda.Stream | None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _on(stream: torch.cuda.Stream | None):
    """`stream` as torch's current stream while a call allocates (or nothing
    when the caller gives none: the current stream is the kernels' stream)."""
    return torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext()


def _on_stream(fn):
    """Runs an entry point with its `stream` argument, when given, as torch's
    current stream.  The outputs and workspaces it allocates then belong to the
    stream its kernels write them on, so the caching allocator neither hands
    the kernels memory that other streams' pending work still uses nor reuses
    an output before that stream is done with it."""
    pos = list(inspect.signature(fn).parameters).index("stream")

    @functools.wraps(fn)
    def call(*args, **kwargs):
        stream = args[pos] if len(args) > pos else kwargs.get("stream")
        with _on(stream):
            return fn(*args, **kwargs)
    return call


def _event_handle(ev: torch.cuda.Event | None) -> int | None:
    """The cudaEvent_t of a torch event (created on first record), or None."""
    if ev is None:
        return None
    h = int(ev.cuda_event)
    if h == 0:
        raise ValueError("the event has not been recorded yet, so it has no CUDA handle")
    return h


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else int(t.data_ptr())


def _need_cuda(name: str, t: torch.Tensor, dtype: torch.dtype | None = None) -> None:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


class Workspace:
    """Device scratch of the persistent kernels, zero-filled once at creation.

    One workspace serves calls ordered on one stream; it grows on demand.
    """

    def __init__(self, device: torch.device | int | None = None):
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None else
                                   (device.index if isinstance(device, torch.device) else device))
        self.buf: torch.Tensor | None = None

    def ensure(self, T: int, E: int, k: int, stream: torch.cuda.Stream | None = None) -> tuple[int, int]:
        need = int(lib().moe_router_workspace_size(T, E, k))
        if need == 0:
            raise ValueError(f"invalid sizes for a workspace: T={T}, E={E}, k={k}")
        if self.buf is None or self.buf.numel() < need:
            with _on(stream):
                self.buf = torch.empty(need, dtype=torch.uint8, device=self.device)
            check(lib().moe_workspace_init(_ptr(self.buf), need, _stream_handle(stream)), "moe_workspace_init")
        return _ptr(self.buf), int(self.buf.numel())


_workspaces: dict[tuple[int, int], Workspace] = {}


def _default_ws(device: torch.device, stream: torch.cuda.Stream | None) -> Workspace:
    key = (device.index, _stream_handle(stream))
    ws = _workspaces.get(key)
    if ws is None:
        ws = _workspaces[key] = Workspace(device)
    return ws


def _out(out: dict | None, name: str, shape, dtype, device) -> torch.Tensor:
    if out is not None and name in out and out[name] is not None:
        t = out[name]
        if tuple(t.shape) != tuple(shape) or t.dtype != dtype or t.device != device or not t.is_contiguous():
            raise ValueError(f"out[{name!r}] must be a contiguous {dtype} tensor of shape {tuple(shape)} on {device}")
        return t
    return torch.empty(shape, dtype=dtype, device=device)


def _fwd_outputs(T: int, E: int, k: int, n_ranks: int, device, out: dict | None) -> dict:
    return {
        "idx": _out(out, "idx", (T, k), torch.int32, device),
        "gate": _out(out, "gate", (T, k), torch.float32, device),
        "counts": _out(out, "counts", (E,), torch.int32, device),
        "f": _out(out, "f", (E,), torch.float32, device),
        "P": _out(out, "P", (E,), torch.float32, device),
        "scalars": _out(out, "scalars", (MOE_NUM_SCALARS,), torch.float32, device),
        "rank_load": _out(out, "rank_load", (max(n_ranks, 0),), torch.int32, device),
    }


def _dispatch_outputs(T: int, E: int, k: int, device, out: dict | None) -> dict:
    return {
        "perm": _out(out, "perm", (T * k,), torch.int32, device),
        "slot": _out(out, "slot", (T * k,), torch.int32, device),
        "offsets": _out(out, "offsets", (E + 1,), torch.int32, device),
        "kept": _out(out, "kept", (E,), torch.int32, device),
        "n_dropped": _out(out, "n_dropped", (1,), torch.int32, device),
    }


@_on_stream
def moe_router_fwd(logits: torch.Tensor, k: int, alpha: float, renorm: int = -1, n_ranks: int = 0,
                   ws: Workspace | None = None, out: dict | None = None,
                   stream: torch.cuda.Stream | None = None) -> dict:
    """Router softmax, top-k, gates, counts, f, P, scalars and rank loads (C: moe_router_fwd)."""
    _need_cuda("logits", logits)
    if logits.dtype not in _DTYPES or logits.dim() != 2:
        raise ValueError("logits must be a 2-D float32 or bfloat16 tensor")
    T, E = logits.shape
    o = _fwd_outputs(T, E, k, n_ranks, logits.device, out)
    ws = ws or _default_ws(logits.device, stream)
    wp, wn = ws.ensure(T, E, k, stream)
    st = lib().moe_router_fwd(_ptr(logits), _DTYPES[logits.dtype], T, E, k, float(alpha), int(renorm), int(n_ranks),
                              _ptr(o["idx"]), _ptr(o["gate"]), _ptr(o["counts"]), _ptr(o["f"]), _ptr(o["P"]),
                              _ptr(o["scalars"]), _ptr(o["rank_load"]) if n_ranks > 0 else None,
                              wp, wn, _stream_handle(stream))
    check(st, "moe_router_fwd")
    return o


@_on_stream
def moe_router_bwd(logits: torch.Tensor, f: torch.Tensor, alpha: float, grad_scale: float = 1.0,
                   dlogits: torch.Tensor | None = None, stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """dL_aux/dlogits with f held constant (C: moe_router_bwd)."""
    _need_cuda("logits", logits)
    _need_cuda("f", f, torch.float32)
    if logits.dtype not in _DTYPES or logits.dim() != 2:
        raise ValueError("logits must be a 2-D float32 or bfloat16 tensor")
    T, E = logits.shape
    if f.numel() != E:
        raise ValueError("f must have E elements")
    dl = _out({"dlogits": dlogits}, "dlogits", (T, E), torch.float32, logits.device)
    st = lib().moe_router_bwd(_ptr(logits), _DTYPES[logits.dtype], T, E, float(alpha), _ptr(f), float(grad_scale),
                              _ptr(dl), _stream_handle(stream))
    check(st, "moe_router_bwd")
    return dl


@_on_stream
def moe_router_fwd_ex(logits: torch.Tensor, k: int, alpha: float, renorm: int = -1, n_ranks: int = 0,
                      bias: torch.Tensor | None = None, masked_p: bool = False, bias_gamma: float = 0.0,
                      bias_out: torch.Tensor | bool | None = None, ws: Workspace | None = None,
                      out: dict | None = None, stream: torch.cuda.Stream | None = None) -> dict:
    """Router forward with bias routing and/or masked P (C: moe_router_fwd_ex).

    ``bias`` [E] fp32 steers selection only; ``bias_out`` is a tensor to
    receive the updated bias (it may be ``bias`` itself), True for a new one,
    or None for no update.  The result holds the outputs of moe_router_fwd
    and, with an update, ``bias_out``.
    """
    _need_cuda("logits", logits)
    if logits.dtype not in _DTYPES or logits.dim() != 2:
        raise ValueError("logits must be a 2-D float32 or bfloat16 tensor")
    T, E = logits.shape
    if bias is not None:
        _need_cuda("bias", bias, torch.float32)
        if bias.numel() != E:
            raise ValueError("bias must have E elements")
    if bias_out is True:
        bias_out = torch.empty(E, dtype=torch.float32, device=logits.device)
    elif bias_out is False:
        bias_out = None
    if bias_out is not None:
        _need_cuda("bias_out", bias_out, torch.float32)
        if bias_out.numel() != E:
            raise ValueError("bias_out must have E elements")
    o = _fwd_outputs(T, E, k, n_ranks, logits.device, out)
    ws = ws or _default_ws(logits.device, stream)
    wp, wn = ws.ensure(T, E, k, stream)
    st = lib().moe_router_fwd_ex(_ptr(logits), _DTYPES[logits.dtype], T, E, k, float(alpha), int(renorm),
                                 int(n_ranks), _ptr(bias), int(bool(masked_p)), float(bias_gamma), _ptr(bias_out),
                                 _ptr(o["idx"]), _ptr(o["gate"]), _ptr(o["counts"]), _ptr(o["f"]), _ptr(o["P"]),
                                 _ptr(o["scalars"]), _ptr(o["rank_load"]) if n_ranks > 0 else None,
                                 wp, wn, _stream_handle(stream))
    check(st, "moe_router_fwd_ex")
    if bias_out is not None:
        o["bias_out"] = bias_out
    return o


@_on_stream
def moe_router_bwd_full(logits: torch.Tensor, f: torch.Tensor, alpha: float, grad_scale: float = 1.0,
                        idx: torch.Tensor | None = None, dgate: torch.Tensor | None = None, renorm: int = -1,
                        masked_p: bool = False, k: int | None = None, dlogits: torch.Tensor | None = None,
                        stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Gradient of sum(dgate * gate) + grad_scale * L_aux with respect to the logits,
    picks and f held constant (C: moe_router_bwd_full)."""
    _need_cuda("logits", logits)
    _need_cuda("f", f, torch.float32)
    if logits.dtype not in _DTYPES or logits.dim() != 2:
        raise ValueError("logits must be a 2-D float32 or bfloat16 tensor")
    T, E = logits.shape
    if f.numel() != E:
        raise ValueError("f must have E elements")
    if idx is not None:
        _need_cuda("idx", idx, torch.int32)
        if idx.dim() != 2 or idx.shape[0] != T:
            raise ValueError("idx must be [T, k]")
        k = idx.shape[1]
    if dgate is not None:
        _need_cuda("dgate", dgate, torch.float32)
        if idx is None or tuple(dgate.shape) != tuple(idx.shape):
            raise ValueError("dgate needs idx of the same [T, k] shape")
    if k is None:
        raise ValueError("k is needed when idx is not given")
    dl = _out({"dlogits": dlogits}, "dlogits", (T, E), torch.float32, logits.device)
    st = lib().moe_router_bwd_full(_ptr(logits), _DTYPES[logits.dtype], T, E, int(k), float(alpha), _ptr(f),
                                   float(grad_scale), int(bool(masked_p)), _ptr(idx), _ptr(dgate), int(renorm),
                                   _ptr(dl), _stream_handle(stream))
    check(st, "moe_router_bwd_full")
    return dl


@functools.lru_cache(maxsize=256)
def _capacity(T: int, E: int, k: int, capacity_factor: float) -> int:
    return int(lib().moe_dispatch_capacity(T, E, k, capacity_factor))


def moe_dispatch_capacity(T: int, E: int, k: int, capacity_factor: float) -> int:
    """Expert capacity ceil(ceil(T*k/E) * capacity_factor) (C: moe_dispatch_capacity; the
    library's answer is remembered per argument tuple)."""
    c = _capacity(int(T), int(E), int(k), float(capacity_factor))
    if c < 0:
        raise ValueError("invalid capacity arguments")
    return c


@_on_stream
def moe_dispatch(idx: torch.Tensor, E: int, capacity_factor: float, ws: Workspace | None = None,
                 out: dict | None = None, stream: torch.cuda.Stream | None = None) -> dict:
    """Stable capacity-limited dispatch of idx [T, k] (C: moe_dispatch)."""
    _need_cuda("idx", idx, torch.int32)
    if idx.dim() != 2:
        raise ValueError("idx must be [T, k]")
    T, k = idx.shape
    o = _dispatch_outputs(T, E, k, idx.device, out)
    ws = ws or _default_ws(idx.device, stream)
    wp, wn = ws.ensure(T, E, k, stream)
    cap = C.c_int64(0)
    st = lib().moe_dispatch(_ptr(idx), T, E, k, float(capacity_factor), _ptr(o["perm"]), _ptr(o["slot"]),
                            _ptr(o["offsets"]), _ptr(o["kept"]), _ptr(o["n_dropped"]), C.byref(cap),
                            wp, wn, _stream_handle(stream))
    check(st, "moe_dispatch")
    o["capacity"] = int(cap.value)
    return o


@_on_stream
def moe_shard_capacity_base(counts: torch.Tensor, rank: int, out: torch.Tensor | None = None,
                            stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """cap_base [E] int32: every expert's assignments on the ranks below `rank`,
    from the ranks' counts stacked [G, E] in rank order (C: moe_shard_capacity_base)."""
    _need_cuda("counts", counts, torch.int32)
    if counts.dim() != 2:
        raise ValueError("counts must be [G, E]")
    G, E = counts.shape
    base = out if out is not None else torch.empty(E, dtype=torch.int32, device=counts.device)
    _need_cuda("out", base, torch.int32)
    if tuple(base.shape) != (E,):
        raise ValueError("out must be [E]")
    st = lib().moe_shard_capacity_base(_ptr(counts), G, E, int(rank), _ptr(base), _stream_handle(stream))
    check(st, "moe_shard_capacity_base")
    return base


@_on_stream
def moe_dispatch_sharded(idx: torch.Tensor, E: int, capacity_factor: float, T_total: int, cap_base: torch.Tensor,
                         ws: Workspace | None = None, out: dict | None = None,
                         stream: torch.cuda.Stream | None = None) -> dict:
    """Dispatch of this rank's idx [T, k] with the capacity of the whole batch of
    T_total rows and slots offset by cap_base [E] (C: moe_dispatch_sharded)."""
    _need_cuda("idx", idx, torch.int32)
    _need_cuda("cap_base", cap_base, torch.int32)
    if idx.dim() != 2:
        raise ValueError("idx must be [T, k]")
    if tuple(cap_base.shape) != (E,):
        raise ValueError("cap_base must be [E]")
    T, k = idx.shape
    o = _dispatch_outputs(T, E, k, idx.device, out)
    ws = ws or _default_ws(idx.device, stream)
    wp, wn = ws.ensure(T, E, k, stream)
    cap = C.c_int64(0)
    st = lib().moe_dispatch_sharded(_ptr(idx), T, E, k, float(capacity_factor), int(T_total), _ptr(cap_base),
                                    _ptr(o["perm"]), _ptr(o["slot"]), _ptr(o["offsets"]), _ptr(o["kept"]),
                                    _ptr(o["n_dropped"]), C.byref(cap), wp, wn, _stream_handle(stream))
    check(st, "moe_dispatch_sharded")
    o["capacity"] = int(cap.value)
    return o


@_on_stream
def moe_router_step(logits: torch.Tensor, k: int, alpha: float, capacity_factor: float, renorm: int = -1,
                    n_ranks: int = 0, grad_scale: float = 1.0, ws: Workspace | None = None,
                    out: dict | None = None, stream: torch.cuda.Stream | None = None) -> dict:
    """Forward + dispatch + backward in one launch (C: moe_router_step)."""
    _need_cuda("logits", logits)
    if logits.dtype not in _DTYPES or logits.dim() != 2:
        raise ValueError("logits must be a 2-D float32 or bfloat16 tensor")
    T, E = logits.shape
    dev = logits.device
    o = _fwd_outputs(T, E, k, n_ranks, dev, out)
    o.update(_dispatch_outputs(T, E, k, dev, out))
    o["dlogits"] = _out(out, "dlogits", (T, E), torch.float32, dev)
    ws = ws or _default_ws(dev, stream)
    wp, wn = ws.ensure(T, E, k, stream)
    st = lib().moe_router_step(_ptr(logits), _DTYPES[logits.dtype], T, E, k, float(alpha), int(renorm), int(n_ranks),
                               float(capacity_factor), float(grad_scale),
                               _ptr(o["idx"]), _ptr(o["gate"]), _ptr(o["counts"]), _ptr(o["f"]), _ptr(o["P"]),
                               _ptr(o["scalars"]), _ptr(o["rank_load"]) if n_ranks > 0 else None,
                               _ptr(o["perm"]), _ptr(o["slot"]), _ptr(o["offsets"]), _ptr(o["kept"]),
                               _ptr(o["n_dropped"]), _ptr(o["dlogits"]), wp, wn, _stream_handle(stream))
    check(st, "moe_router_step")
    o["capacity"] = moe_dispatch_capacity(T, E, k, capacity_factor)
    return o


@_on_stream
def moe_router_step_ex(logits: torch.Tensor, k: int, alpha: float, capacity_factor: float, renorm: int = -1,
                       n_ranks: int = 0, grad_scale: float = 1.0, bias: torch.Tensor | None = None,
                       bias_gamma: float = 0.0, bias_out: torch.Tensor | bool | None = None, masked_p: bool = False,
                       dgate: torch.Tensor | None = None, ws: Workspace | None = None, out: dict | None = None,
                       stream: torch.cuda.Stream | None = None) -> dict:
    """The extended step in one launch: bias routing with its update and masked
    P in the forward, dispatch, and the backward of the gates' upstream
    gradient dgate [T, k] added to the aux loss's (C: moe_router_step_ex).
    ``bias`` / ``bias_out`` as for moe_router_fwd_ex."""
    _need_cuda("logits", logits)
    if logits.dtype not in _DTYPES or logits.dim() != 2:
        raise ValueError("logits must be a 2-D float32 or bfloat16 tensor")
    T, E = logits.shape
    dev = logits.device
    if bias is not None:
        _need_cuda("bias", bias, torch.float32)
        if bias.numel() != E:
            raise ValueError("bias must have E elements")
    if bias_out is True:
        bias_out = torch.empty(E, dtype=torch.float32, device=dev)
    elif bias_out is False:
        bias_out = None
    if bias_out is not None:
        _need_cuda("bias_out", bias_out, torch.float32)
        if bias_out.numel() != E:
            raise ValueError("bias_out must have E elements")
    if dgate is not None:
        _need_cuda("dgate", dgate, torch.float32)
        if tuple(dgate.shape) != (T, k):
            raise ValueError("dgate must be [T, k]")
    o = _fwd_outputs(T, E, k, n_ranks, dev, out)
    o.update(_dispatch_outputs(T, E, k, dev, out))
    o["dlogits"] = _out(out, "dlogits", (T, E), torch.float32, dev)
    ws = ws or _default_ws(dev, stream)
    wp, wn = ws.ensure(T, E, k, stream)
    st = lib().moe_router_step_ex(_ptr(logits), _DTYPES[logits.dtype], T, E, k, float(alpha), int(renorm),
                                  int(n_ranks), float(capacity_factor), float(grad_scale), _ptr(bias),
                                  float(bias_gamma), _ptr(bias_out), int(bool(masked_p)), _ptr(dgate),
                                  _ptr(o["idx"]), _ptr(o["gate"]), _ptr(o["counts"]), _ptr(o["f"]), _ptr(o["P"]),
                                  _ptr(o["scalars"]), _ptr(o["rank_load"]) if n_ranks > 0 else None,
                                  _ptr(o["perm"]), _ptr(o["slot"]), _ptr(o["offsets"]), _ptr(o["kept"]),
                                  _ptr(o["n_dropped"]), _ptr(o["dlogits"]), wp, wn, _stream_handle(stream))
    check(st, "moe_router_step_ex")
    o["capacity"] = moe_dispatch_capacity(T, E, k, capacity_factor)
    if bias_out is not None:
        o["bias_out"] = bias_out
    return o


def moe_router_step_host_device_size(dtype: torch.dtype, T: int, E: int, k: int, n_ranks: int = 0) -> int:
    """Bytes of the device staging buffer moe_router_step_host needs (C: moe_router_step_host_device_size)."""
    return int(lib().moe_router_step_host_device_size(_DTYPES[dtype], T, E, k, n_ranks))


def host_step_outputs(T: int, E: int, k: int, n_ranks: int = 0, pin: bool = True) -> dict:
    """Page-locked host arrays for every output of moe_router_step_host."""
    i32, f32 = torch.int32, torch.float32
    shapes = {"idx": ((T, k), i32), "gate": ((T, k), f32), "counts": ((E,), i32), "f": ((E,), f32),
              "P": ((E,), f32), "scalars": ((_native.MOE_NUM_SCALARS,), f32), "rank_load": ((max(n_ranks, 0),), i32),
              "perm": ((T * k,), i32), "slot": ((T * k,), i32), "offsets": ((E + 1,), i32), "kept": ((E,), i32),
              "n_dropped": ((1,), i32), "dlogits": ((T, E), f32)}
    return {name: torch.empty(shape, dtype=dt, pin_memory=pin) for name, (shape, dt) in shapes.items()}


@_on_stream
def moe_router_step_host(logits: torch.Tensor, k: int, alpha: float, capacity_factor: float, renorm: int = -1,
                         n_ranks: int = 0, grad_scale: float = 1.0, ws: Workspace | None = None,
                         dev: torch.Tensor | None = None, out: dict | None = None,
                         stream: torch.cuda.Stream | None = None, device: torch.device | int | None = None,
                         kernel_after: torch.cuda.Event | None = None,
                         kernel_done: torch.cuda.Event | None = None) -> dict:
    """The step on HOST logits with every output copied back to HOST arrays
    (C: moe_router_step_host).  logits: a contiguous CPU tensor (pinned for
    asynchronous copies); out: host arrays as from host_step_outputs; dev: the
    device staging buffer (uint8, moe_router_step_host_device_size bytes);
    kernel_after / kernel_done: events the step's kernel waits for / records.
    Asynchronous on `stream`: synchronise before reading the outputs."""
    if logits.device.type != "cpu" or not logits.is_contiguous():
        raise ValueError("logits must be a contiguous CPU tensor")
    if logits.dtype not in _DTYPES or logits.dim() != 2:
        raise ValueError("logits must be a 2-D float32 or bfloat16 tensor")
    T, E = logits.shape
    d = torch.device("cuda", torch.cuda.current_device() if device is None else
                     (device.index if isinstance(device, torch.device) else device))
    o = out if out is not None else host_step_outputs(T, E, k, n_ranks)
    need = moe_router_step_host_device_size(logits.dtype, T, E, k, n_ranks)
    if dev is None:
        dev = torch.empty(need, dtype=torch.uint8, device=d)
    ws = ws or _default_ws(d, stream)
    wp, wn = ws.ensure(T, E, k, stream)
    st = lib().moe_router_step_host(_ptr(logits), _DTYPES[logits.dtype], T, E, k, float(alpha), int(renorm),
                                    int(n_ranks), float(capacity_factor), float(grad_scale),
                                    _ptr(o["idx"]), _ptr(o["gate"]), _ptr(o["counts"]), _ptr(o["f"]), _ptr(o["P"]),
                                    _ptr(o["scalars"]), _ptr(o["rank_load"]) if n_ranks > 0 else None,
                                    _ptr(o["perm"]), _ptr(o["slot"]), _ptr(o["offsets"]), _ptr(o["kept"]),
                                    _ptr(o["n_dropped"]), _ptr(o["dlogits"]), _ptr(dev), int(dev.numel()),
                                    wp, wn, _event_handle(kernel_after), _event_handle(kernel_done),
                                    _stream_handle(stream))
    check(st, "moe_router_step_host")
    return o


@_on_stream
def moe_router_step_static(logits: torch.Tensor, k: int, alpha: float, capacity_factor: float, renorm: int = -1,
                           n_ranks: int = 0, grad_scale: float = 1.0, out: dict | None = None,
                           stream: torch.cuda.Stream | None = None) -> dict:
    """moe_router_step without a workspace, for callers that cannot allocate device
    scratch (C: moe_router_step_static; E <= 512; calls that overlap on the GPU race)."""
    _need_cuda("logits", logits)
    if logits.dtype not in _DTYPES or logits.dim() != 2:
        raise ValueError("logits must be a 2-D float32 or bfloat16 tensor")
    T, E = logits.shape
    dev = logits.device
    o = _fwd_outputs(T, E, k, n_ranks, dev, out)
    o.update(_dispatch_outputs(T, E, k, dev, out))
    o["dlogits"] = _out(out, "dlogits", (T, E), torch.float32, dev)
    st = lib().moe_router_step_static(_ptr(logits), _DTYPES[logits.dtype], T, E, k, float(alpha), int(renorm),
                                      int(n_ranks), float(capacity_factor), float(grad_scale),
                                      _ptr(o["idx"]), _ptr(o["gate"]), _ptr(o["counts"]), _ptr(o["f"]), _ptr(o["P"]),
                                      _ptr(o["scalars"]), _ptr(o["rank_load"]) if n_ranks > 0 else None,
                                      _ptr(o["perm"]), _ptr(o["slot"]), _ptr(o["offsets"]), _ptr(o["kept"]),
                                      _ptr(o["n_dropped"]), _ptr(o["dlogits"]), _stream_handle(stream))
    check(st, "moe_router_step_static")
    return o


@_on_stream
def taot_sinkhorn_batched(loads: torch.Tensor, ranks_per_node: int, lam: float, eps: float = 0.0,
                          iters: int = 50, with_plan: bool = True, out: dict | None = None,
                          stream: torch.cuda.Stream | None = None) -> dict:
    """TAOT Phase 1 topology-aware Sinkhorn plan per microbatch (C: taot_sinkhorn_batched)."""
    _need_cuda("loads", loads, torch.float32)
    if loads.dim() != 2:
        raise ValueError("loads must be [B, R]")
    B, R = loads.shape
    dev = loads.device
    o = {
        "u": _out(out, "u", (B, R), torch.float32, dev),
        "v": _out(out, "v", (B, R), torch.float32, dev),
        "plan": _out(out, "plan", (B, R, R), torch.float32, dev) if with_plan else None,
        "status": _out(out, "status", (B,), torch.int32, dev),
    }
    st = lib().taot_sinkhorn_batched(_ptr(loads), B, R, ranks_per_node, float(lam), float(eps), int(iters),
                                     _ptr(o["u"]), _ptr(o["v"]), _ptr(o["plan"]), _ptr(o["status"]),
                                     _stream_handle(stream))
    check(st, "taot_sinkhorn_batched")
    return o


@_on_stream
def moe_eplb_plan(loads: torch.Tensor, num_phys: int, num_gpus: int, num_nodes: int = 1, num_groups: int = 0,
                  out: dict | None = None, stream: torch.cuda.Stream | None = None) -> dict:
    """EPLB replication and balanced packing of B problems (C: moe_eplb_plan).

    loads [B, E] int32 expert token counts; returns phy2log [B, num_phys],
    log_count [B, E] and gpu_load [B, num_gpus]."""
    _need_cuda("loads", loads, torch.int32)
    if loads.dim() != 2:
        raise ValueError("loads must be [B, E]")
    B, E = loads.shape
    dev = loads.device
    o = {
        "phy2log": _out(out, "phy2log", (B, num_phys), torch.int32, dev),
        "log_count": _out(out, "log_count", (B, E), torch.int32, dev),
        "gpu_load": _out(out, "gpu_load", (B, num_gpus), torch.float32, dev),
    }
    st = lib().moe_eplb_plan(_ptr(loads), B, E, int(num_phys), int(num_gpus), int(num_nodes), int(num_groups),
                             _ptr(o["phy2log"]), _ptr(o["log_count"]), _ptr(o["gpu_load"]), _stream_handle(stream))
    check(st, "moe_eplb_plan")
    return o


@_on_stream
def taot_match_batched(expert_loads: torch.Tensor, plan: torch.Tensor, ranks_per_node: int, K: int,
                       out: dict | None = None, stream: torch.cuda.Stream | None = None) -> dict:
    """TAOT Phase 2 column-first matching of hot experts to cold ranks (C: taot_match_batched).

    expert_loads [B, E] int32, plan [B, R, R] fp32 (the Phase 1 flow); returns
    slot_expert and slot_tokens [B, R, K] and rank_load [B, R]."""
    _need_cuda("expert_loads", expert_loads, torch.int32)
    _need_cuda("plan", plan, torch.float32)
    if expert_loads.dim() != 2 or plan.dim() != 3 or plan.shape[0] != expert_loads.shape[0] or plan.shape[1] != plan.shape[2]:
        raise ValueError("expert_loads must be [B, E] and plan [B, R, R]")
    B, E = expert_loads.shape
    R = plan.shape[1]
    dev = expert_loads.device
    o = {
        "slot_expert": _out(out, "slot_expert", (B, R, K), torch.int32, dev),
        "slot_tokens": _out(out, "slot_tokens", (B, R, K), torch.int32, dev),
        "rank_load": _out(out, "rank_load", (B, R), torch.int32, dev),
    }
    st = lib().taot_match_batched(_ptr(expert_loads), _ptr(plan), B, E, R, int(ranks_per_node), int(K),
                                  _ptr(o["slot_expert"]), _ptr(o["slot_tokens"]), _ptr(o["rank_load"]),
                                  _stream_handle(stream))
    check(st, "taot_match_batched")
    return o


@_on_stream
def moe_router_combine(counts: torch.Tensor, P: torch.Tensor, T_shard, k: int, alpha: float, n_ranks: int = 0,
                       masked_p: bool = False, out: dict | None = None,
                       stream: torch.cuda.Stream | None = None) -> dict:
    """The whole batch's counts, f, P, scalars and rank loads from G shards'
    forward statistics (C: moe_router_combine).  counts [G, E] int32, P [G, E]
    fp32 on the GPU; T_shard: the G shards' token counts (host integers)."""
    _need_cuda("counts", counts, torch.int32)
    _need_cuda("P", P, torch.float32)
    if counts.dim() != 2 or tuple(P.shape) != tuple(counts.shape):
        raise ValueError("counts and P must both be [G, E]")
    G, E = counts.shape
    T_list = [int(t) for t in T_shard]
    if len(T_list) != G:
        raise ValueError("T_shard must have G entries")
    dev = counts.device
    o = {
        "counts": _out(out, "counts", (E,), torch.int32, dev),
        "f": _out(out, "f", (E,), torch.float32, dev),
        "P": _out(out, "P", (E,), torch.float32, dev),
        "scalars": _out(out, "scalars", (MOE_NUM_SCALARS,), torch.float32, dev),
        "rank_load": _out(out, "rank_load", (max(n_ranks, 0),), torch.int32, dev),
    }
    tarr = (C.c_int64 * G)(*T_list)
    st = lib().moe_router_combine(_ptr(counts), _ptr(P), tarr, G, E, int(k), float(alpha), int(n_ranks),
                                  int(bool(masked_p)), _ptr(o["counts"]), _ptr(o["f"]), _ptr(o["P"]),
                                  _ptr(o["scalars"]), _ptr(o["rank_load"]) if n_ranks > 0 else None,
                                  _stream_handle(stream))
    check(st, "moe_router_combine")
    return o


def moe_get_device_status(ws: Workspace | None, stream: torch.cuda.Stream | None = None) -> int:
    """Reads and clears the device error flags of a workspace (synchronises);
    ws=None reads those of moe_router_step_static's fixed scratch on the
    current device."""
    if ws is not None and ws.buf is None:
        return 0
    flags = C.c_int32(0)
    st = lib().moe_get_device_status(None if ws is None else _ptr(ws.buf), _stream_handle(stream), C.byref(flags))
    if st not in (_native.MOE_OK, _native.MOE_ERR_TIMEOUT):
        check(st, "moe_get_device_status")
    return int(flags.value)
