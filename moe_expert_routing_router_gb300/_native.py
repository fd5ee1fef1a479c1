"""Loads the in-tree C-ABI library and declares its entry points (ctypes).

There is no fallback: if ``_lib/libmoerouter.so`` is missing or fails to
load, every call raises.  Build it with ``python -m
moe_expert_routing_router_gb300.build``.
"""

from __future__ import annotations

import ctypes as C
import threading
from pathlib import Path

LIB_PATH = Path(__file__).resolve().parent / "_lib" / "libmoerouter.so"

MOE_OK, MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_WORKSPACE = range(6)
MOE_DTYPE_FP32, MOE_DTYPE_BF16 = 0, 1
MOE_NUM_SCALARS = 7
SCALAR_NAMES = ("l_aux", "balance", "cv", "max_over_mean", "min_over_mean", "rank_cv", "rank_max_over_mean")

# Every symbol declared in include/moe_router.h, with (restype, argtypes).
_p, _i32, _i64, _f32, _f64, _sz = C.c_void_p, C.c_int32, C.c_int64, C.c_float, C.c_double, C.c_size_t
SIGNATURES = {
    "moe_router_workspace_size": (_sz, [_i64, _i32, _i32]),
    "moe_workspace_init": (_i32, [_p, _sz, _p]),
    "moe_get_device_status": (_i32, [_p, _p, C.POINTER(_i32)]),
    "moe_router_fwd": (_i32, [_p, _i32, _i64, _i32, _i32, _f32, _i32, _i32,
                              _p, _p, _p, _p, _p, _p, _p, _p, _sz, _p]),
    "moe_router_bwd": (_i32, [_p, _i32, _i64, _i32, _f32, _p, _f32, _p, _p]),
    "moe_dispatch_capacity": (_i64, [_i64, _i32, _i32, _f64]),
    "moe_dispatch": (_i32, [_p, _i64, _i32, _i32, _f64, _p, _p, _p, _p, _p, C.POINTER(_i64), _p, _sz, _p]),
    "moe_shard_capacity_base": (_i32, [_p, _i32, _i32, _i32, _p, _p]),
    "moe_dispatch_sharded": (_i32, [_p, _i64, _i32, _i32, _f64, _i64, _p, _p, _p, _p, _p, _p, C.POINTER(_i64),
                                    _p, _sz, _p]),
    "moe_router_step": (_i32, [_p, _i32, _i64, _i32, _i32, _f32, _i32, _i32, _f64, _f32,
                               _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _sz, _p]),
    "moe_router_step_ex": (_i32, [_p, _i32, _i64, _i32, _i32, _f32, _i32, _i32, _f64, _f32, _p, _f32, _p, _i32, _p,
                                  _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _sz, _p]),
    "moe_router_step_static": (_i32, [_p, _i32, _i64, _i32, _i32, _f32, _i32, _i32, _f64, _f32,
                                      _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p]),
    "moe_router_step_host_device_size": (_sz, [_i32, _i64, _i32, _i32, _i32]),
    "moe_router_step_host": (_i32, [_p, _i32, _i64, _i32, _i32, _f32, _i32, _i32, _f64, _f32,
                                    _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _sz, _p, _sz, _p, _p,
                                    _p]),
    "moe_router_fwd_ex": (_i32, [_p, _i32, _i64, _i32, _i32, _f32, _i32, _i32, _p, _i32, _f32, _p,
                                 _p, _p, _p, _p, _p, _p, _p, _p, _sz, _p]),
    "moe_router_bwd_full": (_i32, [_p, _i32, _i64, _i32, _i32, _f32, _p, _f32, _i32, _p, _p, _i32, _p, _p]),
    "moe_eplb_plan": (_i32, [_p, _i32, _i32, _i32, _i32, _i32, _i32, _p, _p, _p, _p]),
    "taot_match_batched": (_i32, [_p, _p, _i32, _i32, _i32, _i32, _i32, _p, _p, _p, _p]),
    "moe_router_combine": (_i32, [_p, _p, C.POINTER(_i64), _i32, _i32, _i32, _f32, _i32, _i32,
                                  _p, _p, _p, _p, _p, _p]),
    "taot_sinkhorn_batched": (_i32, [_p, _i32, _i32, _i32, _f32, _f32, _i32, _p, _p, _p, _p, _p]),
    "moe_set_wait_timeout_ns": (None, [C.c_uint64]),
    "moe_set_unreachable_barriers": (None, [_i32]),
    "moe_set_trace_buffer": (None, [_p, _i32]),
    "moe_status_string": (C.c_char_p, [_i32]),
    "moe_last_error": (C.c_char_p, []),
    "moe_abi_version": (_i32, []),
}

_lock = threading.Lock()
_lib: C.CDLL | None = None


class MoeRouterError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        super().__init__(f"{where}: status {status}: {detail}")
        self.status = status


def lib() -> C.CDLL:
    """The loaded library (loaded once; raises if it is not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not LIB_PATH.exists():
                raise RuntimeError(f"{LIB_PATH} is not built; run python -m moe_expert_routing_router_gb300.build")
            handle = C.CDLL(str(LIB_PATH))
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
        return _lib


def check(status: int, where: str) -> None:
    if status != MOE_OK:
        detail = lib().moe_last_error().decode(errors="replace")
        raise MoeRouterError(status, where, detail)
