"""The C-ABI library on the host: it loads, exports every declared entry point,
and rejects bad arguments before touching the GPU (no compute calls here)."""

import ctypes as C
import re
import subprocess
from pathlib import Path

import pytest

from moe_expert_routing_router_gb300 import _native

HEADER = Path(__file__).resolve().parents[1] / "include" / "moe_router.h"


def declared_functions() -> list[str]:
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^(?:MOE_API )?[a-z_][\w \*]*?\b((?:moe|taot)_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("moe_router_fwd", "moe_router_bwd", "moe_dispatch", "taot_sinkhorn_batched", "moe_router_step"):
        assert want in names


def test_library_exports_every_declared_symbol(native_lib):
    names = declared_functions()
    for n in names:
        assert hasattr(native_lib, n), n
    assert set(names) == set(_native.SIGNATURES), "ctypes signatures must cover exactly the header"
    out = subprocess.run(["nm", "-D", "--defined-only", str(_native.LIB_PATH)], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if ln.strip()}
    assert set(names) <= exported
    assert not any(s.startswith("_ZN3moe") for s in exported), "internal symbols must stay hidden"


def test_abi_version(native_lib):
    assert native_lib.moe_abi_version() == 2


def test_capacity_worked_example_through_the_abi(native_lib):
    # 1024 tokens, 8 experts, factor 1.25 -> 160 (MoE article, section 4.5)
    assert native_lib.moe_dispatch_capacity(1024, 8, 1, 1.25) == 160
    assert native_lib.moe_dispatch_capacity(65536, 64, 2, 1.25) == 2560
    assert native_lib.moe_dispatch_capacity(10, 4, 1, 1.0) == 3
    assert native_lib.moe_dispatch_capacity(0, 4, 1, 1.0) == -1
    assert native_lib.moe_dispatch_capacity(10, 4, 1, 0.0) == -1


def test_workspace_size(native_lib):
    assert native_lib.moe_router_workspace_size(262144, 384, 6) > 0
    assert native_lib.moe_router_workspace_size(0, 8, 1) == 0
    assert native_lib.moe_router_workspace_size(16, 2000, 1) == 0
    assert native_lib.moe_router_workspace_size(16, 8, 9) == 0


FAKE = 0x10000  # never dereferenced: each call below fails its host-side checks first


@pytest.mark.parametrize("T,E,k,dt,status", [
    (0, 8, 1, 1, _native.MOE_ERR_INVALID),
    (16, 0, 1, 1, _native.MOE_ERR_INVALID),
    (16, 1025, 1, 1, _native.MOE_ERR_INVALID),
    (16, 8, 0, 1, _native.MOE_ERR_INVALID),
    (16, 8, 9, 1, _native.MOE_ERR_INVALID),
    (16, 4, 5, 1, _native.MOE_ERR_INVALID),
    (2 ** 30, 8, 2, 1, _native.MOE_ERR_INVALID),
    (16, 8, 1, 7, _native.MOE_ERR_UNSUPPORTED),
])
def test_router_fwd_rejects_bad_sizes(native_lib, T, E, k, dt, status):
    st = native_lib.moe_router_fwd(FAKE, dt, T, E, k, 0.01, -1, 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None,
                                   FAKE, 1 << 30, None)
    assert st == status
    assert native_lib.moe_last_error()


def test_router_fwd_rejects_bad_arguments(native_lib):
    f = native_lib.moe_router_fwd
    ok = dict(alpha=0.01, renorm=-1, n_ranks=0)
    assert f(None, 1, 16, 8, 1, 0.01, -1, 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 1 << 30, None) == 1
    assert f(FAKE, 1, 16, 8, 1, -1.0, -1, 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 1 << 30, None) == 1
    assert f(FAKE, 1, 16, 8, 1, 0.01, 2, 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 1 << 30, None) == 1
    assert f(FAKE, 1, 16, 8, 1, 0.01, -1, 3, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, None) == 1
    assert f(FAKE, 1, 16, 8, 1, 0.01, -1, 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 1 << 30, None) == 1
    assert f(FAKE, 1, 16, 8, 1, 0.01, -1, 0, FAKE, None, FAKE, FAKE, FAKE, FAKE, None, FAKE, 1 << 30, None) == 1
    assert f(FAKE, 1, 16, 8, 1, 0.01, -1, 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE + 8, 1 << 30, None) == 1
    assert f(FAKE, 1, 16, 8, 1, 0.01, -1, 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 64, None) == 5
    assert f(FAKE + 1, 1, 16, 8, 1, 0.01, -1, 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 1 << 30, None) == 1
    del ok


def test_dispatch_and_step_reject_bad_arguments(native_lib):
    cap = C.c_int64(0)
    d = native_lib.moe_dispatch
    assert d(FAKE, 16, 8, 2, 0.0, FAKE, FAKE, FAKE, FAKE, FAKE, C.byref(cap), FAKE, 1 << 30, None) == 1
    assert d(FAKE, 16, 8, 2, 1.0, None, FAKE, FAKE, FAKE, FAKE, C.byref(cap), FAKE, 1 << 30, None) == 1
    assert d(FAKE, 16, 8, 2, 1.0, FAKE, FAKE, FAKE, FAKE, FAKE, C.byref(cap), FAKE, 8, None) == 5
    s = native_lib.moe_router_step
    args = [FAKE, 1, 16, 8, 2, 0.01, -1, 0, 1.25, 1.0] + [FAKE] * 6 + [None] + [FAKE] * 6 + [FAKE, 1 << 30, None]
    bad = list(args)
    bad[8] = -1.0
    assert s(*bad) == 1
    bad = list(args)
    bad[22] = None                                   # dlogits
    assert s(*bad) == 1
    bad = list(args)
    bad[22] = FAKE + 2                               # misaligned dlogits
    assert s(*bad) == 1


def test_sharded_dispatch_rejects_bad_arguments(native_lib):
    cap = C.c_int64(0)
    d = native_lib.moe_dispatch_sharded
    args = [FAKE, 16, 8, 2, 1.0, 64, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, C.byref(cap), FAKE, 1 << 30, None]
    for pos, val in [(6, None), (6, FAKE + 2), (5, 15), (5, 2 ** 30), (4, 0.0), (7, None), (0, None), (2, 0)]:
        bad = list(args)
        bad[pos] = val
        assert d(*bad) == 1, (pos, val)
    bad = list(args)
    bad[14] = 8                                       # workspace too small
    assert d(*bad) == 5
    b = native_lib.moe_shard_capacity_base
    args = [FAKE, 4, 8, 1, FAKE, None]
    for pos, val in [(0, None), (4, None), (1, 0), (1, 65), (2, 0), (2, 1025), (3, -1), (3, 4), (4, FAKE + 2)]:
        bad = list(args)
        bad[pos] = val
        assert b(*bad) == 1, (pos, val)


def test_bwd_and_sinkhorn_reject_bad_arguments(native_lib):
    b = native_lib.moe_router_bwd
    assert b(FAKE, 1, 16, 8, 0.01, None, 1.0, FAKE, None) == 1
    assert b(FAKE, 1, 16, 8, float("nan"), FAKE, 1.0, FAKE, None) == 1
    assert b(FAKE, 1, 0, 8, 0.01, FAKE, 1.0, FAKE, None) == 1
    sk = native_lib.taot_sinkhorn_batched
    assert sk(FAKE, 4, 65, 8, 10.0, 0.0, 50, FAKE, FAKE, None, FAKE, None) == 1
    assert sk(FAKE, 4, 64, 7, 10.0, 0.0, 50, FAKE, FAKE, None, FAKE, None) == 1
    assert sk(FAKE, 4, 64, 8, 0.0, 0.0, 50, FAKE, FAKE, None, FAKE, None) == 1
    assert sk(FAKE, 0, 64, 8, 10.0, 0.0, 50, FAKE, FAKE, None, FAKE, None) == 1
    assert sk(FAKE, 4, 64, 8, 10.0, 0.0, -1, FAKE, FAKE, None, FAKE, None) == 1
    assert sk(None, 4, 64, 8, 10.0, 0.0, 50, FAKE, FAKE, None, FAKE, None) == 1


def test_status_strings(native_lib):
    for s in range(6):
        assert native_lib.moe_status_string(s)


def test_fwd_ex_and_bwd_full_reject_bad_arguments(native_lib):
    fx = native_lib.moe_router_fwd_ex
    args = [FAKE, 1, 16, 8, 2, 0.01, -1, 0, None, 0, 0.0, None] + [FAKE] * 6 + [None, FAKE, 1 << 30, None]
    for pos, val, want in [(2, 0, 1), (4, 9, 1), (1, 7, 2), (5, -1.0, 1), (6, 3, 1), (7, 3, 1),
                           (10, float("inf"), 1), (8, FAKE + 2, 1), (11, FAKE + 1, 1), (13, None, 1),
                           (19, FAKE + 8, 1), (20, 64, 5)]:
        bad = list(args)
        bad[pos] = val
        assert fx(*bad) == want, (pos, val)
        assert native_lib.moe_last_error()
    bf = native_lib.moe_router_bwd_full
    args = [FAKE, 1, 16, 8, 2, 0.01, FAKE, 1.0, 0, FAKE, FAKE, -1, FAKE, None]
    for pos, val, want in [(6, None, 1), (12, None, 1), (5, float("nan"), 1), (7, float("inf"), 1),
                           (11, 2, 1), (9, None, 1), (12, FAKE + 2, 1), (10, FAKE + 1, 1), (4, 0, 1)]:
        bad = list(args)
        bad[pos] = val
        assert bf(*bad) == want, (pos, val)
    bad = list(args)
    bad[10] = None                                   # no dgate: masked P still needs idx
    bad[8] = 1
    bad[9] = None
    assert bf(*bad) == 1


def test_eplb_rejects_bad_arguments(native_lib):
    f = native_lib.moe_eplb_plan
    args = [FAKE, 4, 48, 64, 16, 4, 8, FAKE, FAKE, FAKE, None]
    for pos, val in [(0, None), (1, 0), (2, 0), (2, 1025), (3, 40), (3, 65), (3, 8192), (4, 0), (4, 257),
                     (5, 3), (5, 0), (6, 5), (6, -1), (7, None), (9, FAKE + 2)]:
        bad = list(args)
        bad[pos] = val
        assert f(*bad) == 1, (pos, val)
        assert native_lib.moe_last_error()


def test_taot_match_rejects_bad_arguments(native_lib):
    f = native_lib.taot_match_batched
    args = [FAKE, FAKE, 4, 384, 64, 8, 4, FAKE, FAKE, FAKE, None]
    for pos, val in [(0, None), (1, None), (2, 0), (3, 0), (3, 1025), (4, 0), (4, 65), (4, 5), (5, 3), (6, -1),
                     (6, 17), (9, None), (7, FAKE + 2), (7, None), (8, None)]:
        bad = list(args)
        bad[pos] = val
        assert f(*bad) == 1, (pos, val)


def test_combine_rejects_bad_arguments(native_lib):
    f = native_lib.moe_router_combine
    T2 = (C.c_int64 * 2)(100, 200)
    bad_T = (C.c_int64 * 2)(-1, 200)
    args = [FAKE, FAKE, T2, 2, 8, 2, 0.01, 0, 0, FAKE, FAKE, FAKE, FAKE, None, None]
    for pos, val in [(0, None), (2, None), (3, 0), (3, 65), (4, 0), (5, 9), (6, -1.0), (7, 3), (9, None),
                     (12, None), (2, bad_T), (10, FAKE + 2)]:
        bad = list(args)
        bad[pos] = val
        assert f(*bad) == 1, (pos, val)
    bad = list(args)
    bad[7] = 4                                        # rank loads requested without a buffer
    assert f(*bad) == 1


def test_host_step_staging_size_and_argument_checks(native_lib):
    # logits 256 x 64 bf16 (32 KiB); idx, gate, perm, slot 2 KiB each; counts, f, P, scalars, kept, n_dropped one
    # 256-byte region each; offsets (65 ints) two; 64 KiB of dlogits: every region 256-byte aligned
    T, E, k = 256, 64, 2
    want = 32768 + 4 * 2048 + 6 * 256 + 512 + 65536
    assert native_lib.moe_router_step_host_device_size(1, T, E, k, 0) == want
    assert native_lib.moe_router_step_host_device_size(1, T, E, k, 8) == want + 256
    assert native_lib.moe_router_step_host_device_size(0, T, E, k, 0) == want + 32768
    assert native_lib.moe_router_step_host_device_size(1, 0, E, k, 0) == 0
    host = [FAKE] * 13
    args = [FAKE, 1, T, E, k, 0.01, -1, 0, 1.25, 1.0]
    # a NULL host output
    st = native_lib.moe_router_step_host(*args, *([None] + host[1:]), FAKE, want, FAKE, 1 << 20, None, None, None)
    assert st == _native.MOE_ERR_INVALID
    # a staging buffer one byte short
    st = native_lib.moe_router_step_host(*args, *host, FAKE, want - 1, FAKE, 1 << 20, None, None, None)
    assert st == _native.MOE_ERR_WORKSPACE
    # a misaligned staging buffer
    st = native_lib.moe_router_step_host(*args, *host, FAKE + 16, want, FAKE, 1 << 20, None, None, None)
    assert st == _native.MOE_ERR_INVALID
    # an unknown dtype
    args_bad = [FAKE, 7, T, E, k, 0.01, -1, 0, 1.25, 1.0]
    st = native_lib.moe_router_step_host(*args_bad, *host, FAKE, want, FAKE, 1 << 20, None, None, None)
    assert st == _native.MOE_ERR_UNSUPPORTED
