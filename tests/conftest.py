import sys
from pathlib import Path

ROOT = Path(__file__).resolve().parents[1]
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))
TESTS = Path(__file__).resolve().parent
if str(TESTS) not in sys.path:
    sys.path.insert(0, str(TESTS))


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")

import pytest  # noqa: E402


def _lib_is_stale() -> bool:
    from moe_expert_routing_router_gb300 import build as b
    lib = b.LIBDIR / b.LIBNAME
    if not lib.exists():
        return True
    newest = max(p.stat().st_mtime for p in list(b.CSRC.iterdir()) + [b.INCLUDE / "moe_router.h"])
    return lib.stat().st_mtime < newest


@pytest.fixture(scope="session")
def native_lib():
    """The built C-ABI library (built in-tree first when missing or older than its sources)."""
    from moe_expert_routing_router_gb300 import _native, build
    if _lib_is_stale():
        build.build(quiet=True)
    return _native.lib()
