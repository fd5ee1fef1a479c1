"""Builds the in-tree C-ABI library ``_lib/libmoerouter.so`` for sm_103a.

Each CUDA translation unit is compiled by its own nvcc process (in parallel),
then the objects are linked into one shared library with the CUDA runtime
linked statically.  Run as ``python -m moe_expert_routing_router_gb300.build``.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys
import time
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
LIBDIR = PKG / "_lib"
LIBNAME = "libmoerouter.so"
ARCH = "-gencode=arch=compute_103a,code=sm_103a"

SOURCES = ["router_bf16_staged.cu", "router_bf16_direct.cu", "router_fp32_staged.cu", "router_fp32_direct.cu",
           "router_step_ext_bf16_staged.cu", "router_step_ext_bf16_direct.cu", "router_step_ext_fp32_staged.cu",
           "router_step_ext_fp32_direct.cu",
           "router_dispatch.cu", "router_ext_bf16.cu", "router_ext_fp32.cu", "router_combine.cu", "sinkhorn.cu", "taot_match.cu", "eplb.cu", "abi.cu"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found")


def common_flags(verbose_ptxas: bool) -> list[str]:
    flags = [ARCH, "-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr",
             "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
             f"-I{INCLUDE}", f"-I{CSRC}"]
    if verbose_ptxas:
        flags += ["-Xptxas", "-v"]
    return flags


def _compile(src: Path, obj: Path, verbose_ptxas: bool) -> tuple[str, float, str]:
    t0 = time.time()
    cmd = [nvcc(), *common_flags(verbose_ptxas), "-c", str(src), "-o", str(obj)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src.name}:\n{r.stdout}\n{r.stderr}")
    return src.name, time.time() - t0, r.stderr


def build(verbose_ptxas: bool = False, jobs: int | None = None, quiet: bool = False) -> Path:
    """Compiles every translation unit and links the library; returns its path."""
    LIBDIR.mkdir(exist_ok=True)
    objdir = LIBDIR / "obj"
    objdir.mkdir(exist_ok=True)
    srcs = [CSRC / s for s in SOURCES]
    objs = [objdir / (s.stem + ".o") for s in srcs]
    jobs = jobs or min(len(srcs), os.cpu_count() or 1)
    t0 = time.time()
    logs = []
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        futs = [ex.submit(_compile, s, o, verbose_ptxas) for s, o in zip(srcs, objs)]
        for fu in futs:
            logs.append(fu.result())
    out = LIBDIR / LIBNAME
    tmp = LIBDIR / (LIBNAME + ".tmp")
    cmd = [nvcc(), ARCH, "-shared", "-o", str(tmp), *map(str, objs), "-Xcompiler", "-fPIC"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    if not quiet:
        for name, dt, err in logs:
            print(f"  {name}: {dt:.1f}s")
            if verbose_ptxas and err:
                print(err)
        print(f"built {out} in {time.time() - t0:.1f}s")
    return out


if __name__ == "__main__":
    build(verbose_ptxas="-v" in sys.argv)
