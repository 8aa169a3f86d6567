"""Compile the CUDA library (csrc/*.cu) into an in-tree shared object.

Each translation unit is compiled by its own nvcc process (in parallel) with
one -gencode (sm_103a) and no fast-math, then nvcc links the objects.  The
result lives at precision_quantization_token_gb300/_build/libtk_cast.so and
is loaded by the ctypes binding in __init__.py.
"""
from __future__ import annotations

import glob
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libtk_cast.so")

ARCH = "-gencode=arch=compute_103a,code=sm_103a"
COMPILE_FLAGS = [
    ARCH, "-O3", "-lineinfo", "-std=c++17",
    "-ftz=false", "-prec-div=true", "-prec-sqrt=true", "-fmad=false",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "-Xcompiler", "-Wall", "-Xcompiler", "-Wextra", f"-I{INCLUDE}",
]
# One-shot form (compile and link every source in one nvcc call).
NVCC_FLAGS = COMPILE_FLAGS + ["-shared"]


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + \
        sorted(glob.glob(os.path.join(INCLUDE, "*.h")))


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(s) <= t for s in _inputs())


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def build(force: bool = False, verbose: bool = False,
          extra: list[str] | None = None) -> str:
    """Build libtk_cast.so (skipped when it is newer than every source)."""
    if not force and not extra and up_to_date():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    tag = f"{os.getpid()}.tmp"
    objs, procs = [], []
    for src in sources():
        obj = os.path.join(BUILD_DIR, os.path.basename(src) + f".{tag}.o")
        cmd = [nvcc(), *COMPILE_FLAGS, *(extra or []), "-c", "-o", obj, src]
        if verbose:
            print(" ".join(cmd), flush=True)
        objs.append(obj)
        procs.append((cmd, subprocess.Popen(cmd)))
    failed = [cmd for cmd, p in procs if p.wait() != 0]
    try:
        if failed:
            raise subprocess.CalledProcessError(1, failed[0])
        tmp = LIB_PATH + f".{tag}"
        subprocess.run([nvcc(), ARCH, "-shared", "-o", tmp, *objs], check=True)
        os.replace(tmp, LIB_PATH)
    finally:
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
    return LIB_PATH


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True,
                extra=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None))
