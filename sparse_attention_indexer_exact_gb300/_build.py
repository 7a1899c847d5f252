"""Build step for libgvrtopk.so (the CUDA kernels and their C ABI), in-tree, for sm_103a.

``build_library()`` runs nvcc once over ``csrc/gvr_topk.cu`` and writes
``libgvrtopk.so`` beside this file; it rebuilds only when a source is newer
than the library.  No CMake, no torch extension machinery: the library is a
plain shared object with an ``extern "C"`` interface (``include/gvr_topk.h``).
"""
from __future__ import annotations

import glob
import os
import subprocess
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG, "libgvrtopk.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
_lock = threading.Lock()


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return "nvcc"


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                  glob.glob(os.path.join(INCLUDE, "*.h")))


def nvcc_command(out: str = LIB_PATH, extra=()) -> list[str]:
    return [nvcc_path(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
            "-I", INCLUDE, *extra, os.path.join(CSRC, "gvr_topk.cu"), "-o", out]


def stale(out: str = LIB_PATH) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(s) > t for s in sources())


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Compile libgvrtopk.so for sm_103a if it is missing or older than its sources."""
    with _lock:
        if force or stale():
            cmd = nvcc_command(extra=["-Xptxas", "-v"] if verbose else [])
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
            if verbose:
                print(r.stdout + r.stderr)
    return LIB_PATH


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))
