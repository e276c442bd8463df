"""Build step for the CUDA library ``libfa.so`` (nvcc, sm_103a only).

The library is built in-tree next to this file so the tests and the benchmark
load the copy compiled from this checkout.  Two translation units (forward and
backward), one ``-gencode``: a build takes a few seconds.
"""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libfa.so")
SOURCES = [os.path.join(CSRC, "fa_fwd.cu"), os.path.join(CSRC, "fa_bwd.cu")]
DEPS = SOURCES + [os.path.join(CSRC, "sm103_ptx.cuh"), os.path.join(CSRC, "fa_internal.h"),
                  os.path.join(INCLUDE, "fa.h")]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo", "-O3", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libfa.so unless it is newer than every source; return its path."""
    if not force and up_to_date():
        return LIB
    tmp = LIB + ".tmp"
    cmd = [nvcc(), *NVCC_FLAGS, "-I" + INCLUDE, "-o", tmp, *SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
