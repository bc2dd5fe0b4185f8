"""Compile the CUDA library ``libhcread.so`` in-tree for sm_103a.

Two translation units (the read's host C ABI + kernels, and the Q2_0
matrix-vector product's), one ``-gencode``:
``nvcc -gencode arch=compute_103a,code=sm_103a``.  The library links the
CUDA runtime statically, so it only needs the driver at run time.
"""

from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libhcread.so")
SOURCES = [os.path.join(CSRC, "hc_read.cu"), os.path.join(CSRC, "hc_q2.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in (
    "hc_kernels.cuh", "hc_kernels_tc.cuh", "hc_kernels_umma.cuh", "hc_kernels_wide.cuh", "hc_window.cuh",
    "hc_ptx.cuh")] + [
    os.path.join(INCLUDE, "hc_read.h"), os.path.join(INCLUDE, "hc_q2.h")]

NVCC_FLAGS = [
    "-O3", "-std=c++17", "-lineinfo",
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "-shared",
]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libhcread.so")


def compile_cmd(out: str = LIB, extra: list[str] | None = None) -> list[str]:
    return [nvcc(), *NVCC_FLAGS, *(extra or []), f"-I{INCLUDE}", "-o", out, *SOURCES]


def stale(out: str = LIB) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(p) > t for p in DEPS)


def build(out: str = LIB, force: bool = False) -> str:
    if force or stale(out):
        subprocess.run(compile_cmd(out), check=True)
    return out
