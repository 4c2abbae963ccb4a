"""Builds the CUDA library in place: exact_attention_20_gb300/libfa_gb300.so.

One translation unit, one -gencode (sm_103a), compiled with nvcc; the result
links only the CUDA runtime (statically), so it loads on a machine without a
GPU (for symbol checks) and runs on a GB300.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB_NAME = "libfa_gb300.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
SOURCES = [os.path.join(PKG, "csrc", n) for n in ("fa_api.cu", "fa_noalloc.cu")]
DEPENDS = SOURCES + [
    os.path.join(PKG, "csrc", n)
    for n in ("fa_fwd_kernel.cuh", "sm103_ptx.cuh", "tma_host.h", "fa_internal.h")
] + [os.path.join(ROOT, "include", "fa_gb300.h")]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-std=c++17", "-lineinfo",
    "-shared", "-Xcompiler", "-fPIC",
    "-cudart", "static",
]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(s) <= t for s in DEPENDS)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB_PATH
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc(), *NVCC_FLAGS, "-I", os.path.join(ROOT, "include"), "-o", tmp, *SOURCES]
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
