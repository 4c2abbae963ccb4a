"""Builds the CUDA library in place: exact_attention_20_gb300/libfa_gb300.so.

A few translation units, compiled in parallel by nvcc with one -gencode
(sm_103a) and linked into one shared library; the result links only the CUDA
runtime (statically), so it loads on a machine without a GPU (for symbol
checks) and runs on a GB300.
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
SOURCES = [os.path.join(PKG, "csrc", n) for n in ("fa_api.cu", "fa_noalloc.cu", "fa_bwd.cu", "fa_fp8.cu")]
DEPENDS = SOURCES + [
    os.path.join(PKG, "csrc", n)
    for n in ("fa_fwd_kernel.cuh", "fa_bwd_kernel.cuh", "fa_fp8_quant.cuh", "fa_decode.cuh", "sm103_ptx.cuh", "tma_host.h",
              "fa_internal.h")
] + [os.path.join(ROOT, "include", "fa_gb300.h")]

COMPILE_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-std=c++17", "-lineinfo",
    "-Xcompiler", "-fPIC",
]
LINK_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-cudart", "static"]


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
    objs, procs = [], []
    for src in SOURCES:
        obj = os.path.join(PKG, "_build", os.path.basename(src) + ".o")
        os.makedirs(os.path.dirname(obj), exist_ok=True)
        cmd = [nvcc(), *COMPILE_FLAGS, "-I", os.path.join(ROOT, "include"), "-c", "-o", obj, src]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((cmd, subprocess.Popen(cmd)))
        objs.append(obj)
    for cmd, proc in procs:
        if proc.wait() != 0:
            raise subprocess.CalledProcessError(proc.returncode, cmd)
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc(), *LINK_FLAGS, "-o", tmp, *objs]
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
