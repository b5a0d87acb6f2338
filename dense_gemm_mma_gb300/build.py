"""Build libdgemm_gb300.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel into ``_build/`` and linked
into ``dense_gemm_mma_gb300/libdgemm_gb300.so`` with the CUDA runtime linked
statically, so the library loads on a machine without a GPU (the entry points
then report GEMM_ERR_NO_DEVICE).  ``build(debug=True)`` compiles the same
sources with DG_DEBUG into ``_build_debug/`` and
``dense_gemm_mma_gb300/libdgemm_gb300_debug.so``: every kernel then checks its
plain global accesses and TMA coordinates on the device and reports a failed
check through the plan's error word (include/gemm.h, gemm_debug_build).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libdgemm_gb300.so")
LIB_DEBUG = os.path.join(PKG, "libdgemm_gb300_debug.so")

SOURCES = [
    "api.cpp",
    "gemv.cu",
    "gemm_tc_dispatch.cu",
    "gemm_tc_bn64.cu",
    "gemm_tc_bn128.cu",
    "gemm_tc_bn256.cu",
    "gemm_tc_tf32_bn64.cu",
    "gemm_tc_tf32_bn128.cu",
    "gemm_tc_tf32_bn256.cu",
    "noalloc.cu",
]
HEADERS = ["ptx.cuh", "kernels.h", "gemm_tc.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newest_input() -> float:
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "gemm.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    lib = LIB_DEBUG if debug else LIB
    build_dir = BUILD + "_debug" if debug else BUILD
    flags = FLAGS + (["-DDG_DEBUG"] if debug else [])
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _newest_input():
        return lib
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *ARCH, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose and src.endswith(".cu"):
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
