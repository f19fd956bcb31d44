"""Builds libfp8q.so (the C-ABI CUDA library) in-tree with nvcc for sm_103a.

Each translation unit compiles in parallel; the result lands in
``fp8_absmax_reduce_gb300/_lib/libfp8q.so``.  Run ``python -m
fp8_absmax_reduce_gb300.build`` or call :func:`build`.
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
OUT_DIR = os.path.join(PKG, "_lib")
OBJ_DIR = os.path.join(OUT_DIR, "obj")
LIB = os.path.join(OUT_DIR, "libfp8q.so")
SOURCES = ["fp8q_api.cu", "fp8q_quant.cu", "fp8q_gemm.cu", "fp8q_attn.cu", "fp8q_noalloc.cu", "fp8q_mx.cu"]
HEADERS = ["fp8q_common.cuh", "fp8q_internal.h"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfp8q.so")
    return cand


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, verbose_ptxas: bool) -> str:
    obj = os.path.join(OBJ_DIR, os.path.splitext(src)[0] + ".o")
    deps = [os.path.join(CSRC, src), os.path.join(INCLUDE, "fp8q.h")] + [os.path.join(CSRC, h) for h in HEADERS]
    if _stale(obj, deps) or verbose_ptxas:
        cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose_ptxas:
            cmd += ["-Xptxas", "-v"]
        subprocess.run(cmd, check=True)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile (when sources changed) and link libfp8q.so; return its path."""
    os.makedirs(OBJ_DIR, exist_ok=True)
    if force:
        for f in os.listdir(OBJ_DIR):
            os.remove(os.path.join(OBJ_DIR, f))
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas), SOURCES))
    if force or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs], check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
