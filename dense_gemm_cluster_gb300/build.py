"""Builds libdensegemm.so (the C-ABI CUDA library) in-tree with nvcc for sm_103a.

    python -m dense_gemm_cluster_gb300.build [--force]

The library goes to ``dense_gemm_cluster_gb300/_build/libdensegemm.so``. It
links the CUDA runtime statically and reaches the driver's tensor-map encoder
through ``cudaGetDriverEntryPointByVersion``, so it needs no ``-lcuda``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libdensegemm.so")
SOURCES = [os.path.join(CSRC, "gemm_host.cu"), os.path.join(CSRC, "host_io.cu"), os.path.join(CSRC, "tma_bench.cu"), os.path.join(CSRC, "stencil.cu"),
           os.path.join(CSRC, "attention.cu"), os.path.join(CSRC, "attention_host.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, "gemm_kernel.cuh"), os.path.join(CSRC, "ptx.cuh"),
                     os.path.join(CSRC, "gemm_internal.h"), os.path.join(CSRC, "host_env.h"),
                     os.path.join(INCLUDE, "densegemm.h"), os.path.join(INCLUDE, "tma_bench.h"),
                     os.path.join(INCLUDE, "stencil.h"), os.path.join(INCLUDE, "attention.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdensegemm.so")


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(p) > t for p in DEPENDS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compiles the library if it is missing or older than its sources; returns its path.

    Each translation unit compiles in its own nvcc process (in parallel), then one
    nvcc call links the shared library."""
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    tag = f"{os.getpid()}"
    flags = [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE]
    if verbose:
        flags.insert(0, "-Xptxas=-v")
    objs, procs = [], []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, os.path.basename(src) + f".{tag}.o")
        cmd = [nvcc(), *flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((subprocess.Popen(cmd), cmd))
        objs.append(obj)
    failed = [cmd for proc, cmd in procs if proc.wait() != 0]
    try:
        if failed:
            raise subprocess.CalledProcessError(1, failed[0])
        tmp = LIB_PATH + f".{tag}.tmp"
        subprocess.run([nvcc(), *ARCH, "-shared", *objs, "-o", tmp], check=True)
        os.replace(tmp, LIB_PATH)
    finally:
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
