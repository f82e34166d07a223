"""CPU oracle for the dense contraction -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package. The library under
``dense_gemm_cluster_gb300`` never imports it and shares no code with it.

The arithmetic lives in ``gemm_oracle.c`` (plain C, fp64 accumulation, OpenMP
over output rows); this module compiles it with gcc on first use and wraps it
with numpy. Inputs are bf16 bit patterns (``numpy.uint16``) laid out as
row-major (``"row"``) or column-major (``"col"``) buffers with a leading
dimension, exactly the bytes the GPU path receives.

Every function here is pinned by ``tests/test_oracle_pins.py`` against closed
forms (identity, permutation, all-ones, rank-1, alpha/beta special cases) and
against exact rational brute force on tiny shapes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_LAYOUT = {"row": 0, "col": 1}


def build(force: bool = False) -> str:
    """Compile gemm_oracle.c into oracle/_build/liboracle.so (gcc, OpenMP, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
               "-std=c11", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, i32, f64, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
            lib.oracle_gemm.argtypes = [i64, i64, i64, vp, i64, i32, vp, i64, i32,
                                        vp, i64, i32, i32, f64, f64, vp, i64]
            lib.oracle_gemm.restype = i32
            lib.oracle_gemm_entries.argtypes = [i64, vp, vp, i64, vp, i64, i32, vp, i64, i32,
                                                vp, i64, i32, i32, f64, f64, vp]
            lib.oracle_gemm_entries.restype = i32
            lib.oracle_attention_scores.argtypes = [i64, i64, i64, i64, vp, i64, i64, vp, i64, i64, vp]
            lib.oracle_attention_scores.restype = i32
            lib.oracle_attention_forward.argtypes = [i64, i64, i64, i64, i64, vp, vp, vp, f64, i32, vp, vp]
            lib.oracle_attention_forward.restype = i32
            lib.oracle_stencil_1d.argtypes = [i64, vp, vp]
            lib.oracle_stencil_1d.restype = i32
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = i32
            _lib = lib
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    return int(_load().oracle_num_threads())


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c_args(C_in, ldc, layout_c):
    if C_in is None:
        return None, 0, 0, 0
    C_in = np.ascontiguousarray(C_in)
    if C_in.dtype == np.uint16:
        dc = 0
    elif C_in.dtype == np.float32:
        dc = 1
    else:
        raise TypeError("C_in must hold bf16 bits (uint16) or float32")
    return C_in, int(ldc), _LAYOUT[layout_c], dc


def gemm(M, N, K, A, lda, layout_a, B, ldb, layout_b, alpha=1.0, beta=0.0,
         C_in=None, ldc=0, layout_c="row"):
    """C_ref = alpha * A @ B + beta * C_in as a row-major (M, N) float64 array."""
    A = np.ascontiguousarray(A, dtype=np.uint16)
    B = np.ascontiguousarray(B, dtype=np.uint16)
    C_in, ldc, lc, dc = _c_args(C_in if beta != 0.0 else None, ldc, layout_c)
    out = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_gemm(M, N, K, _ptr(A), lda, _LAYOUT[layout_a], _ptr(B), ldb,
                             _LAYOUT[layout_b], _ptr(C_in), ldc, lc, dc,
                             float(alpha), float(beta), _ptr(out), N)
    if rc != 0:
        raise ValueError(f"oracle_gemm rejected its arguments (code {rc})")
    return out


def gemm_entries(rows, cols, K, A, lda, layout_a, B, ldb, layout_b, alpha=1.0, beta=0.0,
                 C_in=None, ldc=0, layout_c="row"):
    """The same definition evaluated only at positions (rows[t], cols[t])."""
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    A = np.ascontiguousarray(A, dtype=np.uint16)
    B = np.ascontiguousarray(B, dtype=np.uint16)
    C_in, ldc, lc, dc = _c_args(C_in if beta != 0.0 else None, ldc, layout_c)
    out = np.empty(rows.shape[0], dtype=np.float64)
    rc = _load().oracle_gemm_entries(rows.shape[0], _ptr(rows), _ptr(cols), K, _ptr(A), lda,
                                     _LAYOUT[layout_a], _ptr(B), ldb, _LAYOUT[layout_b],
                                     _ptr(C_in), ldc, lc, dc, float(alpha), float(beta), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_gemm_entries rejected its arguments (code {rc})")
    return out


def attention_scores(Q, Kmat):
    """S[b] = Q[b] @ K[b]^T for Q (batch, sq, d) and K (batch, sk, d) bf16 bits; float64 out."""
    Q = np.ascontiguousarray(Q, dtype=np.uint16)
    Kmat = np.ascontiguousarray(Kmat, dtype=np.uint16)
    batch, sq, d = Q.shape
    sk = Kmat.shape[1]
    if Kmat.shape[0] != batch or Kmat.shape[2] != d:
        raise ValueError("Q and K disagree on batch or head dimension")
    out = np.empty((batch, sq, sk), dtype=np.float64)
    rc = _load().oracle_attention_scores(batch, sq, sk, d, _ptr(Q), d, sq * d, _ptr(Kmat), d,
                                         sk * d, _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_attention_scores rejected its arguments (code {rc})")
    return out


def stencil_1d(x):
    """y[i] = 0.25 x[i-1] + 0.5 x[i] + 0.25 x[i+1] (x = 0 outside the array), float64 out."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape[0], dtype=np.float64)
    rc = _load().oracle_stencil_1d(x.shape[0], _ptr(x), _ptr(y))
    if rc != 0:
        raise ValueError(f"oracle_stencil_1d rejected its arguments (code {rc})")
    return y


def attention_forward(Q, Kmat, V, scale=None, with_lse=False, causal=False):
    """O = softmax(scale Q K^T) V per batch for bf16-bit arrays Q (b, sq, d), K (b, sk, d),
    V (b, sk, dv); float64 out (and the row log-sum-exp when with_lse). scale defaults to 1/sqrt(d).
    causal: query i attends keys 0..i only (the others take no part in its softmax)."""
    Q = np.ascontiguousarray(Q, dtype=np.uint16)
    Kmat = np.ascontiguousarray(Kmat, dtype=np.uint16)
    V = np.ascontiguousarray(V, dtype=np.uint16)
    b, sq, d = Q.shape
    sk, dv = V.shape[1], V.shape[2]
    if Kmat.shape != (b, sk, d) or V.shape[0] != b:
        raise ValueError("Q, K, V disagree on batch, key count or head dimension")
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    O = np.empty((b, sq, dv), dtype=np.float64)
    lse = np.empty((b, sq), dtype=np.float64)
    rc = _load().oracle_attention_forward(b, sq, sk, d, dv, _ptr(Q), _ptr(Kmat), _ptr(V), float(scale),
                                          1 if causal else 0, _ptr(O), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_attention_forward rejected its arguments (code {rc})")
    return (O, lse) if with_lse else O
