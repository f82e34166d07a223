"""Seeded synthetic inputs, shared by the CUDA path's tests/bench and by the oracle.

This module holds no arithmetic of the contraction itself. It turns a seed into
bf16 bit patterns (``numpy.uint16``) with the distributions the workloads name:

* ``splitmix64``: the counter-based generator of Steele, Lea and Flood
  ("Fast splittable pseudorandom number generators", OOPSLA 2014). Output i of
  the stream with seed s is ``mix(s + (i + 1) * 0x9E3779B97F4A7C15)``.
* uniform in [0, 1): the top 53 bits of each 64-bit output times 2**-53.
* N(0, 1): the Box-Muller transform on consecutive uniform pairs
  (u1, u2) -> sqrt(-2 ln(1 - u1)) * (cos 2 pi u2, sin 2 pi u2).
* U(-1, 1): 2u - 1.
* bf16: the float64 value is rounded to float32 (round-to-nearest-even) and
  then to bf16 (round-to-nearest-even on the 16 dropped bits).

Operand streams use seed+0 for A (or Q), seed+1 for B (or K) and seed+2 for
C_in. Both sides receive the same bytes; neither computes them differently.
"""
from __future__ import annotations

import numpy as np

GOLDEN_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

STREAM_A = 0
STREAM_B = 1
STREAM_C = 2


def splitmix64(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """Outputs ``offset .. offset+n-1`` of the splitmix64 stream started at ``seed``."""
    out = np.empty(n, dtype=np.uint64)
    s = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
    with np.errstate(over="ignore"):
        for lo in range(0, n, _CHUNK):
            hi = min(n, lo + _CHUNK)
            idx = np.arange(offset + lo + 1, offset + hi + 1, dtype=np.uint64)
            z = s + idx * GOLDEN_GAMMA
            z = (z ^ (z >> np.uint64(30))) * _M1
            z = (z ^ (z >> np.uint64(27))) * _M2
            out[lo:hi] = z ^ (z >> np.uint64(31))
    return out


def uniform01(seed: int, n: int) -> np.ndarray:
    """n doubles in [0, 1) from the top 53 bits of each splitmix64 output."""
    return (splitmix64(seed, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, n: int) -> np.ndarray:
    """n N(0,1) doubles by Box-Muller over consecutive uniform pairs."""
    pairs = (n + 1) // 2
    out = np.empty(2 * pairs, dtype=np.float64)
    step = _CHUNK // 2
    for p0 in range(0, pairs, step):
        p1 = min(pairs, p0 + step)
        u = (splitmix64(seed, 2 * (p1 - p0), offset=2 * p0) >> np.uint64(11)).astype(np.float64)
        u *= 2.0 ** -53
        u1 = u[0::2]
        u2 = u[1::2]
        r = np.sqrt(-2.0 * np.log1p(-u1))
        t = 2.0 * np.pi * u2
        out[2 * p0:2 * p1:2] = r * np.cos(t)
        out[2 * p0 + 1:2 * p1:2] = r * np.sin(t)
    return out[:n]


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float64 -> float32 (RNE) -> bf16 (RNE), returned as uint16 bit patterns.

    Inputs here are finite; NaN handling is not needed by the generators.
    """
    u = np.ascontiguousarray(x, dtype=np.float64).astype(np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    with np.errstate(over="ignore"):
        return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (for display and fixtures)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_matrix(rows: int, cols: int, dist: str, seed: int, scale: float = 1.0) -> np.ndarray:
    """A (rows, cols) C-ordered uint16 array of bf16 bits.

    dist: ``"normal"`` (N(0,1)), ``"uniform"`` (U(-1,1)) or ``"ones"``.
    ``scale`` multiplies the float64 draw before rounding (e.g. 1/sqrt(K)).
    """
    n = rows * cols
    if dist == "normal":
        v = normal(seed, n)
    elif dist == "uniform":
        v = 2.0 * uniform01(seed, n) - 1.0
    elif dist == "ones":
        v = np.ones(n, dtype=np.float64)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    if scale != 1.0:
        v = v * scale
    return f64_to_bf16_bits(v).reshape(rows, cols)


def f32_matrix(rows: int, cols: int, dist: str, seed: int, scale: float = 1.0) -> np.ndarray:
    """A (rows, cols) float32 array (for an fp32 C_in)."""
    n = rows * cols
    if dist == "normal":
        v = normal(seed, n)
    elif dist == "uniform":
        v = 2.0 * uniform01(seed, n) - 1.0
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return (v * scale).astype(np.float32).reshape(rows, cols)


def store(logical: np.ndarray, layout: str, ld: int | None = None) -> tuple[np.ndarray, int]:
    """Lay a logical (rows, cols) matrix out in memory.

    layout ``"row"``: element (i, j) at ``i*ld + j``; ``"col"``: at ``j*ld + i``.
    ``ld`` defaults to the tight leading dimension rounded up to 8 elements, so
    that every row (or column) starts on a 16-byte boundary for 2-byte types.
    Returns (buffer, ld); padding elements are zero.
    """
    rows, cols = logical.shape
    inner, outer = (cols, rows) if layout == "row" else (rows, cols)
    if ld is None:
        ld = max(8, (inner + 7) // 8 * 8)
    if ld < inner:
        raise ValueError("leading dimension smaller than the contiguous extent")
    buf = np.zeros((outer, ld), dtype=logical.dtype)
    if layout == "row":
        buf[:, :inner] = logical
    else:
        buf[:, :inner] = logical.T
    return buf, ld
