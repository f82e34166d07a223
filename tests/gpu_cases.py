"""Shared helpers for the GPU parity tests: seeded inputs -> device -> C ABI -> compare with the oracle.

The tolerance is the one the workloads state: for bf16 output
    max|C_gpu - C_ref| <= 1e-2 * sqrt(K / 256) * max|C_ref|,
floored at one bf16 unit in the last place of max|C_ref| (2^-8 relative) so
that shapes with K < 256 are not held to less than the single output
rounding; for fp32 output max|C_gpu - C_ref| <= 2e-3 * max|C_ref|.
"""
from __future__ import annotations

import math

import numpy as np

from dense_gemm_cluster_gb300 import inputs

BF16_NAN = np.uint16(0x7FC0)


def tolerance(K: int, out: str) -> float:
    if out == "f32":
        return 2e-3
    return max(1e-2 * math.sqrt(max(K, 1) / 256.0), 2.0 ** -8)


def torch_dev(buf: np.ndarray):
    import torch
    if buf.dtype == np.uint16:
        return torch.from_numpy(buf.view(np.int16).copy()).cuda()
    return torch.from_numpy(buf.copy()).cuda()


def from_dev(t, dtype) -> np.ndarray:
    a = t.cpu().numpy()
    return a.view(np.uint16) if dtype == np.uint16 else a


def decode(buf: np.ndarray, rows: int, cols: int, layout: str) -> np.ndarray:
    """Logical (rows, cols) float64 view of an output buffer."""
    vals = inputs.bf16_bits_to_f32(buf).astype(np.float64) if buf.dtype == np.uint16 else buf.astype(np.float64)
    if layout == "row":
        return vals[:rows, :cols].copy()
    return vals[:cols, :rows].T.copy()


class Problem:
    """One seeded GEMM instance: logical matrices, stored buffers, and their leading dimensions."""

    def __init__(self, M, N, K, la="row", lb="col", lc="row", out="bf16", beta=0.0, seed=0,
                 dist="normal", scale=1.0, c_dist="normal"):
        self.M, self.N, self.K = M, N, K
        self.la, self.lb, self.lc, self.out = la, lb, lc, out
        self.A_log = inputs.bf16_matrix(M, K, dist, seed + inputs.STREAM_A, scale)
        self.B_log = inputs.bf16_matrix(K, N, dist, seed + inputs.STREAM_B, scale)
        self.A, self.lda = inputs.store(self.A_log, la)
        self.B, self.ldb = inputs.store(self.B_log, lb)
        if beta != 0.0:
            if out == "bf16":
                C_log = inputs.bf16_matrix(M, N, c_dist, seed + inputs.STREAM_C)
            else:
                C_log = inputs.f32_matrix(M, N, c_dist, seed + inputs.STREAM_C)
        else:
            # beta == 0 must not read C: fill it with NaN.
            C_log = np.full((M, N), BF16_NAN, np.uint16) if out == "bf16" else np.full((M, N), np.nan, np.float32)
        self.C_in, self.ldc = inputs.store(C_log, lc)
        self.C_dtype = np.uint16 if out == "bf16" else np.float32

    def reference(self, alpha=1.0, beta=0.0) -> np.ndarray:
        import oracle
        return oracle.gemm(self.M, self.N, self.K, self.A, self.lda, self.la, self.B, self.ldb, self.lb,
                           alpha, beta, self.C_in if beta != 0.0 else None, self.ldc, self.lc)

    def reference_entries(self, rows, cols, alpha=1.0, beta=0.0) -> np.ndarray:
        import oracle
        return oracle.gemm_entries(rows, cols, self.K, self.A, self.lda, self.la, self.B, self.ldb, self.lb,
                                   alpha, beta, self.C_in if beta != 0.0 else None, self.ldc, self.lc)

    def run(self, handle_gemm, alpha=1.0, beta=0.0, stream=None):
        """Runs on the GPU through the C ABI; returns the device output buffer (torch)."""
        dA, dB, dC = torch_dev(self.A), torch_dev(self.B), torch_dev(self.C_in)
        handle_gemm.run(self.M, self.N, self.K, dA, self.lda, dB, self.ldb, dC, self.ldc, alpha, beta, stream)
        return dC

    def result(self, dC) -> np.ndarray:
        return decode(from_dev(dC, self.C_dtype), self.M, self.N, self.lc)


def options_for(p: Problem, **kw) -> dict:
    d = dict(layout_a=p.la, layout_b=p.lb, layout_c=p.lc, out_type=p.out)
    d.update(kw)
    return d


def max_rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    if ref.size == 0:
        return 0.0
    err = float(np.max(np.abs(got - ref)))
    return err / scale if scale > 0 else err


def assert_close(got: np.ndarray, ref: np.ndarray, K: int, out: str, what: str = "") -> None:
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    e = max_rel_err(got, ref)
    tol = tolerance(K, out)
    assert e <= tol, f"{what}: max|err|/max|ref| = {e:.3e} > {tol:.3e}"


def sample_positions(M: int, N: int, n: int, seed: int = 0, tile_m: int = 128, tile_n: int = 256):
    """Positions that hit every corner of the matrix, tile edges, and random interior points."""
    rng = np.random.default_rng(seed)
    rows = [0, M - 1, 0, M - 1, M // 2]
    cols = [0, N - 1, N - 1, 0, N // 2]
    for e in (tile_m - 1, tile_m, 2 * tile_m - 1):
        if e < M:
            rows.append(e); cols.append(int(rng.integers(N)))
    for e in (tile_n - 1, tile_n, 2 * tile_n - 1):
        if e < N:
            rows.append(int(rng.integers(M))); cols.append(e)
    k = max(0, n - len(rows))
    rows += list(rng.integers(0, M, size=k))
    cols += list(rng.integers(0, N, size=k))
    return np.array(rows, dtype=np.int64), np.array(cols, dtype=np.int64)
