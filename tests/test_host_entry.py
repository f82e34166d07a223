"""gemm_run_host: the GEMM on host buffers, copied in and out through the handle's staging.

Problems larger than one part are split along the larger of M and N; each part's
slice of the sliced operand (and of C) is copied in, computed and copied back
while the next part's copies run. These cases cover both chunked dimensions, the
slices that are whole lines of the stored matrix and those that are the same
columns of every line (pitched copies), padded leading dimensions whose padding
must come back untouched, beta != 0, K = 0 and several operand-sharing modes.
"""
import numpy as np
import pytest

from dense_gemm_cluster_gb300 import inputs
from gpu_cases import Problem, assert_close, decode, options_for

pytestmark = pytest.mark.gpu

SENTINEL_BF16 = np.uint16(0x4321)
SENTINEL_F32 = np.float32(-12345.0)


@pytest.fixture(scope="module")
def G():
    from dense_gemm_cluster_gb300 import build
    build.build()
    from dense_gemm_cluster_gb300 import gemm
    return gemm


def pad_ld(extent: int) -> int:
    return (extent + 7) // 8 * 8 + 8           # 16-byte aligned lines with 8 elements of padding


def padded(p: Problem):
    """Re-stores A, B and C_in of `p` with padded leading dimensions; C's padding holds a sentinel."""
    p.A, p.lda = inputs.store(p.A_log, p.la, pad_ld(p.K if p.la == "row" else p.M))
    p.B, p.ldb = inputs.store(p.B_log, p.lb, pad_ld(p.N if p.lb == "row" else p.K))
    c_inner = p.N if p.lc == "row" else p.M
    c_log = p.C_in[:, :c_inner] if p.lc == "row" else p.C_in[:, :c_inner].T
    p.C_in, p.ldc = inputs.store(np.ascontiguousarray(c_log), p.lc, pad_ld(c_inner))
    p.C_in[:, c_inner:] = SENTINEL_BF16 if p.out == "bf16" else SENTINEL_F32
    return p, c_inner


@pytest.mark.parametrize("M,N,K,la,lb,lc,out,beta,opts", [
    # along M (M >= N)
    (2100, 300, 256, "row", "col", "row", "bf16", 0.0,
     dict(mode="mcast", mcast_b=1, cluster_m=2, host_parts=3)),                     # 768, 768, 564 rows
    (2100, 300, 256, "col", "row", "col", "f32", 0.5, dict(host_parts=8)),           # 4 x 512 + 52; A, C by columns
    (2100, 300, 320, "row", "row", "row", "bf16", 0.5, dict(cta_group=2, cluster_m=2, host_parts=3)),
    # along N (N > M): B and C sliced
    (200, 1800, 320, "row", "row", "row", "bf16", 0.5,
     dict(mode="mcast", mcast_a=1, cluster_n=2, host_parts=8)),                     # 7 x 256 + a part of 8 columns
    (200, 1800, 320, "row", "col", "col", "f32", 0.0, dict(host_parts=4)),           # 3 x 512 + 264 lines
    (130, 4700, 192, "col", "col", "row", "f32", 0.0, dict(schedule="stream_k", host_parts=8)),  # 6 x 768 + 92
    (2100, 300, 256, "row", "col", "row", "bf16", 0.0, dict()),                      # the modelled count
])
def test_host_entry_matches_oracle_with_padding_untouched(G, M, N, K, la, lb, lc, out, beta, opts):
    p, c_inner = padded(Problem(M, N, K, la=la, lb=lb, lc=lc, out=out, beta=beta, seed=41))
    g = G.Gemm(0, **options_for(p, **opts))
    try:
        C = p.C_in.copy()
        g.run_host(M, N, K, p.A, p.lda, p.B, p.ldb, C, p.ldc, 1.0, beta)
        assert g.query_status() == G.GEMM_OK
    finally:
        g.close()
    assert_close(decode(C, M, N, lc), p.reference(1.0, beta), K, out, f"host entry {M}x{N}x{K} {la}{lb}{lc}")
    sentinel = SENTINEL_BF16 if out == "bf16" else SENTINEL_F32
    assert (C[:, c_inner:] == sentinel).all(), "the host copy-back wrote into C's padding"


def test_host_entry_k0_scales_c(G):
    # K = 0: C = beta * C, copied in and out in parts; A and B are never read.
    M, N = 1500, 100
    p, _ = padded(Problem(M, N, 0, la="row", lb="row", lc="row", out="f32", beta=0.5, seed=42))
    g = G.Gemm(0, **options_for(p, host_parts=2))
    try:
        C = p.C_in.copy()
        g.run_host(M, N, 0, None, 8, None, p.ldb, C, p.ldc, 1.0, 0.5)
    finally:
        g.close()
    np.testing.assert_array_equal(C[:, :N], (0.5 * p.C_in[:, :N].astype(np.float64)).astype(np.float32))
    assert (C[:, N:] == SENTINEL_F32).all()


def test_host_entry_repeats_on_one_handle(G):
    # The staging buffers, streams and events are reused across calls of different shapes.
    g = G.Gemm(0, layout_a="row", layout_b="col", layout_c="row", out_type="f32", host_parts=4)
    try:
        for (M, N, K, seed) in ((1100, 260, 128, 43), (260, 1300, 64, 44), (1100, 260, 128, 45)):
            p = Problem(M, N, K, la="row", lb="col", lc="row", out="f32", seed=seed)
            C = p.C_in.copy()
            g.run_host(M, N, K, p.A, p.lda, p.B, p.ldb, C, p.ldc, 1.0, 0.0)
            assert_close(decode(C, M, N, "row"), p.reference(), K, "f32", f"repeat {M}x{N}x{K}")
    finally:
        g.close()


def _batched_case(batch, M, N, K, la, lb, lc, out, beta, seed, a_stride_pad=0, c_extra=0, share_a=False):
    """Per-batch problems stored at strides (padding between batches and lines); returns buffers and refs."""
    probs = [Problem(M, N, K, la=la, lb=lb, lc=lc, out=out, beta=beta, seed=seed + 7 * i) for i in range(batch)]
    if share_a:
        for p in probs[1:]:
            p.A_log, p.A, p.lda = probs[0].A_log, probs[0].A, probs[0].lda
    p0 = probs[0]
    lda, ldb = p0.lda, p0.ldb
    ldc = pad_ld(N if lc == "row" else M) if c_extra else p0.ldc
    a_elems, b_elems = p0.A.size, p0.B.size
    c_outer = M if lc == "row" else N
    sA = 0 if share_a else a_elems + a_stride_pad
    sB = b_elems
    sC = c_outer * ldc + c_extra
    A = np.zeros(max(1, (batch - 1) * sA + a_elems), np.uint16)
    B = np.zeros((batch - 1) * sB + b_elems, np.uint16)
    cdt = np.uint16 if out == "bf16" else np.float32
    C = np.full((batch - 1) * sC + c_outer * ldc, SENTINEL_BF16 if out == "bf16" else SENTINEL_F32, cdt)
    refs = []
    c_inner = N if lc == "row" else M
    for i, p in enumerate(probs):
        A[i * sA:i * sA + a_elems] = p.A.reshape(-1)
        B[i * sB:i * sB + b_elems] = p.B.reshape(-1)
        c_log = p.C_in[:, :c_inner] if lc == "row" else p.C_in[:, :c_inner].T
        cb, _ = inputs.store(np.ascontiguousarray(c_log), lc, ldc)
        view = C[i * sC:i * sC + c_outer * ldc].reshape(c_outer, ldc)
        view[:, :c_inner] = cb[:, :c_inner]
        p.C_in, p.ldc = cb, ldc
        refs.append(p.reference(1.0, beta))
    return A, lda, sA, B, ldb, sB, C, ldc, sC, refs, c_inner, c_outer


@pytest.mark.parametrize("batch,M,N,K,la,lb,lc,out,beta,opts,extra", [
    (12, 300, 200, 128, "row", "col", "row", "f32", 0.0, dict(host_parts=4), {}),     # the score form, dense
    (7, 260, 300, 192, "row", "row", "row", "bf16", 0.5, dict(mode="mcast", mcast_b=1, cluster_m=2),
     dict(a_stride_pad=64, c_extra=40)),                                               # padded batches and lines
    (5, 256, 384, 64, "col", "col", "col", "f32", 0.5, dict(cta_group=2, cluster_n=2, host_parts=2),
     dict(share_a=True, c_extra=8)),                                                   # one A for every product
    (1, 300, 200, 128, "row", "col", "row", "bf16", 0.0, dict(), {}),                  # batch 1: gemm_run_host
])
def test_batched_host_entry_matches_oracle(G, batch, M, N, K, la, lb, lc, out, beta, opts, extra):
    A, lda, sA, B, ldb, sB, C, ldc, sC, refs, c_inner, c_outer = _batched_case(batch, M, N, K, la, lb, lc, out,
                                                                                beta, 60, **extra)
    g = G.Gemm(0, layout_a=la, layout_b=lb, layout_c=lc, out_type=out, **opts)
    try:
        g.run_strided_batched_host(M, N, K, A, lda, sA, B, ldb, sB, C, ldc, sC, batch, 1.0, beta)
        assert g.query_status() == G.GEMM_OK
    finally:
        g.close()
    sentinel = SENTINEL_BF16 if out == "bf16" else SENTINEL_F32
    for i in range(batch):
        view = C[i * sC:i * sC + c_outer * ldc].reshape(c_outer, ldc)
        assert_close(decode(view, M, N, lc), refs[i], K, out, f"batched host entry, product {i}")
        assert (view[:, c_inner:] == sentinel).all(), "line padding written"
        if i + 1 < batch:
            assert (C[i * sC + c_outer * ldc:(i + 1) * sC] == sentinel).all(), "padding between products written"
