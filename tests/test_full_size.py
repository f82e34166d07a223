"""Parity at the workloads' full sizes, in the launch configuration bench.py times.

Every output of the GEMM workloads and of all 128 heads of the score form is
compared with the fp64 oracle (max|C - C_ref| <= tol * max|C_ref|, the
workloads' tolerance). The oracle reads B as a column-major copy of the same
logical matrix, so its k loop runs over contiguous memory; the GPU gets the
workload's own layout. The attention forward and the 2^31-element case (whose
whole product does not fit the oracle's time) are checked on sampled rows and
positions the oracle computes one by one.
"""
import math

import numpy as np
import pytest

from gpu_cases import BF16_NAN, decode, from_dev, sample_positions, tolerance, torch_dev

pytestmark = pytest.mark.gpu


def _workload(name):
    from dense_gemm_cluster_gb300.workloads import WORKLOADS
    return WORKLOADS[name]


def _gemm_for(w):
    from dense_gemm_cluster_gb300 import gemm
    return gemm.Gemm(0, layout_a=w.layout_a, layout_b=w.layout_b, layout_c=w.layout_c, out_type=w.out, **w.options)


def _check_sampled(got_vals, ref_vals, K, out, what):
    scale = float(np.max(np.abs(ref_vals)))
    err = float(np.max(np.abs(got_vals - ref_vals))) / scale
    assert err <= tolerance(K, out), f"{what}: sampled max|err|/max|ref| = {err:.3e}"


def _check_all(got, ref, K, out, what):
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = float(np.max(np.abs(got - ref))) / float(np.max(np.abs(ref)))
    assert err <= tolerance(K, out), f"{what}: max|err|/max|ref| over all {got.size} outputs = {err:.3e}"


@pytest.mark.parametrize("name", ["gemm4096_bf16_cluster2x1", "gemm4096_bf16_pair2x1", "gemm8192_bf16_pair_mcastB4",
                                  "skinny_16384x128x8192", "skinny_128x16384x8192"])
def test_gemm_workload_every_output(name):
    import oracle
    from dense_gemm_cluster_gb300 import inputs
    w = _workload(name)
    A_log = inputs.bf16_matrix(w.M, w.K, w.dist, inputs.STREAM_A, w.scale)
    B_log = inputs.bf16_matrix(w.K, w.N, w.dist, inputs.STREAM_B, w.scale)
    A, lda = inputs.store(A_log, w.layout_a)
    B, ldb = inputs.store(B_log, w.layout_b)
    B_k, ldb_k = inputs.store(B_log, "col")          # the oracle's copy: k contiguous
    A_k, lda_k = inputs.store(A_log, "row")
    del A_log, B_log
    if w.beta != 0.0:
        C_in, ldc = inputs.store(inputs.bf16_matrix(w.M, w.N, w.c_dist, inputs.STREAM_C), w.layout_c)
    else:
        C_in, ldc = inputs.store(np.full((w.M, w.N), BF16_NAN, np.uint16), w.layout_c)
    g = _gemm_for(w)
    dC = torch_dev(C_in)
    g.run(w.M, w.N, w.K, torch_dev(A), lda, torch_dev(B), ldb, dC, ldc, w.alpha, w.beta)
    assert g.query_status() == 0
    g.close()
    got = decode(from_dev(dC, np.uint16), w.M, w.N, w.layout_c)
    del dC, A, B
    ref = oracle.gemm(w.M, w.N, w.K, A_k, lda_k, "row", B_k, ldb_k, "col", w.alpha, w.beta,
                      C_in if w.beta != 0.0 else None, ldc, w.layout_c)
    _check_all(got, ref, w.K, w.out, name)
    # magnitudes: A and B iid with variances va, vb -> sum over K has variance K va vb (+ beta^2 var C)
    va = {"normal": 1.0, "uniform": 1.0 / 3.0}[w.dist] * w.scale ** 2
    expect = math.sqrt(w.K * va * va + (w.beta ** 2 if w.beta else 0.0))
    assert 0.8 < float(np.std(got)) / expect < 1.25


def test_scores_workload_every_output():
    # All 128 (batch, head) products of the score form, one head at a time against the oracle.
    import torch
    import oracle
    from dense_gemm_cluster_gb300 import inputs
    w = _workload("scores_8x16x4096x4096x128")
    Q = inputs.bf16_matrix(w.batch * w.M, w.K, w.dist, inputs.STREAM_A)
    Kt = inputs.bf16_matrix(w.batch * w.N, w.K, w.dist, inputs.STREAM_B)
    g = _gemm_for(w)
    dS = torch.empty(w.batch * w.M * w.N, dtype=torch.float32, device="cuda")
    g.run_strided_batched(w.M, w.N, w.K, torch_dev(Q), w.K, w.M * w.K, torch_dev(Kt), w.K, w.N * w.K, dS, w.N,
                          w.M * w.N, w.batch)
    assert g.query_status() == 0
    g.close()
    assert bool(torch.isfinite(dS).all())
    for b in range(w.batch):
        got = dS[b * w.M * w.N:(b + 1) * w.M * w.N].view(w.M, w.N).cpu().numpy().astype(np.float64)
        ref = oracle.attention_scores(Q[b * w.M:(b + 1) * w.M].reshape(1, w.M, w.K),
                                      Kt[b * w.N:(b + 1) * w.N].reshape(1, w.N, w.K))[0]
        _check_all(got, ref, w.K, "f32", f"scores batch {b}")
        if b in (0, w.batch - 1):
            assert 0.8 < float(np.std(got)) / math.sqrt(w.K) < 1.25


@pytest.mark.parametrize("name", ["attention_fwd_8x16x4096x4096x128", "attention_fwd_causal_8x16x4096x4096x128"])
def test_attention_workload_full_size_sampled(name):
    # The bench's attention launch (all 128 heads, its cluster size); rows of six heads
    # are checked against the oracle, which treats each query row independently (a causal
    # row r is the plain softmax over keys 0..r).
    import torch
    import oracle
    from dense_gemm_cluster_gb300 import gemm, inputs
    from dense_gemm_cluster_gb300.workloads import ATTENTION_WORKLOADS
    w = ATTENTION_WORKLOADS[name]
    Q = inputs.bf16_matrix(w.batch * w.sq, w.d, w.dist, inputs.STREAM_A).reshape(w.batch, w.sq, w.d)
    K = inputs.bf16_matrix(w.batch * w.sk, w.d, w.dist, inputs.STREAM_B).reshape(w.batch, w.sk, w.d)
    V = inputs.bf16_matrix(w.batch * w.sk, w.d, w.dist, inputs.STREAM_C).reshape(w.batch, w.sk, w.d)
    dev = lambda a: torch.from_numpy(a.reshape(-1).view(np.int16)).cuda()
    O = torch.empty(w.batch * w.sq * w.d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(w.batch * w.sq, dtype=torch.float32, device="cuda")
    s = gemm.attention_forward_run(dev(Q), dev(K), dev(V), O, lse, w.batch, w.sq, w.sk, w.d, 0.0, 0, w.cluster,
                                   w.cta_group, causal=w.causal)
    assert s == gemm.GEMM_OK and gemm.attention_forward_query_status() == gemm.GEMM_OK
    O = O.view(w.batch, w.sq, w.d)
    lse = lse.view(w.batch, w.sq)
    assert bool(torch.isfinite(O).all()) and bool(torch.isfinite(lse).all())
    rng = np.random.default_rng(3)
    vmax = float(np.max(np.abs(inputs.bf16_bits_to_f32(V))))
    for b in sorted(set([0, w.batch - 1] + list(rng.integers(0, w.batch, size=4)))):
        rows = np.unique(np.concatenate([[0, 127, 128, 255, 256, w.sq - 1], rng.integers(0, w.sq, size=26)]))
        if w.causal:
            parts = [oracle.attention_forward(Q[b:b + 1, [r]], K[b:b + 1, :r + 1], V[b:b + 1, :r + 1], with_lse=True)
                     for r in rows]
            ref = np.concatenate([o for o, _ in parts], axis=1)
            ref_lse = np.concatenate([l for _, l in parts], axis=1)
        else:
            ref, ref_lse = oracle.attention_forward(Q[b:b + 1, rows], K[b:b + 1], V[b:b + 1], with_lse=True)
        got = O[b, torch.from_numpy(rows).cuda()].float().cpu().numpy().astype(np.float64)
        got_lse = lse[b, torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64)
        assert np.max(np.abs(got - ref[0])) <= 1e-2 * vmax, f"head {b}"
        assert np.max(np.abs(got_lse - ref_lse[0]) / (1.0 + np.abs(ref_lse[0]))) <= 1e-4, f"head {b}"


@pytest.mark.parametrize("opts", [dict(mode="mcast", mcast_b=1, cluster_m=2),
                                  dict(cta_group=2, cluster_m=2, schedule="stream_k")])
def test_output_past_2_31_elements(opts):
    # One C of 131272 x 16512 bf16 (2.17e9 elements, more rows than a 16-bit coordinate):
    # element offsets past 2^31 in the beta * C_in reads, the TMA stores and (stream-K)
    # the partial slots. C_in is the pattern c[i, j] = ((i mod 61) - 30 - (j mod 53)) / 16,
    # exact in bf16 and known at every position, so the expected value is the oracle's
    # product plus beta times the pattern.
    import torch
    import oracle
    from dense_gemm_cluster_gb300 import gemm, inputs
    M, N, K, beta = 131272, 16512, 128, 0.5
    A, lda = inputs.store(inputs.bf16_matrix(M, K, "normal", 51), "row")
    B, ldb = inputs.store(inputs.bf16_matrix(K, N, "normal", 52), "row")
    pattern = lambda i, j: ((i % 61) - 30.0 - (j % 53)) / 16.0
    ri = torch.arange(M, device="cuda", dtype=torch.float32).view(M, 1)
    cj = torch.arange(N, device="cuda", dtype=torch.float32).view(1, N)
    dC = ((ri.remainder(61) - 30.0) - cj.remainder(53)).mul_(1.0 / 16.0).to(torch.bfloat16).view(-1)
    g = gemm.Gemm(0, layout_a="row", layout_b="row", layout_c="row", out_type="bf16", **opts)
    try:
        g.run(M, N, K, torch_dev(A), lda, torch_dev(B), ldb, dC, N, 1.0, beta)
        assert g.query_status() == 0
    finally:
        g.close()
    rows, cols = sample_positions(M, N, 2000, seed=3)
    rng = np.random.default_rng(4)
    far = int(2 ** 31 // N) + 1                  # rows whose every element lies past 2^31
    rows = np.concatenate([rows, rng.integers(far, M, 500), [M - 1, far]])
    cols = np.concatenate([cols, rng.integers(0, N, 500), [N - 1, 0]])
    flat = torch.from_numpy(rows * N + cols).cuda()
    got = inputs.bf16_bits_to_f32(dC.view(torch.int16)[flat].cpu().numpy().view(np.uint16)).astype(np.float64)
    ref = oracle.gemm_entries(rows, cols, K, A, lda, "row", B, ldb, "row") + beta * pattern(rows, cols)
    _check_sampled(got, ref, K, "bf16", f"2^31+ elements {opts}")
    del dC
    torch.cuda.empty_cache()
