"""Cluster launch control (hardware work stealing) as the tile scheduler.

"Clusters, distributed shared memory & cluster launch control", sections
"Cluster launch control" and "The work-stealing loop": the grid has one
cluster per tile, resident clusters cancel pending launches and take their
tiles, asking before computing, and stop at the first request that comes back
not canceled. The product is unchanged, so the oracle is too; every tile must
be computed exactly once (a tile taken twice or never shows up as a mismatch).
"""
import numpy as np
import pytest

from gpu_cases import Problem, assert_close, options_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def G():
    import torch
    from dense_gemm_cluster_gb300 import gemm
    assert torch.cuda.is_available()
    return gemm


def _run(G, p, alpha=1.0, beta=0.0, **opts):
    g = G.Gemm(0, **options_for(p, **opts))
    try:
        dC = p.run(g, alpha, beta)
        assert g.query_status() == G.GEMM_OK, G.gemm_last_error(g.handle)
        return p.result(dC)
    finally:
        g.close()


@pytest.mark.parametrize("mode", [
    dict(),
    dict(mode="mcast", mcast_b=1, cluster_m=2),
    dict(mode="mcast", mcast_a=1, mcast_b=1, cluster_m=2, cluster_n=2),
    dict(cta_group=2, cluster_m=2),
    dict(cta_group=2, cluster_m=4, mode="mcast", mcast_b=1),
    dict(block_n=128, block_k=128),
])
def test_clc_matches_oracle_and_whole_tile_schedule(G, mode):
    # 3072 x 4096 with 128x256 tiles: 384 tiles, well over one wave, so most are stolen
    p = Problem(3072, 4096, 320, la="row", lb="col", out="bf16", seed=40)
    got = _run(G, p, schedule="clc", **mode)
    assert_close(got, p.reference(), 320, "bf16", f"clc {mode}")
    dp = _run(G, p, schedule="dp", **mode)
    assert np.array_equal(got, dp)        # same per-tile arithmetic, only the assignment differs


def test_clc_ragged_and_beta(G):
    p = Problem(1100, 2500, 200, la="col", lb="row", out="f32", beta=0.5, seed=41)
    got = _run(G, p, 1.0, 0.5, schedule="clc", mode="mcast", mcast_b=1, cluster_m=2)
    assert_close(got, p.reference(1.0, 0.5), 200, "f32", "clc ragged beta")


def test_clc_batched_scores_form(G):
    import torch
    from dense_gemm_cluster_gb300 import inputs
    import oracle
    b, s, d = 6, 640, 128
    Q = inputs.bf16_matrix(b * s, d, "normal", 42)
    K = inputs.bf16_matrix(b * s, d, "normal", 43)
    dQ = torch.from_numpy(Q.view(np.int16).copy()).cuda()
    dK = torch.from_numpy(K.view(np.int16).copy()).cuda()
    dS = torch.empty(b * s * s, dtype=torch.float32, device="cuda")
    g = G.Gemm(0, layout_a="row", layout_b="col", out_type="f32", schedule="clc", mode="mcast", mcast_b=1,
               cluster_m=2)
    g.run_strided_batched(s, s, d, dQ, d, s * d, dK, d, s * d, dS, s, s * s, b)
    assert g.query_status() == G.GEMM_OK
    g.close()
    ref = oracle.attention_scores(Q.reshape(b, s, d), K.reshape(b, s, d))
    got = dS.cpu().numpy().reshape(b, s, s).astype(np.float64)
    assert_close(got.reshape(-1, s), ref.reshape(-1, s), d, "f32", "clc scores")
