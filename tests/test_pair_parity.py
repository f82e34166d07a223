"""GPU parity of the 2-SM pair MMA (tcgen05 cta_group::2), alone and with cluster multicast.

"Clusters, distributed shared memory & cluster launch control", section "Two
CTAs, one MMA -- cta_group::2": A is split by rows across the pair, B by
columns, each CTA keeps its half of the 256-row accumulator; the product is
the same GEMM, so the oracle is unchanged.
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


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("la,lb", [("row", "col"), ("row", "row"), ("col", "row")])
def test_pair_unicast(G, bn, la, lb):
    p = Problem(512, 768, 384, la=la, lb=lb, out="bf16", seed=11)
    got = _run(G, p, cta_group=2, cluster_m=2, block_n=bn)
    assert_close(got, p.reference(), 384, "bf16", f"pair bn={bn} {la}/{lb}")


@pytest.mark.parametrize("cm,cn,ma,mb", [(4, 1, 0, 1), (2, 2, 1, 0), (4, 2, 1, 1), (2, 4, 1, 0), (8, 1, 0, 1)])
def test_pair_with_multicast_bitwise_equals_pair_unicast(G, cm, cn, ma, mb):
    p = Problem(1100, 1300, 512, la="row", lb="row", out="bf16", seed=12)
    base = _run(G, p, cta_group=2, cluster_m=2, cluster_n=1, schedule="dp")
    got = _run(G, p, cta_group=2, cluster_m=cm, cluster_n=cn, mode="mcast", mcast_a=ma, mcast_b=mb, schedule="dp")
    assert_close(got, p.reference(), 512, "bf16", f"pair cluster {cm}x{cn} A{ma} B{mb}")
    assert np.array_equal(got, base)


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (129, 257, 65), (383, 130, 300), (256, 1, 17)])
def test_pair_ragged(G, M, N, K):
    p = Problem(M, N, K, la="row", lb="row", out="f32", seed=13)
    got = _run(G, p, cta_group=2, cluster_m=4, mode="mcast", mcast_b=1)
    assert_close(got, p.reference(), K, "f32", f"pair ragged {M}x{N}x{K}")


def test_pair_beta_and_column_major_c(G):
    p = Problem(640, 520, 256, la="row", lb="row", lc="col", out="bf16", beta=0.5, seed=14)
    got = _run(G, p, 1.0, 0.5, cta_group=2, cluster_m=1, cluster_n=2)   # C^T: cluster_n becomes the pair axis
    assert_close(got, p.reference(1.0, 0.5), 256, "bf16", "pair beta col-major C")


def test_pair_persistent_few_clusters(G):
    p = Problem(1536, 1024, 512, seed=15)
    got = _run(G, p, cta_group=2, cluster_m=4, mode="mcast", mcast_b=1, max_clusters=2, stages=3)
    assert_close(got, p.reference(), 512, "bf16", "pair persistent")


@pytest.mark.parametrize("la,lb", [("row", "col"), ("row", "row"), ("col", "col")])
@pytest.mark.parametrize("cm,cn,ma,mb,bn", [(2, 1, 0, 0, 256), (4, 1, 0, 1, 256), (8, 1, 0, 1, 128),
                                            (2, 4, 1, 0, 256), (4, 2, 1, 1, 128)])
def test_pair_128_wide_stages(G, la, lb, cm, cn, ma, mb, bn):
    # K = 448 = 3.5 stages of 128: the last stage's second atom lies past K and must read as zeros
    p = Problem(700, 1100, 448, la=la, lb=lb, out="bf16", seed=16)
    base = _run(G, p, cta_group=2, cluster_m=2, block_k=64, schedule="dp")
    got = _run(G, p, cta_group=2, cluster_m=cm, cluster_n=cn, mode="mcast", mcast_a=ma, mcast_b=mb,
               block_n=bn, block_k=128, schedule="dp")
    assert_close(got, p.reference(), 448, "bf16", f"pair bk128 {la}/{lb} cluster {cm}x{cn} A{ma} B{mb} bn{bn}")
    if bn == 256:
        assert np.array_equal(got, base)   # same MMA sequence per k: bit-identical


@pytest.mark.parametrize("K", [200, 65, 1])
def test_pair_auto_stage_width_with_ragged_k(G, K):
    p = Problem(300, 520, K, la="row", lb="col", out="f32", seed=17)
    got = _run(G, p, cta_group=2, cluster_m=2)
    assert_close(got, p.reference(), K, "f32", f"pair ragged K={K}")


@pytest.mark.parametrize("cm,cn,ma,mb", [(2, 1, 0, 0), (4, 1, 0, 1), (2, 2, 1, 0)])
def test_pair_stream_k_tail(G, cm, cn, ma, mb):
    p = Problem(1024, 1536, 1152, la="row", lb="row", out="bf16", beta=0.5, seed=18)
    got = _run(G, p, 1.0, 0.5, cta_group=2, cluster_m=cm, cluster_n=cn, mode="mcast", mcast_a=ma, mcast_b=mb,
               schedule="stream_k", max_clusters=5)
    assert_close(got, p.reference(1.0, 0.5), 1152, "bf16", f"pair stream-K {cm}x{cn}")


def test_pair_stream_k_spreads_when_most_pairs_are_busy(G):
    # 4 pair tiles on 6 pairs: an explicit stream-K schedule splits every tile's k-blocks
    p = Problem(1024, 256, 4096, la="row", lb="row", out="f32", seed=20)
    got = _run(G, p, cta_group=2, cluster_m=2, schedule="stream_k", max_clusters=6)
    assert_close(got, p.reference(), 4096, "f32", "pair stream-K spread")


def test_pair_sub_wave_problem_spreads_over_more_clusters(G):
    # 2 pair tiles of 256x256 with 64 k-blocks each: the auto schedule splits them over more pairs
    p = Problem(512, 256, 8192, la="row", lb="col", out="bf16", beta=0.5, seed=19)
    a = _run(G, p, 1.0, 0.5, cta_group=2, cluster_m=2)
    b = _run(G, p, 1.0, 0.5, cta_group=2, cluster_m=2)
    assert_close(a, p.reference(1.0, 0.5), 8192, "bf16", "pair sub-wave")
    assert np.array_equal(a, b)


def test_auto_cta_group_picks_the_pair_and_matches_the_oracle(G):
    # cta_group 0 with an even cluster extent along M runs the pair MMA: the same launch,
    # bit for bit, as asking for cta_group 2, and within the tolerance of the oracle.
    p = Problem(700, 1100, 448, la="row", lb="col", out="bf16", beta=0.5, seed=21)
    s, plan = G.gemm_plan(G.make_options(**options_for(p, cta_group=0, cluster_m=4, mode="mcast", mcast_b=1)),
                          p.M, p.N, p.K, 1, 152)
    assert s == 0 and plan.cta_group == 2
    auto = _run(G, p, 1.0, 0.5, cta_group=0, cluster_m=4, mode="mcast", mcast_b=1)
    pair = _run(G, p, 1.0, 0.5, cta_group=2, cluster_m=4, mode="mcast", mcast_b=1)
    assert np.array_equal(auto, pair)
    assert_close(auto, p.reference(1.0, 0.5), 448, "bf16", "auto cta_group")
