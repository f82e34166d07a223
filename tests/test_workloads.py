"""The synthetic workloads the bench and the full-size tests run, held to their stated
configurations: sizes, distributions, layouts, output type, alpha/beta and the operand-sharing
mode. (No GPU needed.)"""
import math

from dense_gemm_cluster_gb300.workloads import ATTENTION_WORKLOADS, DEFAULT, WORKLOADS


def test_small_gemm_256_fp32_with_b_multicast_over_a_2_cta_cluster():
    w = WORKLOADS["gemm256_f32_mcastB"]
    assert (w.M, w.N, w.K, w.batch) == (256, 256, 256, 1)
    assert w.dist == "normal" and w.scale == 1.0 and w.out == "f32"
    assert (w.layout_a, w.layout_b, w.layout_c) == ("row", "row", "row")
    assert w.options == dict(mode="mcast", mcast_b=1, cluster_m=2, cluster_n=1)


def test_gemm_4096_uniform_a_row_b_col_bf16_on_a_2x1_cluster():
    w = WORKLOADS["gemm4096_bf16_cluster2x1"]
    assert (w.M, w.N, w.K) == (4096, 4096, 4096)
    assert w.dist == "uniform" and (w.layout_a, w.layout_b) == ("row", "col") and w.out == "bf16"
    assert (w.alpha, w.beta) == (1.0, 0.0)
    assert w.options == dict(mode="mcast", mcast_a=1, mcast_b=1, cluster_m=2, cluster_n=1)
    pair = WORKLOADS["gemm4096_bf16_pair2x1"]      # the same problem on a pair
    assert (pair.M, pair.N, pair.K, pair.dist, pair.layout_a, pair.layout_b, pair.out) == \
        (w.M, w.N, w.K, w.dist, w.layout_a, w.layout_b, w.out)
    assert pair.options["cta_group"] == 2 and pair.options["cluster_m"] == 2


def test_gemm_8192_scaled_normal_pair_tiles_b_multicast_beta_half():
    w = WORKLOADS["gemm8192_bf16_pair_mcastB4"]
    assert (w.M, w.N, w.K) == (8192, 8192, 8192)
    assert w.dist == "normal" and math.isclose(w.scale, 1.0 / math.sqrt(8192))
    assert w.out == "bf16" and w.beta == 0.5 and w.c_dist == "normal"
    o = w.options
    assert o["cta_group"] == 2 and o["block_n"] == 256 and o["cluster_m"] == 4 and o["mcast_b"] == 1
    uni = WORKLOADS["gemm8192_bf16_unicast"]       # the comparison: same problem, unicast tiles
    assert (uni.M, uni.N, uni.K, uni.dist, uni.scale, uni.beta) == (w.M, w.N, w.K, w.dist, w.scale, w.beta)
    assert uni.options["mode"] == "unicast" and uni.options.get("cta_group", 1) == 1
    assert DEFAULT == w.name                       # the bench's default: the largest single-GPU GEMM


def test_unicast_twins_compute_the_same_output():
    from dense_gemm_cluster_gb300.workloads import UNICAST_TWIN
    for name, twin in UNICAST_TWIN.items():
        w, u = WORKLOADS[name], WORKLOADS[twin]
        same = lambda x: (x.M, x.N, x.K, x.batch, x.dist, x.scale, x.layout_a, x.layout_b, x.layout_c, x.out,
                          x.alpha, x.beta)
        assert same(w) == same(u)
        assert u.options["mode"] == "unicast" and u.options.get("cta_group", 1) == 1
        assert u.options.get("cluster_m", 1) == 1 and u.options.get("cluster_n", 1) == 1


def test_attention_scores_8x16_heads_4096_by_4096_by_128_fp32():
    w = WORKLOADS["scores_8x16x4096x4096x128"]
    assert (w.M, w.N, w.K, w.batch) == (4096, 4096, 128, 8 * 16)
    assert w.dist == "normal" and w.out == "f32" and (w.alpha, w.beta) == (1.0, 0.0)   # no 1/sqrt(d)
    assert (w.layout_a, w.layout_b) == ("row", "col")          # Q row-major, K row-major = B column-major
    assert w.options["mcast_b"] == 1 and w.options["cluster_m"] > 1   # K tiles shared by Q-tile CTAs


def test_skinny_gemms_share_their_small_operand():
    a = WORKLOADS["skinny_16384x128x8192"]
    b = WORKLOADS["skinny_128x16384x8192"]
    assert (a.M, a.N, a.K) == (16384, 128, 8192) and (b.M, b.N, b.K) == (128, 16384, 8192)
    for w in (a, b):
        assert w.dist == "uniform" and w.out == "bf16" and w.options["mode"] == "mcast"
    assert a.options["mcast_b"] == 1 and b.options["mcast_a"] == 1


def test_attention_forward_workloads():
    w = ATTENTION_WORKLOADS["attention_fwd_8x16x4096x4096x128"]
    assert (w.batch, w.sq, w.sk, w.d) == (8 * 16, 4096, 4096, 128) and not w.causal
    assert w.flops == 4 * 128 * 4096 * 4096 * 128
    c = ATTENTION_WORKLOADS["attention_fwd_causal_8x16x4096x4096x128"]
    assert c.causal and c.pairs == 4096 * 4097 // 2
