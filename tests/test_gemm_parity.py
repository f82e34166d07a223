"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

cta_group 1 here (unicast and cluster multicast); the pair MMA has its own file.
"""
import numpy as np
import pytest

from gpu_cases import Problem, assert_close, decode, options_for, torch_dev

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


def test_small_256_fp32_cluster2_multicast_b(G):
    # 256^3, N(0,1), fp32 out, all row-major, a 2-CTA cluster sharing B by multicast
    p = Problem(256, 256, 256, la="row", lb="row", lc="row", out="f32", seed=0)
    got = _run(G, p, mode="mcast", mcast_b=1, cluster_m=2, cluster_n=1)
    assert_close(got, p.reference(), 256, "f32", "256^3 mcast B")


@pytest.mark.parametrize("la,lb", [("row", "col"), ("row", "row"), ("col", "col"), ("col", "row")])
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_layouts_unicast(G, la, lb, out):
    p = Problem(384, 512, 320, la=la, lb=lb, out=out, seed=1)
    got = _run(G, p)
    assert_close(got, p.reference(), 320, out, f"{la}/{lb}/{out}")


def test_identity_is_bit_exact(G):
    from dense_gemm_cluster_gb300 import inputs
    p = Problem(256, 384, 256, la="row", lb="row", out="bf16", seed=2)
    p.A_log = inputs.f64_to_bf16_bits(np.eye(256))
    p.A, p.lda = inputs.store(p.A_log, "row")
    got = _run(G, p)
    assert np.array_equal(got, inputs.bf16_bits_to_f32(p.B_log).astype(np.float64))


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (17, 130, 257), (130, 17, 64), (257, 257, 17),
                                   (129, 300, 130), (1, 513, 65), (300, 1, 200)])
@pytest.mark.parametrize("lc", ["row", "col"])
def test_ragged_shapes(G, M, N, K, lc):
    p = Problem(M, N, K, la="row", lb="row", lc=lc, out="bf16", seed=3)
    got = _run(G, p)
    assert_close(got, p.reference(), K, "bf16", f"{M}x{N}x{K} C {lc}")


@pytest.mark.parametrize("alpha,beta,out", [(0.5, 0.0, "bf16"), (1.0, 1.0, "bf16"), (-2.0, 0.5, "f32"),
                                            (0.0, -1.5, "bf16"), (1.0, 0.5, "f32")])
def test_alpha_beta(G, alpha, beta, out):
    p = Problem(300, 600, 192, out=out, beta=beta, seed=4)
    got = _run(G, p, alpha, beta)
    assert_close(got, p.reference(alpha, beta), 192, out, f"alpha={alpha} beta={beta}")


@pytest.mark.parametrize("cm,cn,ma,mb", [(2, 1, 0, 1), (1, 2, 1, 0), (2, 2, 1, 1), (4, 1, 0, 1),
                                         (1, 4, 1, 0), (4, 2, 1, 1), (2, 4, 1, 1), (8, 1, 0, 1),
                                         (2, 1, 0, 0), (2, 2, 0, 0)])
@pytest.mark.parametrize("bn", [128, 256])
def test_cluster_modes_match_oracle_and_unicast_bitwise(G, cm, cn, ma, mb, bn):
    p = Problem(1000, 1100, 448, la="row", lb="col", out="bf16", seed=5)
    uni = _run(G, p, block_n=bn, schedule="dp")
    got = _run(G, p, mode="mcast", mcast_a=ma, mcast_b=mb, cluster_m=cm, cluster_n=cn, block_n=bn, schedule="dp")
    assert_close(got, p.reference(), 448, "bf16", f"cluster {cm}x{cn} mcast A{ma} B{mb}")
    # multicast moves the same operand bytes: the product is bit-identical
    assert np.array_equal(got, uni)


@pytest.mark.parametrize("opts", [dict(block_n=128),
                                  dict(cta_group=2, cluster_m=4, mode="mcast", mcast_b=1, block_n=128),
                                  dict(block_n=128, schedule="stream_k", max_clusters=6)])
def test_rotated_k_walk_with_l2_hints_matches_oracle(G, opts):
    # One tile along N: the planner streams A with an evict-first policy, keeps the B that
    # every tile reads with evict-last, and starts each whole tile's k walk at its own
    # k-block, wrapping around. K = 1000 leaves a partial last k-block, which the rotated
    # walk must still load exactly once; the stream-K case mixes split pieces (in order)
    # with rotated whole tiles.
    p = Problem(1536, 100, 1000, la="row", lb="row", out="f32", seed=97)
    s, plan = G.gemm_plan(G.make_options(**options_for(p, **opts)), p.M, p.N, p.K, 1, 152)
    assert s == 0 and (plan.k_rotate, plan.l2_hint_a, plan.l2_hint_b) == (1, 1, 2)
    got = _run(G, p, **opts)
    assert_close(got, p.reference(), p.K, "f32", f"rotated k walk {opts}")


@pytest.mark.parametrize("opts", [dict(max_clusters=20, schedule="dp"),
                                  dict(max_clusters=20, schedule="stream_k"),
                                  dict(cta_group=2, cluster_m=4, mode="mcast", mcast_b=1, max_clusters=6)])
def test_serpentine_k_walk_matches_oracle(G, opts):
    # Long K on several waves of whole tiles: every other whole tile of a cluster walks its
    # k-blocks backwards, so it starts on the partial last k-block (K = 1100 is 17.2 blocks
    # of 64). With stream-K the last waves' split pieces stay in order.
    p = Problem(2048, 1536, 1100, la="row", lb="col", out="bf16", beta=0.5, seed=98)
    s, plan = G.gemm_plan(G.make_options(**options_for(p, **opts)), p.M, p.N, p.K, 1, 152)
    assert s == 0 and plan.k_serpentine == 1 and plan.tiles >= 2 * plan.clusters
    got = _run(G, p, 1.0, 0.5, **opts)
    assert_close(got, p.reference(1.0, 0.5), p.K, "bf16", f"serpentine {opts}")


def test_serpentine_walk_and_snaking_bands_over_a_batch(G):
    # Three products of 1024 x 1280 x 2048 on 8 clusters: 32 k-blocks, several waves of whole
    # tiles per product, bands of 4 tile rows that snake within each product.
    import torch
    M, N, K, batch = 1024, 1280, 2048, 3
    s, plan = G.gemm_plan(G.make_options(layout_a="row", layout_b="col", out_type="f32", max_clusters=8),
                          M, N, K, batch, 152)
    assert s == 0 and plan.k_serpentine == 1
    probs = [Problem(M, N, K, la="row", lb="col", out="f32", seed=70 + i) for i in range(batch)]
    dA = torch.cat([torch_dev(p.A).view(-1) for p in probs])
    dB = torch.cat([torch_dev(p.B).view(-1) for p in probs])
    dC = torch.full((batch * M * N,), float("nan"), dtype=torch.float32, device="cuda")
    g = G.Gemm(0, layout_a="row", layout_b="col", layout_c="row", out_type="f32", max_clusters=8)
    try:
        g.run_strided_batched(M, N, K, dA, probs[0].lda, M * probs[0].lda, dB, probs[0].ldb, N * probs[0].ldb,
                              dC, N, M * N, batch)
        assert g.query_status() == G.GEMM_OK
    finally:
        g.close()
    out = dC.cpu().numpy().astype(np.float64).reshape(batch, M, N)
    for i, p in enumerate(probs):
        assert_close(out[i], p.reference(), K, "f32", f"batch {i}")


def test_one_tile_wide_hints_through_a_column_major_c(G):
    # C column-major runs C^T = B^T A^T: a 1536 x 100 C becomes a launched 100 x 1536 grid one
    # tile tall, so the launched B (= A^T) streams evict-first and A (= B^T) stays evict-last.
    p = Problem(1536, 100, 1000, la="row", lb="row", lc="col", out="bf16", beta=0.5, seed=99)
    s, plan = G.gemm_plan(G.make_options(**options_for(p, block_n=128)), p.M, p.N, p.K, 1, 152)
    assert s == 0 and plan.transposed == 1 and (plan.l2_hint_a, plan.l2_hint_b) == (2, 1)
    got = _run(G, p, 1.0, 0.5, block_n=128)
    assert_close(got, p.reference(1.0, 0.5), p.K, "bf16", "one tile wide, column-major C")


@pytest.mark.parametrize("lb", ["row", "col"])
def test_multicast_mn_major_operands(G, lb):
    p = Problem(520, 700, 256, la="col", lb=lb, out="f32", seed=6)
    got = _run(G, p, mode="mcast", mcast_a=1, mcast_b=1, cluster_m=2, cluster_n=2)
    assert_close(got, p.reference(), 256, "f32", f"mn-major mcast lb={lb}")


@pytest.mark.parametrize("stages", [2, 3, 4])
def test_persistent_loop_and_stages(G, stages):
    # a handful of clusters walking many tiles, with a shallow ring
    p = Problem(1024, 1536, 640, seed=7)
    got = _run(G, p, max_clusters=3, stages=stages, mode="mcast", mcast_b=1, cluster_m=2)
    assert_close(got, p.reference(), 640, "bf16", f"persistent stages={stages}")


def test_k_zero_scales_c(G):
    import torch
    from dense_gemm_cluster_gb300 import inputs
    g = G.Gemm(0, out_type="f32", layout_b="row")
    C = torch.randn(40, 48, device="cuda")
    ref = (0.5 * C).cpu().numpy()
    g.run(40, 48, 0, None, 8, None, 48, C, 48, 1.0, 0.5)
    assert g.query_status() == G.GEMM_OK
    assert np.array_equal(C.cpu().numpy(), ref)
    C.fill_(float("nan"))
    g.run(40, 48, 0, None, 8, None, 48, C, 48, 1.0, 0.0)
    torch.cuda.synchronize()
    assert (C == 0).all().item()
    g.close()


@pytest.mark.parametrize("cm,cn,ma,mb", [(1, 1, 0, 0), (2, 1, 0, 1), (1, 4, 1, 0), (4, 2, 1, 1), (8, 1, 0, 1)])
@pytest.mark.parametrize("la,lb", [("row", "col"), ("col", "row")])
def test_128_wide_stages_single_cta_tiles(G, cm, cn, ma, mb, la, lb):
    # K = 576 = 4.5 stages of 128 (half-empty last stage); 128-wide tiles keep three stages
    p = Problem(900, 1000, 576, la=la, lb=lb, out="f32", seed=8)
    got = _run(G, p, mode="mcast", mcast_a=ma, mcast_b=mb, cluster_m=cm, cluster_n=cn, block_n=128, block_k=128)
    assert_close(got, p.reference(), 576, "f32", f"bk128 {cm}x{cn} A{ma} B{mb} {la}/{lb}")


@pytest.mark.parametrize("M,N,K,max_clusters,bn,out,beta", [
    (1000, 1100, 448, 5, 256, "bf16", 0.0),     # 5 clusters, 20 tiles: a 5-tile tail split by k-blocks
    (520, 384, 1024, 7, 128, "f32", 0.5),       # ragged tiles, beta read once by each finisher
    (256, 256, 2048, 3, 256, "bf16", 1.0),      # 2 tiles over 3 clusters: every tile split
    (129, 1000, 960, 6, 128, "f32", 0.0),       # many contributors per tile
    (1024, 128, 4096, 12, 128, "bf16", 0.0),    # 8 tiles spread over 12 clusters (more than half busy)
])
def test_stream_k_tail_matches_oracle(G, M, N, K, max_clusters, bn, out, beta):
    p = Problem(M, N, K, la="row", lb="col", out=out, beta=beta, seed=9)
    got = _run(G, p, 1.0, beta, schedule="stream_k", max_clusters=max_clusters, block_n=bn)
    assert_close(got, p.reference(1.0, beta), K, out, f"stream-K {M}x{N}x{K} on {max_clusters} clusters")


def test_stream_k_with_multicast_clusters_is_deterministic(G):
    p = Problem(1300, 1500, 704, la="col", lb="row", out="f32", seed=10)
    a = _run(G, p, schedule="stream_k", mode="mcast", mcast_a=1, mcast_b=1, cluster_m=2, cluster_n=2, max_clusters=9)
    b = _run(G, p, schedule="stream_k", mode="mcast", mcast_a=1, mcast_b=1, cluster_m=2, cluster_n=2, max_clusters=9)
    assert_close(a, p.reference(), 704, "f32", "stream-K 2x2 multicast")
    assert np.array_equal(a, b)          # partials are summed in a fixed order


@pytest.mark.parametrize("M,N,K,opts", [
    (300, 200, 8192, dict(block_n=128)),                                       # 6 tiles over 24 clusters
    (1024, 128, 4096, dict(block_n=128, mode="mcast", mcast_b=1, cluster_m=4)),  # 2 cluster tiles over 4
    (130, 1000, 3000, dict(block_n=256)),                                      # ragged K and tiles
])
def test_sub_wave_problem_spreads_over_more_clusters(G, M, N, K, opts):
    # Fewer tiles than clusters: the auto schedule splits k-blocks over more clusters
    # (at least 16 each); partials are summed in a fixed order, so reruns are bitwise equal.
    import torch
    s, plan = G.gemm_plan(G.make_options(layout_a="row", layout_b="row", out_type="f32", **opts), M, N, K, 1,
                          torch.cuda.get_device_properties(0).multi_processor_count)
    assert s == 0 and plan.clusters > plan.tiles and plan.stream_k_tiles == plan.tiles
    p = Problem(M, N, K, la="row", lb="row", out="f32", seed=11)
    a = _run(G, p, **opts)
    b = _run(G, p, **opts)
    assert_close(a, p.reference(), K, "f32", f"sub-wave {M}x{N}x{K} {opts}")
    assert np.array_equal(a, b)


@pytest.mark.parametrize("opts", [dict(schedule="stream_k", max_clusters=5, block_n=256),
                                  dict(mode="mcast", mcast_b=1, cluster_m=2)])
def test_gemm_replays_in_a_cuda_graph(G, opts):
    # A captured gemm_run replays correctly: stream-K partial flags are lowered by the
    # kernel itself, so no per-launch host state is frozen into the graph. Each replay
    # recomputes C (beta = 0) into a NaN-filled buffer.
    import torch
    from gpu_cases import torch_dev
    p = Problem(1000, 1100, 448, la="row", lb="col", out="f32", seed=22)
    g = G.Gemm(0, **options_for(p, **opts))
    try:
        dA, dB, dC = torch_dev(p.A), torch_dev(p.B), torch_dev(p.C_in)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):          # first run: workspace, flags, attributes, occupancy
            g.run(p.M, p.N, p.K, dA, p.lda, dB, p.ldb, dC, p.ldc, 1.0, 0.0, s)
        s.synchronize()
        assert g.query_status(s) == G.GEMM_OK
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            g.run(p.M, p.N, p.K, dA, p.lda, dB, p.ldb, dC, p.ldc, 1.0, 0.0, s)
        ref = p.reference()
        for rep in range(3):
            dC.fill_(float("nan"))
            graph.replay()
            torch.cuda.synchronize()
            assert_close(p.result(dC), ref, p.K, "f32", f"graph replay {rep} {opts}")
        assert g.query_status() == G.GEMM_OK
    finally:
        g.close()


@pytest.mark.parametrize("shared", ["A", "B"])
@pytest.mark.parametrize("opts", [dict(), dict(mode="mcast", mcast_a=1, mcast_b=1, cluster_m=2, cluster_n=2),
                                  dict(cta_group=2, cluster_m=2)])
def test_batch_stride_zero_shares_one_matrix(G, shared, opts):
    # strideA (or strideB) = 0: every product of the batch reads the same matrix.
    import torch
    from gpu_cases import torch_dev
    M, N, K, batch = 300, 260, 192, 3
    probs = [Problem(M, N, K, la="row", lb="col", out="f32", seed=70 + i) for i in range(batch)]
    for p in probs[1:]:
        if shared == "A":
            p.A = probs[0].A
        else:
            p.B = probs[0].B
    A = np.concatenate([probs[0].A.reshape(-1)] if shared == "A" else [p.A.reshape(-1) for p in probs])
    B = np.concatenate([probs[0].B.reshape(-1)] if shared == "B" else [p.B.reshape(-1) for p in probs])
    sA = 0 if shared == "A" else probs[0].A.size
    sB = 0 if shared == "B" else probs[0].B.size
    lda, ldb, ldc = probs[0].lda, probs[0].ldb, probs[0].ldc
    sC = probs[0].C_in.size
    dC = torch.full((batch * sC,), float("nan"), dtype=torch.float32, device="cuda")
    g = G.Gemm(0, **options_for(probs[0], **opts))
    try:
        g.run_strided_batched(M, N, K, torch_dev(A), lda, sA, torch_dev(B), ldb, sB, dC, ldc, sC, batch)
        assert g.query_status() == G.GEMM_OK
        # overlapping (non-zero, shorter than one matrix) strides are refused before any launch
        s = G.gemm_run_strided_batched(g.handle, M, N, K, torch_dev(A), lda, 16, torch_dev(B), ldb, sB, dC, ldc, sC,
                                       batch, 1.0, 0.0)
        assert s == G.GEMM_ERR_INVALID_ARG
    finally:
        g.close()
    out = dC.cpu().numpy()
    for i, p in enumerate(probs):
        assert_close(decode(out[i * sC:(i + 1) * sC].reshape(M, ldc), M, N, "row"), p.reference(), K, "f32",
                     f"stride 0 on {shared}, product {i}")


@pytest.mark.parametrize("opts", [dict(mode="mcast", mcast_b=1, cluster_m=2),
                                  dict(schedule="stream_k", max_clusters=7, block_n=128),
                                  dict(cta_group=2, cluster_m=2)])
def test_back_to_back_launches_read_the_previous_result(G, opts):
    # Launches overlap their prologue with the previous kernel (programmatic dependent
    # launch); each must still read what the previous one wrote. A chain of GEMMs, each
    # taking the previous output as its A, runs once back to back on one stream and once
    # with a device synchronisation between launches: the results must be bitwise equal.
    import torch
    from gpu_cases import torch_dev
    M, K = 700, 512
    dims = [512, 384, 640, 512]
    Bs = [torch_dev(inputs_bf16(K if i == 0 else dims[i - 1], dims[i], 90 + i)) for i in range(len(dims))]
    A0 = torch_dev(inputs_bf16(M, K, 89))

    def chain(sync):
        g = G.Gemm(0, layout_a="row", layout_b="row", layout_c="row", out_type="bf16", **opts)
        try:
            a, outs = A0, []
            for i, b in enumerate(Bs):
                k = K if i == 0 else dims[i - 1]
                c = torch.empty(M * dims[i], dtype=torch.int16, device="cuda")
                g.run(M, dims[i], k, a, k, b, dims[i], c, dims[i], 1.0 / 16.0, 0.0)
                if sync:
                    torch.cuda.synchronize()
                outs.append(c)
                a = c
            assert g.query_status() == G.GEMM_OK
        finally:
            g.close()
        return [o.cpu().numpy() for o in outs]

    for x, y in zip(chain(False), chain(True)):
        assert np.array_equal(x, y)
    assert np.isfinite(decode(chain(False)[-1].view(np.uint16).reshape(M, dims[-1]), M, dims[-1], "row")).all()


def inputs_bf16(rows, cols, seed):
    from dense_gemm_cluster_gb300 import inputs
    buf, _ = inputs.store(inputs.bf16_matrix(rows, cols, "normal", seed), "row")
    return buf


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (1, 700, 96), (700, 1, 96), (5, 3, 4100), (2, 2, 8)])
@pytest.mark.parametrize("opts", [dict(mode="mcast", mcast_a=1, mcast_b=1, cluster_m=2, cluster_n=2),
                                  dict(cta_group=2, cluster_m=4, mode="mcast", mcast_b=1),
                                  dict(mode="mcast", mcast_b=1, cluster_m=8),
                                  dict(schedule="clc", mode="mcast", mcast_a=1, cluster_n=2)])
def test_degenerate_shapes_in_every_sharing_mode(G, M, N, K, opts):
    # One row, one column, or a tiny output with a long K: a cluster's other CTAs (and a
    # pair's odd CTA) hold only out-of-range rows and columns and must still take part.
    p = Problem(M, N, K, la="row", lb="col", out="f32", beta=0.5, seed=80)
    got = _run(G, p, 1.0, 0.5, **opts)
    assert_close(got, p.reference(1.0, 0.5), K, "f32", f"{M}x{N}x{K} {opts}")


@pytest.mark.parametrize("K,stages,out", [
    (8192, 2, "bf16"),    # one tile over 8 clusters: 7 partials do not fit in the staging region
    (3072, 2, "bf16"),    # 2 partials staged one column chunk per pass
    (3072, 4, "f32"),     # 2 partials staged 6 column chunks, then 2
])
def test_stream_k_finisher_staging_paths(G, K, stages, out):
    # A sub-wave problem: one 128 x 256 tile whose k-blocks are split over several
    # clusters; the finisher adds the others' partials from staged shared memory, a
    # pass at a time, or straight from global memory when they do not fit.
    p = Problem(128, 256, K, la="row", lb="col", out=out, beta=0.5, seed=85)
    a = _run(G, p, 1.0, 0.5, stages=stages)
    b = _run(G, p, 1.0, 0.5, stages=stages)
    assert_close(a, p.reference(1.0, 0.5), K, out, f"finisher staging K={K} stages={stages}")
    assert np.array_equal(a, b)


@pytest.mark.parametrize("opts", [
    dict(max_clusters=10),                                                    # single CTAs
    dict(mode="mcast", mcast_b=1, cluster_m=2, max_clusters=5),               # 2x1 clusters
    dict(cta_group=2, cluster_m=2, max_clusters=5),                           # pairs
])
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_stream_k_finisher_followed_by_whole_tiles(G, opts, out):
    # 1024 x 1536 is 48 tiles of 128 x 256 (24 cluster tiles of 256 x 256): on 10 (or 5)
    # clusters three whole waves run and the last 1.8 waves' tiles are split by k-blocks,
    # 1.8 tiles' worth per cluster, so ranges start and end inside tiles. Each cluster
    # runs its split pieces first: a finisher adds its contributors' partials from global
    # memory while the whole tiles after it stream through the operand ring.
    p = Problem(1024, 1536, 1000, la="row", lb="col", out=out, beta=0.5, seed=95)
    a = _run(G, p, 1.0, 0.5, schedule="stream_k", **opts)
    b = _run(G, p, 1.0, 0.5, schedule="stream_k", **opts)
    assert_close(a, p.reference(1.0, 0.5), 1000, out, f"stream-K with whole tiles after {opts}")
    assert np.array_equal(a, b)
    s, plan = G.gemm_plan(G.make_options(layout_a="row", layout_b="col", out_type=out, schedule="stream_k", **opts),
                          1024, 1536, 1000, 1, 152)
    kb = -(-1000 // plan.block_k)
    assert s == 0 and 0 < plan.stream_k_tiles < plan.tiles
    assert (plan.stream_k_tiles * kb) % plan.clusters != 0 or (plan.stream_k_tiles * kb // plan.clusters) % kb != 0
