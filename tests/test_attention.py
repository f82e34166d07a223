"""GPU parity of the fused attention forward against the fp64 oracle.

O is a convex combination of V rows; P is rounded to bf16 before P V, so the
bound is 1e-2 * max|V| (about four bf16 roundings); the log-sum-exp is
accumulated in fp32 from unrounded probabilities and held to 1e-4 relative.
K/V multicast only moves data: clusters of 2 and 4 must equal cluster 1 bit
for bit.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _inputs(b, sq, sk, seed, k_growth=0.0, d=128):
    from dense_gemm_cluster_gb300 import inputs
    Q = inputs.bf16_matrix(b * sq, d, "normal", seed).reshape(b, sq, d)
    Kf = inputs.bf16_bits_to_f32(inputs.bf16_matrix(b * sk, d, "normal", seed + 1)).reshape(b, sk, d).astype(np.float64)
    if k_growth:
        # keys grow along the sequence so each key tile raises the row max
        Kf = Kf * (1.0 + k_growth * np.arange(sk)[None, :, None] / sk)
    K = inputs.f64_to_bf16_bits(Kf).reshape(b, sk, d)
    V = inputs.bf16_matrix(b * sk, d, "normal", seed + 2).reshape(b, sk, d)
    return Q, K, V


def _run(Q, K, V, cluster, out_f32=0, scale=0.0, cta_group=1, causal=False):
    import torch
    from dense_gemm_cluster_gb300 import gemm
    b, sq, d = Q.shape
    sk = K.shape[1]
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
    O = torch.full((b * sq * d,), float("nan"), dtype=torch.float32 if out_f32 else torch.bfloat16, device="cuda")
    lse = torch.full((b * sq,), float("nan"), dtype=torch.float32, device="cuda")
    s = gemm.attention_forward_run(dev(Q), dev(K), dev(V), O, lse, b, sq, sk, d, scale, out_f32, cluster, cta_group,
                                   causal=causal)
    assert s == gemm.GEMM_OK
    assert gemm.attention_forward_query_status() == gemm.GEMM_OK
    o = O.float().cpu().numpy().reshape(b, sq, d).astype(np.float64)
    return o, lse.cpu().numpy().reshape(b, sq).astype(np.float64)


MODES = [(1, 1), (2, 1), (4, 1), (2, 2)]          # (cluster, cta_group)


@pytest.mark.parametrize("b,sq,sk", [(2, 128, 128), (3, 300, 500), (1, 1000, 130), (2, 256, 2048), (1, 77, 1),
                                    (3, 1, 1), (2, 1, 300), (1, 257, 129)])
@pytest.mark.parametrize("cluster,cta_group", MODES)
def test_attention_matches_oracle(b, sq, sk, cluster, cta_group):
    import oracle
    from dense_gemm_cluster_gb300 import inputs
    Q, K, V = _inputs(b, sq, sk, 100 + sq)
    o, lse = _run(Q, K, V, cluster, cta_group=cta_group)
    ref, ref_lse = oracle.attention_forward(Q, K, V, with_lse=True)
    vmax = float(np.max(np.abs(inputs.bf16_bits_to_f32(V))))
    assert np.isfinite(o).all()
    assert np.max(np.abs(o - ref)) <= 1e-2 * vmax
    assert np.max(np.abs(lse - ref_lse) / (1.0 + np.abs(ref_lse))) <= 1e-4


@pytest.mark.parametrize("cta_group", [1, 2])
def test_attention_rescales_when_the_row_max_grows(cta_group):
    import oracle
    from dense_gemm_cluster_gb300 import inputs
    Q, K, V = _inputs(2, 256, 1024, 7, k_growth=3.0)
    for scale in (0.0, 0.35):
        o, lse = _run(Q, K, V, 2, out_f32=1, scale=scale, cta_group=cta_group)
        ref, ref_lse = oracle.attention_forward(Q, K, V, scale=scale if scale else None, with_lse=True)
        vmax = float(np.max(np.abs(inputs.bf16_bits_to_f32(V))))
        assert np.max(np.abs(o - ref)) <= 1e-2 * vmax
        assert np.max(np.abs(lse - ref_lse) / (1.0 + np.abs(ref_lse))) <= 1e-4


def test_attention_sharing_modes_are_bit_identical():
    # multicast only moves data; the pair MMA splits each 256-row product across two SMs
    # but sums the same products in the same order
    Q, K, V = _inputs(2, 512, 640, 9)
    base, base_lse = _run(Q, K, V, 1, out_f32=1)
    for c, g in MODES[1:]:
        o, lse = _run(Q, K, V, c, out_f32=1, cta_group=g)
        assert np.array_equal(o, base) and np.array_equal(lse, base_lse), (c, g)


def test_attention_argument_errors():
    import torch
    from dense_gemm_cluster_gb300 import gemm
    x = torch.zeros(128 * 128, dtype=torch.int16, device="cuda")
    assert gemm.attention_forward_run(x, x, x, x, None, 1, 128, 128, 96) == gemm.GEMM_ERR_UNSUPPORTED
    assert gemm.attention_forward_run(x, x, x, x, None, 1, 128, 128, 64, 0.0, 0, 2, 2) == gemm.GEMM_ERR_UNSUPPORTED
    assert gemm.attention_forward_run(x, x, x, x, None, 1, 128, 128, 128, 0.0, 0, 3) == gemm.GEMM_ERR_UNSUPPORTED
    assert gemm.attention_forward_run(x, x, x, x, None, 1, 128, 128, 128, 0.0, 0, 4, 2) == gemm.GEMM_ERR_UNSUPPORTED
    assert gemm.attention_forward_run(x, x, x, x, None, 1, 128, 128, 128, 0.0, 0, 2, 3) == gemm.GEMM_ERR_UNSUPPORTED
    assert gemm.attention_forward_run(x, x, x, x, None, 1, 128, 0, 128) == gemm.GEMM_ERR_INVALID_ARG
    assert gemm.attention_forward_run(x.data_ptr() + 2, x, x, x, None, 1, 128, 128, 128) == gemm.GEMM_ERR_ALIGNMENT


def test_attention_row_max_sees_every_column():
    # Query row r and key k share a large component when r = k (mod 128): every row has
    # a score of ~200 (base 2) at column r mod 128 of each key tile and ~0 elsewhere.
    # Over a tile's 128 rows the spike visits every column; a row max that missed a
    # column would leave 2^(~200) in P, which overflows fp32.
    import oracle
    from dense_gemm_cluster_gb300 import inputs
    b, sq, sk, d = 1, 256, 512, 128
    amp = float(np.sqrt(200.0 / np.log2(np.e)))
    noise = lambda rows, seed: inputs.bf16_bits_to_f32(inputs.bf16_matrix(rows, d, "normal", seed)).astype(np.float64) * 0.05
    eye = lambda rows: np.eye(d)[np.arange(rows) % d] * amp
    Q = inputs.f64_to_bf16_bits(eye(sq) + noise(sq, 31)).reshape(b, sq, d)
    K = inputs.f64_to_bf16_bits(eye(sk) + noise(sk, 32)).reshape(b, sk, d)
    V = inputs.bf16_matrix(sk, d, "normal", 33).reshape(b, sk, d)
    for cluster, g in ((1, 1), (2, 1), (2, 2)):
        o, lse = _run(Q, K, V, cluster, out_f32=1, scale=1.0, cta_group=g)
        ref, ref_lse = oracle.attention_forward(Q, K, V, scale=1.0, with_lse=True)
        assert np.isfinite(o).all() and np.isfinite(lse).all()
        vmax = float(np.max(np.abs(inputs.bf16_bits_to_f32(V))))
        assert np.max(np.abs(o - ref)) <= 1e-2 * vmax
        assert np.max(np.abs(lse - ref_lse) / (1.0 + np.abs(ref_lse))) <= 1e-4


def test_attention_more_query_blocks_than_sms():
    # 320 CTAs (160 heads x 2 query blocks, one ragged) on 152 SMs, ragged key tiles
    # and rescales of the reference max; clusters of 2 and 4 must equal cluster 1.
    import oracle
    from dense_gemm_cluster_gb300 import inputs
    Q, K, V = _inputs(160, 300, 640, 41, k_growth=2.0)
    ref, ref_lse = oracle.attention_forward(Q, K, V, with_lse=True)
    vmax = float(np.max(np.abs(inputs.bf16_bits_to_f32(V))))
    base = None
    for cluster, g in MODES:
        o, lse = _run(Q, K, V, cluster, out_f32=1, cta_group=g)
        assert np.isfinite(o).all()
        assert np.max(np.abs(o - ref)) <= 1e-2 * vmax, f"cluster {cluster} cta_group {g}"
        assert np.max(np.abs(lse - ref_lse) / (1.0 + np.abs(ref_lse))) <= 1e-4
        if base is None:
            base = (o, lse)
        else:
            assert np.array_equal(o, base[0]) and np.array_equal(lse, base[1])


@pytest.mark.parametrize("cluster,cta_group", [(2, 1), (2, 2)])
def test_attention_replays_in_a_cuda_graph(cluster, cta_group):
    import torch
    import oracle
    from dense_gemm_cluster_gb300 import gemm, inputs
    Q, K, V = _inputs(2, 300, 500, 51)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
    dQ, dK, dV = dev(Q), dev(K), dev(V)
    O = torch.empty(2 * 300 * 128, dtype=torch.float32, device="cuda")
    lse = torch.empty(2 * 300, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    args = (dQ, dK, dV, O, lse, 2, 300, 500, 128, 0.0, 1, cluster, cta_group)
    with torch.cuda.stream(s):                      # first call sets the kernel's attributes
        assert gemm.attention_forward_run(*args, stream=s) == gemm.GEMM_OK
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        assert gemm.attention_forward_run(*args, stream=s) == gemm.GEMM_OK
    ref, ref_lse = oracle.attention_forward(Q, K, V, with_lse=True)
    vmax = float(np.max(np.abs(inputs.bf16_bits_to_f32(V))))
    for _ in range(3):
        O.fill_(float("nan"))
        lse.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        o = O.cpu().numpy().reshape(2, 300, 128).astype(np.float64)
        assert np.max(np.abs(o - ref)) <= 1e-2 * vmax
        assert np.max(np.abs(lse.cpu().numpy().reshape(2, 300) - ref_lse) / (1.0 + np.abs(ref_lse))) <= 1e-4
    assert gemm.attention_forward_query_status() == gemm.GEMM_OK


@pytest.mark.parametrize("b,sq,sk,cluster,cta_group,with_lse", [
    (10, 300, 500, 2, 1, True),       # 5 parts of 2 heads
    (11, 301, 257, 1, 1, True),       # sq odd: parts of 4 heads keep each lse view 16-byte aligned
    (9, 258, 130, 2, 2, False),       # sq even, not a multiple of 4: parts of 2 heads; no lse
    (1, 128, 128, 4, 1, True),        # a single part
])
def test_attention_host_entry_equals_device_entry(b, sq, sk, cluster, cta_group, with_lse):
    # attention_forward_run_host copies host Q, K, V into the workspace part by part and
    # runs the same kernel on each part, so it must equal the device entry bit for bit.
    import torch
    from dense_gemm_cluster_gb300 import gemm
    Q, K, V = _inputs(b, sq, sk, 300 + sq)
    ref_o, ref_lse = _run(Q, K, V, cluster, out_f32=1, cta_group=cta_group)
    O_h = np.full(b * sq * 128, np.nan, dtype=np.float32)
    lse_h = np.full(b * sq, np.nan, dtype=np.float32) if with_lse else None
    ws_bytes = gemm.attention_forward_host_workspace_bytes(b, sq, sk, 128, 1)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    host = lambda a: np.ascontiguousarray(a).view(np.int16)
    s = gemm.attention_forward_run_host(host(Q), host(K), host(V), O_h, lse_h, b, sq, sk, 128, ws, ws_bytes, 0.0, 1,
                                        cluster, cta_group)
    assert s == gemm.GEMM_OK
    assert np.array_equal(O_h.reshape(b, sq, 128).astype(np.float64), ref_o)
    if with_lse:
        assert np.array_equal(lse_h.reshape(b, sq).astype(np.float64), ref_lse)


def test_attention_more_heads_than_one_grid_dimension_holds():
    # 70000 heads of 8 queries and 8 keys: the heads continue in grid z past 65535.
    import torch
    import oracle
    from dense_gemm_cluster_gb300 import gemm, inputs
    b, sq, sk = 70000, 8, 8
    Q, K, V = _inputs(b, sq, sk, 500)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
    O = torch.full((b * sq * 128,), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((b * sq,), float("nan"), dtype=torch.float32, device="cuda")
    assert gemm.attention_forward_run(dev(Q), dev(K), dev(V), O, lse, b, sq, sk, 128, 0.0, 1, 2, 1) == gemm.GEMM_OK
    assert gemm.attention_forward_query_status() == gemm.GEMM_OK
    o = O.cpu().numpy().reshape(b, sq, 128).astype(np.float64)
    l = lse.cpu().numpy().reshape(b, sq).astype(np.float64)
    assert np.isfinite(o).all() and np.isfinite(l).all()
    heads = np.array([0, 1, 65534, 65535, 65536, 69999])
    ref, ref_lse = oracle.attention_forward(Q[heads], K[heads], V[heads], with_lse=True)
    vmax = float(np.max(np.abs(inputs.bf16_bits_to_f32(V[heads]))))
    assert np.max(np.abs(o[heads] - ref)) <= 1e-2 * vmax
    assert np.max(np.abs(l[heads] - ref_lse) / (1.0 + np.abs(ref_lse))) <= 1e-4


@pytest.mark.parametrize("b,sq,sk", [(2, 256, 256), (1, 300, 500), (1, 700, 300), (3, 1000, 1000), (1, 129, 1),
                                    (2, 1300, 1300)])
@pytest.mark.parametrize("cluster,cta_group", MODES)
@pytest.mark.parametrize("out_f32", [0, 1])
def test_causal_attention_matches_oracle(b, sq, sk, cluster, cta_group, out_f32):
    # Query i attends keys 0..i: diagonal tiles are masked row by row, a cluster stops at
    # the key tiles its last query needs, and query blocks run last-first.
    import oracle
    from dense_gemm_cluster_gb300 import inputs
    Q, K, V = _inputs(b, sq, sk, 700 + sq)
    o, lse = _run(Q, K, V, cluster, out_f32=out_f32, cta_group=cta_group, causal=True)
    ref, ref_lse = oracle.attention_forward(Q, K, V, with_lse=True, causal=True)
    vmax = float(np.max(np.abs(inputs.bf16_bits_to_f32(V))))
    assert np.isfinite(o).all()
    assert np.max(np.abs(o - ref)) <= 1e-2 * vmax
    assert np.max(np.abs(lse - ref_lse) / (1.0 + np.abs(ref_lse))) <= 1e-4


def test_causal_sharing_modes_are_bit_identical():
    Q, K, V = _inputs(2, 900, 900, 19)
    base, base_lse = _run(Q, K, V, 1, out_f32=1, causal=True)
    for c, g in MODES[1:]:
        o, lse = _run(Q, K, V, c, out_f32=1, cta_group=g, causal=True)
        assert np.array_equal(o, base) and np.array_equal(lse, base_lse), (c, g)


MODES_D64 = [(1, 1), (2, 1), (4, 1)]      # the pair MMA needs d = 128


@pytest.mark.parametrize("b,sq,sk", [(2, 128, 128), (3, 300, 500), (1, 1000, 130), (1, 77, 1), (2, 1, 300)])
@pytest.mark.parametrize("cluster,cta_group", MODES_D64)
@pytest.mark.parametrize("causal", [False, True])
def test_head_dim_64_matches_oracle(b, sq, sk, cluster, cta_group, causal):
    # d = 64: one 128-byte swizzle atom per row of Q, K and V; the same kernel otherwise
    import oracle
    from dense_gemm_cluster_gb300 import inputs
    Q, K, V = _inputs(b, sq, sk, 900 + sq, d=64)
    o, lse = _run(Q, K, V, cluster, out_f32=1, cta_group=cta_group, causal=causal)
    ref, ref_lse = oracle.attention_forward(Q, K, V, with_lse=True, causal=causal)
    vmax = float(np.max(np.abs(inputs.bf16_bits_to_f32(V))))
    assert np.isfinite(o).all()
    assert np.max(np.abs(o - ref)) <= 1e-2 * vmax
    assert np.max(np.abs(lse - ref_lse) / (1.0 + np.abs(ref_lse))) <= 1e-4


def test_head_dim_64_rescales_and_modes_are_bit_identical():
    import oracle
    from dense_gemm_cluster_gb300 import inputs
    Q, K, V = _inputs(2, 512, 1024, 31, k_growth=3.0, d=64)
    base, base_lse = _run(Q, K, V, 1, out_f32=1, scale=0.2)
    ref, ref_lse = oracle.attention_forward(Q, K, V, scale=0.2, with_lse=True)
    vmax = float(np.max(np.abs(inputs.bf16_bits_to_f32(V))))
    assert np.max(np.abs(base - ref)) <= 1e-2 * vmax
    assert np.max(np.abs(base_lse - ref_lse) / (1.0 + np.abs(ref_lse))) <= 1e-4
    for c, g in MODES_D64[1:]:
        o, lse = _run(Q, K, V, c, out_f32=1, scale=0.2, cta_group=g)
        assert np.array_equal(o, base) and np.array_equal(lse, base_lse), (c, g)


def test_head_dim_64_host_entry_equals_device_entry():
    import torch
    from dense_gemm_cluster_gb300 import gemm
    b, sq, sk = 3, 300, 500
    Q, K, V = _inputs(b, sq, sk, 41, d=64)
    ref_o, ref_lse = _run(Q, K, V, 2, out_f32=1, causal=True)
    host = lambda a: np.ascontiguousarray(a).view(np.int16)
    O_h = np.full(b * sq * 64, np.nan, dtype=np.float32)
    lse_h = np.full(b * sq, np.nan, dtype=np.float32)
    ws_bytes = gemm.attention_forward_host_workspace_bytes(b, sq, sk, 64, 1)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    s = gemm.attention_forward_run_host(host(Q), host(K), host(V), O_h, lse_h, b, sq, sk, 64, ws, ws_bytes, 0.0, 1,
                                        2, 1, causal=1)
    assert s == gemm.GEMM_OK
    assert np.array_equal(O_h.reshape(b, sq, 64).astype(np.float64), ref_o)
    assert np.array_equal(lse_h.reshape(b, sq).astype(np.float64), ref_lse)
