"""Pins for the CPU oracle: closed forms, invariants and exact brute force.

Each case is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign, a swapped index, a transposed operand, a wrong layout offset, beta
applied when it should not be) fails at least one of them. None of these tests
retypes the oracle's own formula: they compare it with facts that hold by
construction (identity, permutation, all-ones, rank one), with exact rational
arithmetic, or with an independent library routine.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from dense_gemm_cluster_gb300 import inputs

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def bf16(rows, cols, seed, dist="normal", scale=1.0):
    return inputs.bf16_matrix(rows, cols, dist, seed, scale)


def val(bits):
    return inputs.bf16_bits_to_f32(bits).astype(np.float64)


def eye_bf16(n):
    return inputs.f64_to_bf16_bits(np.eye(n))


def perm_bf16(perm):
    n = len(perm)
    P = np.zeros((n, n))
    P[np.arange(n), perm] = 1.0          # row i of P selects column perm[i]
    return inputs.f64_to_bf16_bits(P)


def run(A_log, B_log, la="row", lb="row", alpha=1.0, beta=0.0, C_log=None, lc="row"):
    M, K = A_log.shape
    N = B_log.shape[1]
    A, lda = inputs.store(A_log, la)
    B, ldb = inputs.store(B_log, lb)
    if C_log is not None:
        C, ldc = inputs.store(C_log, lc, ld=None if C_log.dtype == np.uint16 else max(4, (C_log.shape[1 if lc == "row" else 0] + 3) // 4 * 4))
    else:
        C, ldc = None, 0
    return oracle.gemm(M, N, K, A, lda, la, B, ldb, lb, alpha, beta, C, ldc, lc)


@pytest.mark.parametrize("la,lb", [("row", "row"), ("row", "col"), ("col", "row"), ("col", "col")])
def test_identity_left_is_exact(la, lb):
    B = bf16(48, 37, seed=11)
    C = run(eye_bf16(48), B, la, lb)
    assert np.array_equal(C, val(B))


@pytest.mark.parametrize("la,lb", [("row", "col"), ("col", "row")])
def test_identity_right_is_exact(la, lb):
    A = bf16(29, 40, seed=12)
    C = run(A, eye_bf16(40), la, lb)
    assert np.array_equal(C, val(A))


def test_permutation_left_permutes_rows():
    rng = np.random.default_rng(3)
    perm = rng.permutation(32)
    assert not np.array_equal(perm, np.argsort(perm))  # not an involution: a transpose would show
    B = bf16(32, 21, seed=13)
    C = run(perm_bf16(perm), B, "row", "col")
    assert np.array_equal(C, val(B)[perm])


def test_permutation_right_permutes_columns():
    rng = np.random.default_rng(4)
    perm = rng.permutation(24)
    A = bf16(19, 24, seed=14)
    P = perm_bf16(perm)                  # (A P)[:, j] = A[:, q] where P[q, j] = 1
    C = run(A, P, "col", "row")
    inv = np.empty_like(perm)
    inv[perm] = np.arange(24)
    assert np.array_equal(C, val(A)[:, inv])


def test_all_ones_gives_column_sums():
    K = 256
    B = bf16(K, 33, seed=15)
    C = run(bf16(7, K, seed=0, dist="ones"), B, "row", "row")
    sums = np.array([math.fsum(col) for col in val(B).T])  # correctly rounded sums
    for i in range(7):
        assert np.array_equal(C[i], sums)


def test_rank_one_is_exact_outer_product():
    u = bf16(23, 1, seed=16)
    v = bf16(1, 31, seed=17)
    C = run(u, v, "row", "col", alpha=0.5)
    assert np.array_equal(C, 0.5 * np.outer(val(u)[:, 0], val(v)[0]))


def test_alpha_zero_gives_scaled_c_exactly():
    A = bf16(9, 16, seed=18)
    B = bf16(16, 11, seed=19)
    Cin = bf16(9, 11, seed=20)
    C = run(A, B, alpha=0.0, beta=-0.75, C_log=Cin)
    assert np.array_equal(C, -0.75 * val(Cin))


def test_beta_zero_never_reads_c():
    A = bf16(9, 16, seed=21)
    B = bf16(16, 11, seed=22)
    nan_c = np.full((9, 11), np.nan, dtype=np.float32)
    C = run(A, B, beta=0.0, C_log=nan_c)
    assert np.isfinite(C).all()


def test_fp32_c_in_is_read_as_float32():
    A = bf16(5, 8, seed=23)
    B = bf16(8, 6, seed=24)
    Cin = inputs.f32_matrix(5, 6, "normal", seed=25)
    ref = run(A, B) + 2.0 * Cin.astype(np.float64)
    got = run(A, B, beta=2.0, C_log=Cin)
    assert np.allclose(got, ref, rtol=0, atol=1e-12)


def exact_gemm(A_log, B_log, alpha, beta, C_log):
    Av = val(A_log)
    Bv = val(B_log)
    M, K = Av.shape
    N = Bv.shape[1]
    out = [[None] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            s = sum((Fraction(float(Av[i, k])) * Fraction(float(Bv[k, j])) for k in range(K)), Fraction(0))
            r = Fraction(alpha) * s
            if beta != 0.0:
                r += Fraction(beta) * Fraction(float(val(C_log)[i, j]))
            out[i][j] = r
    return out


@pytest.mark.parametrize("trial", range(12))
def test_brute_force_rational_tiny(trial):
    rng = np.random.default_rng(100 + trial)
    M, N, K = (int(x) for x in rng.integers(1, 9, size=3))
    la, lb, lc = (("row", "col")[int(b)] for b in rng.integers(0, 2, size=3))
    alpha = float(rng.choice([1.0, -0.5, 0.375, 3.0]))
    beta = float(rng.choice([0.0, 1.0, 0.5, -2.0]))
    A = bf16(M, K, seed=200 + trial)
    B = bf16(K, N, seed=300 + trial)
    Cin = bf16(M, N, seed=400 + trial)
    got = run(A, B, la, lb, alpha, beta, Cin, lc)
    ref = exact_gemm(A, B, alpha, beta, Cin)
    Av, Bv, Cv = val(A), val(B), val(Cin)
    for i in range(M):
        for j in range(N):
            mag = abs(alpha) * float(np.abs(Av[i]) @ np.abs(Bv[:, j])) + abs(beta) * abs(Cv[i, j])
            bound = (K + 2) * 2.0 ** -53 * mag
            assert abs(Fraction(float(got[i, j])) - ref[i][j]) <= Fraction(bound)


@pytest.mark.parametrize("shape", [(100, 70, 300), (64, 129, 257)])
def test_matches_numpy_float64_matmul(shape):
    M, N, K = shape
    A = bf16(M, K, seed=31, dist="uniform")
    B = bf16(K, N, seed=32, dist="uniform")
    got = run(A, B, "row", "col")
    ref = val(A) @ val(B)
    scale = np.abs(val(A)) @ np.abs(val(B))
    assert np.all(np.abs(got - ref) <= 2 * K * 2.0 ** -53 * scale)


def test_layouts_give_identical_bits():
    A = bf16(37, 45, seed=41)
    B = bf16(45, 29, seed=42)
    outs = [run(A, B, la, lb) for la in ("row", "col") for lb in ("row", "col")]
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def test_padded_leading_dimension_is_respected():
    A = bf16(13, 10, seed=43)
    B = bf16(10, 7, seed=44)
    Ab, lda = inputs.store(A, "row", ld=24)
    Ab[:, 10:] = inputs.f64_to_bf16_bits(np.full((13, 14), 1e4))  # garbage in the padding
    Bb, ldb = inputs.store(B, "col", ld=16)
    got = oracle.gemm(13, 7, 10, Ab, lda, "row", Bb, ldb, "col")
    assert np.array_equal(got, run(A, B))


def test_entries_match_full_product_and_rationals():
    A = bf16(6, 5, seed=51)
    B = bf16(5, 4, seed=52)
    Cin = bf16(6, 4, seed=53)
    Ab, lda = inputs.store(A, "row")
    Bb, ldb = inputs.store(B, "row")
    Cb, ldc = inputs.store(Cin, "row")
    rows = np.array([0, 5, 3, 2, 5])
    cols = np.array([0, 3, 1, 2, 0])
    got = oracle.gemm_entries(rows, cols, 5, Ab, lda, "row", Bb, ldb, "row", 1.5, 0.5, Cb, ldc)
    ref = exact_gemm(A, B, 1.5, 0.5, Cin)
    for t in range(len(rows)):
        assert abs(Fraction(float(got[t])) - ref[rows[t]][cols[t]]) <= Fraction(1, 2 ** 40)
    full = oracle.gemm(6, 4, 5, Ab, lda, "row", Bb, ldb, "row", 1.5, 0.5, Cb, ldc)
    assert np.array_equal(got, full[rows, cols])


def test_attention_scores_with_identity_keys_returns_queries():
    d = 16
    Q = np.stack([bf16(10, d, seed=60 + b) for b in range(3)])
    Kmat = np.stack([eye_bf16(d)] * 3)
    S = oracle.attention_scores(Q, Kmat)
    assert np.array_equal(S, val(Q))


def test_attention_scores_rational_and_per_batch():
    Q = np.stack([bf16(4, 6, seed=70 + b) for b in range(2)])
    Kmat = np.stack([bf16(5, 6, seed=80 + b) for b in range(2)])
    S = oracle.attention_scores(Q, Kmat)
    for b in range(2):
        ref = exact_gemm(Q[b], Kmat[b].T.copy(), 1.0, 0.0, None)
        for i in range(4):
            for j in range(5):
                assert abs(Fraction(float(S[b, i, j])) - ref[i][j]) <= Fraction(1, 2 ** 40)
    # batches must not mix: swapping the key batches swaps the results
    S2 = oracle.attention_scores(Q, Kmat[::-1].copy())
    assert not np.array_equal(S2[0], S[0])


def test_empty_shapes():
    A = np.zeros((0, 8), dtype=np.uint16)
    B = bf16(8, 8, seed=90)
    assert oracle.gemm(0, 8, 8, A, 8, "row", B, 8, "row").shape == (0, 8)
    z = oracle.gemm(3, 4, 0, np.zeros((3, 8), np.uint16), 8, "row", np.zeros((0, 8), np.uint16), 8, "row")
    assert np.array_equal(z, np.zeros((3, 4)))


# ---------------------------------------------------------------- 1-D stencil pins
def test_stencil_constant_and_linear_interiors_are_exact():
    c = np.full(50, 3.5, dtype=np.float32)
    y = oracle.stencil_1d(c)
    assert np.array_equal(y[1:-1], np.full(48, 3.5))
    assert y[0] == y[-1] == 0.75 * 3.5                 # one neighbour is outside: counts as zero
    lin = np.arange(40, dtype=np.float32)
    y = oracle.stencil_1d(lin)
    assert np.array_equal(y[1:-1], np.arange(1, 39, dtype=np.float64))   # a linear ramp is reproduced
    assert y[-1] == 0.25 * 38 + 0.5 * 39


def test_stencil_impulse_response_is_quarter_half_quarter():
    x = np.zeros(9, dtype=np.float32)
    x[4] = 8.0
    assert list(oracle.stencil_1d(x)) == [0, 0, 0, 2.0, 4.0, 2.0, 0, 0, 0]
    x = np.zeros(5, dtype=np.float32)
    x[0] = 4.0                                          # at the edge only one side spreads
    assert list(oracle.stencil_1d(x)) == [2.0, 1.0, 0, 0, 0]


def test_stencil_is_linear_and_symmetric():
    rng = np.random.default_rng(5)
    a = rng.standard_normal(33).astype(np.float32)
    b = rng.standard_normal(33).astype(np.float32)
    lhs = oracle.stencil_1d(a) + oracle.stencil_1d(b)
    rhs = oracle.stencil_1d((a.astype(np.float64) + b).astype(np.float32))
    assert np.allclose(lhs, rhs, atol=1e-6)
    assert np.array_equal(oracle.stencil_1d(a[::-1].copy())[::-1], oracle.stencil_1d(a))  # mirror symmetry
    assert oracle.stencil_1d(np.zeros(0, np.float32)).shape == (0,)
    assert oracle.stencil_1d(np.array([2.0], np.float32))[0] == 1.0


# ---------------------------------------------------------------- attention forward pins
def _attn_inputs(b, sq, sk, d, dv, seed):
    Q = np.stack([bf16(sq, d, seed=seed + 3 * i) for i in range(b)])
    K = np.stack([bf16(sk, d, seed=seed + 3 * i + 1) for i in range(b)])
    V = np.stack([bf16(sk, dv, seed=seed + 3 * i + 2) for i in range(b)])
    return Q, K, V


def test_attention_zero_queries_average_the_values():
    _, K, V = _attn_inputs(2, 5, 37, 16, 8, 500)
    Q = np.zeros((2, 5, 16), np.uint16)
    O, lse = oracle.attention_forward(Q, K, V, with_lse=True)
    for b in range(2):
        means = np.array([math.fsum(col) / 37 for col in val(V[b]).T])
        assert np.allclose(O[b], means[None, :], rtol=0, atol=1e-15)
        assert np.allclose(lse[b], math.log(37.0), rtol=0, atol=1e-15)     # all scores 0


def test_attention_rows_are_convex_combinations():
    Q, K, _ = _attn_inputs(1, 9, 50, 32, 4, 510)
    ones = np.full((1, 50, 4), 0x3F80, np.uint16)                         # V = 1
    assert np.allclose(oracle.attention_forward(Q, K, ones), 1.0, rtol=0, atol=1e-14)


def test_attention_dominant_key_selects_its_value():
    # keys are scaled one-hots; with a large scale the matching key takes all the weight
    d, sk = 8, 8
    K = inputs.f64_to_bf16_bits(np.eye(sk, d))[None]
    Q = inputs.f64_to_bf16_bits(np.eye(sk, d)[[3, 6, 0]])[None]
    V = bf16(sk, 5, seed=520)[None]
    O = oracle.attention_forward(Q, K, V, scale=80.0)
    for r, j in enumerate([3, 6, 0]):
        assert np.allclose(O[0, r], val(V[0])[j], rtol=0, atol=1e-30)


@pytest.mark.parametrize("d", [64, 128])
def test_attention_default_scale_is_one_over_sqrt_d(d):
    # q = e0 and keys 8 e0 and 0: the two scores differ by 8 / sqrt(d) under the default
    # scale, so with V = (1, 0) the output is the logistic function of that difference
    # and the log-sum-exp is log(1 + e^(8 / sqrt(d))).
    Q = np.zeros((1, 1, d)); Q[0, 0, 0] = 1.0
    K = np.zeros((1, 2, d)); K[0, 0, 0] = 8.0
    V = np.array([[[1.0], [0.0]]])
    bits = inputs.f64_to_bf16_bits
    O, lse = oracle.attention_forward(bits(Q), bits(K), bits(V), with_lse=True)
    z = 8.0 / math.sqrt(d)
    assert O[0, 0, 0] == pytest.approx(1.0 / (1.0 + math.exp(-z)), rel=1e-15)
    assert lse[0, 0] == pytest.approx(math.log1p(math.exp(z)), rel=1e-15)


def test_attention_is_invariant_to_key_order_and_keeps_batches_apart():
    Q, K, V = _attn_inputs(2, 6, 23, 16, 12, 530)
    perm = np.random.default_rng(1).permutation(23)
    O = oracle.attention_forward(Q, K, V)
    assert np.allclose(O, oracle.attention_forward(Q, K[:, perm], V[:, perm]), rtol=0, atol=1e-14)
    O2 = oracle.attention_forward(Q, K[::-1].copy(), V[::-1].copy())
    assert not np.allclose(O2[0], O[0])


def test_attention_matches_high_precision_brute_force():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    Q, K, V = _attn_inputs(1, 3, 7, 5, 4, 540)
    scale = 0.61
    O, lse = oracle.attention_forward(Q, K, V, scale=scale, with_lse=True)
    q, k, v = val(Q[0]), val(K[0]), val(V[0])
    for i in range(3):
        s = [mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(q[i, t]) * mpmath.mpf(k[j, t]) for t in range(5))
             for j in range(7)]
        e = [mpmath.exp(x) for x in s]
        tot = mpmath.fsum(e)
        assert abs(float(mpmath.log(tot)) - lse[0, i]) <= 1e-13
        for c in range(4):
            ref = mpmath.fsum(e[j] * mpmath.mpf(v[j, c]) for j in range(7)) / tot
            assert abs(float(ref) - O[0, i, c]) <= 1e-13 * (1.0 + abs(float(ref)))


# ---- causal attention: query i attends keys 0..i only

def test_causal_first_row_is_the_first_value_exactly():
    Q, K, V = _attn_inputs(2, 6, 9, 16, 8, 600)
    O, lse = oracle.attention_forward(Q, K, V, scale=0.25, with_lse=True, causal=True)
    for b in range(2):
        assert np.array_equal(O[b, 0], val(V[b])[0])                       # a softmax over one key is 1
        dot = sum(Fraction(float(x)) * Fraction(float(y)) for x, y in zip(val(Q[b])[0], val(K[b])[0]))
        assert lse[b, 0] == pytest.approx(float(Fraction(1, 4) * dot), rel=1e-15, abs=1e-15)


def test_causal_rows_ignore_later_keys():
    # Replacing keys and values after the diagonal leaves every earlier row unchanged.
    Q, K, V = _attn_inputs(1, 12, 12, 16, 8, 610)
    O = oracle.attention_forward(Q, K, V, causal=True)
    for i in range(11):
        K2, V2 = K.copy(), V.copy()
        K2[0, i + 1:] = bf16(11 - i, 16, seed=620 + i)
        V2[0, i + 1:] = bf16(11 - i, 8, seed=640 + i)
        O2 = oracle.attention_forward(Q, K2, V2, causal=True)
        assert np.array_equal(O2[0, :i + 1], O[0, :i + 1])
        assert not np.array_equal(O2[0, i + 1:], O[0, i + 1:])


def test_causal_last_rows_see_every_key():
    # With more queries than keys, rows from sk - 1 on attend every key: the plain softmax.
    Q, K, V = _attn_inputs(2, 10, 6, 16, 8, 650)
    Oc, lc = oracle.attention_forward(Q, K, V, with_lse=True, causal=True)
    O, l = oracle.attention_forward(Q, K, V, with_lse=True)
    assert np.array_equal(Oc[:, 5:], O[:, 5:]) and np.array_equal(lc[:, 5:], l[:, 5:])
    assert not np.allclose(Oc[:, :5], O[:, :5])


def test_causal_matches_high_precision_brute_force():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    Q, K, V = _attn_inputs(1, 5, 4, 6, 3, 660)
    scale = 0.47
    O, lse = oracle.attention_forward(Q, K, V, scale=scale, with_lse=True, causal=True)
    q, k, v = val(Q[0]), val(K[0]), val(V[0])
    for i in range(5):
        keys = range(min(i + 1, 4))
        s = [mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(q[i, t]) * mpmath.mpf(k[j, t]) for t in range(6)) for j in keys]
        e = [mpmath.exp(x) for x in s]
        tot = mpmath.fsum(e)
        assert abs(float(mpmath.log(tot)) - lse[0, i]) <= 1e-13
        for c in range(3):
            ref = mpmath.fsum(e[n] * mpmath.mpf(v[j, c]) for n, j in enumerate(keys)) / tot
            assert abs(float(ref) - O[0, i, c]) <= 1e-13 * (1.0 + abs(float(ref)))
