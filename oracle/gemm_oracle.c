/*
 * CPU oracle for the tiled dense contraction -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg use
 * this file. The library's GPU path shares no code with it and never calls it.
 *
 * What it computes is the plain definition of the contraction the pages tile:
 *
 *   C_ref[i][j] = alpha * sum_k double(A[i][k]) * double(B[k][j]) + beta * double(C_in[i][j])
 *
 * with one double accumulator per output, k increasing, and the bf16 inputs
 * widened exactly to double. ("Hopper TMA Multicast 深度解析与实测", section
 * 经典应用场景: a CTA tile computes a product of operand tiles; "Clusters,
 * distributed shared memory & cluster launch control", sections "Two CTAs, one
 * MMA -- cta_group::2" and "TMA multicast": pairing CTAs and multicasting tiles
 * move operands differently but compute the same product.) beta == 0 means
 * C_in is not read (BLAS convention), so NaN in C_in cannot reach the result.
 *
 * The attention-score form S = Q * K^T follows the page-1 section 经典应用场景
 * (S_i = Q_i K^T): S[b][i][j] = sum_d Q[b][i][d] * K[b][j][d], no scale.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared (no fused multiply-add,
 * so x86 and Arm builds round identically).
 */
#include <stdint.h>
#include <string.h>
#include <omp.h>
#include <math.h>
#include <stdlib.h>

/* Exact widening of a bf16 bit pattern: it is the top half of a float32. */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* layout 0: row-major, element (r, c) at r*ld + c; layout 1: column-major, at c*ld + r. */
static int64_t offset_of(int layout, int64_t ld, int64_t r, int64_t c)
{
    return layout == 0 ? r * ld + c : c * ld + r;
}

/* dtype 0: bf16 bit patterns (uint16); 1: float32. */
static double load_c(const void *C, int dtype, int layout, int64_t ld, int64_t r, int64_t c)
{
    int64_t o = offset_of(layout, ld, r, c);
    if (dtype == 0)
        return bf16_to_double(((const uint16_t *)C)[o]);
    return (double)((const float *)C)[o];
}

static double dot_entry(int64_t K, const uint16_t *A, int64_t lda, int la,
                        const uint16_t *B, int64_t ldb, int lb, int64_t i, int64_t j)
{
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k)
        acc += bf16_to_double(A[offset_of(la, lda, i, k)]) * bf16_to_double(B[offset_of(lb, ldb, k, j)]);
    return acc;
}

/*
 * Full product: out is a row-major M x N double array with leading dimension ldo.
 * A is M x K (layout la), B is K x N (layout lb), C_in is M x N (layout lc, dtype dc)
 * and may be NULL when beta == 0.
 */
int oracle_gemm(int64_t M, int64_t N, int64_t K,
                const uint16_t *A, int64_t lda, int la,
                const uint16_t *B, int64_t ldb, int lb,
                const void *C_in, int64_t ldc, int lc, int dc,
                double alpha, double beta, double *out, int64_t ldo)
{
    if (M < 0 || N < 0 || K < 0)
        return 1;
    if (beta != 0.0 && C_in == NULL)
        return 2;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double r = alpha * dot_entry(K, A, lda, la, B, ldb, lb, i, j);
            if (beta != 0.0)
                r += beta * load_c(C_in, dc, lc, ldc, i, j);
            out[i * ldo + j] = r;
        }
    }
    return 0;
}

/*
 * The same definition evaluated only at n listed positions (rows[t], cols[t]);
 * used where the whole product is too large for the CPU.
 */
int oracle_gemm_entries(int64_t n, const int64_t *rows, const int64_t *cols, int64_t K,
                        const uint16_t *A, int64_t lda, int la,
                        const uint16_t *B, int64_t ldb, int lb,
                        const void *C_in, int64_t ldc, int lc, int dc,
                        double alpha, double beta, double *out)
{
    if (n < 0 || K < 0)
        return 1;
    if (beta != 0.0 && C_in == NULL)
        return 2;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t t = 0; t < n; ++t) {
        double r = alpha * dot_entry(K, A, lda, la, B, ldb, lb, rows[t], cols[t]);
        if (beta != 0.0)
            r += beta * load_c(C_in, dc, lc, ldc, rows[t], cols[t]);
        out[t] = r;
    }
    return 0;
}

/*
 * Batched attention scores S[b] = Q[b] * K[b]^T. Q[b] is sq x d and K[b] is
 * sk x d, both row-major with leading dimensions ldq / ldk and batch strides
 * sq_stride / sk_stride (elements). out is batch x sq x sk, row-major, dense.
 */
int oracle_attention_scores(int64_t batch, int64_t sq, int64_t sk, int64_t d,
                            const uint16_t *Q, int64_t ldq, int64_t q_stride,
                            const uint16_t *Kmat, int64_t ldk, int64_t k_stride,
                            double *out)
{
    if (batch < 0 || sq < 0 || sk < 0 || d < 0)
        return 1;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t i = 0; i < sq; ++i) {
            const uint16_t *q = Q + b * q_stride + i * ldq;
            for (int64_t j = 0; j < sk; ++j) {
                const uint16_t *kr = Kmat + b * k_stride + j * ldk;
                double acc = 0.0;
                for (int64_t t = 0; t < d; ++t)
                    acc += bf16_to_double(q[t]) * bf16_to_double(kr[t]);
                out[(b * sq + i) * sk + j] = acc;
            }
        }
    }
    return 0;
}

/* Number of OpenMP threads a parallel region here will use (for reporting). */
int oracle_num_threads(void)
{
    return omp_get_max_threads();
}

/*
 * 1-D three-point stencil of the cluster halo-exchange example ("集群编程",
 * section 实践示例：Halo 交换): y[i] = 0.25*x[i-1] + 0.5*x[i] + 0.25*x[i+1],
 * float32 inputs widened to double, x taken as 0 outside [0, n).
 */
int oracle_stencil_1d(int64_t n, const float *x, double *y)
{
    if (n < 0)
        return 1;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        const double l = i > 0 ? (double)x[i - 1] : 0.0;
        const double r = i + 1 < n ? (double)x[i + 1] : 0.0;
        y[i] = 0.25 * l + 0.5 * (double)x[i] + 0.25 * r;
    }
    return 0;
}

/*
 * Attention forward: O = softmax(scale * Q K^T) V per (batch, head), the fused
 * form of the score product above ("Hopper TMA Multicast 深度解析与实测",
 * section 经典应用场景: FlashAttention-type operators whose Q-tile CTAs share
 * the K/V tiles). Plain definition per query row i:
 *   s_j = scale * sum_t Q[i][t] K[j][t];  m = max_j s_j;  p_j = exp(s_j - m);
 *   l = sum_j p_j;  O[i] = sum_j p_j V[j] / l;  lse[i] = m + log(l)
 * (subtracting m leaves the softmax unchanged). Q is batch x sq x d, K is
 * batch x sk x d, V is batch x sk x dv, all bf16 bits, row-major and dense;
 * O is batch x sq x dv and lse batch x sq, in double. lse may be NULL.
 */
int oracle_attention_forward(int64_t batch, int64_t sq, int64_t sk, int64_t d, int64_t dv,
                             const uint16_t *Q, const uint16_t *Kmat, const uint16_t *V,
                             double scale, int causal, double *O, double *lse)
{
    if (batch < 0 || sq < 0 || sk < 1 || d < 0 || dv < 0)
        return 1;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t i = 0; i < sq; ++i) {
            const uint16_t *q = Q + (b * sq + i) * d;
            double *o = O + (b * sq + i) * dv;
            double *s = (double *)malloc(sizeof(double) * (size_t)sk);
            double m = -HUGE_VAL;
            /* causal: query i sees keys 0..i only (the others are left out of the softmax) */
            const int64_t nk = causal ? (i + 1 < sk ? i + 1 : sk) : sk;
            for (int64_t j = 0; j < nk; ++j) {
                const uint16_t *kr = Kmat + (b * sk + j) * d;
                double acc = 0.0;
                for (int64_t t = 0; t < d; ++t)
                    acc += bf16_to_double(q[t]) * bf16_to_double(kr[t]);
                s[j] = scale * acc;
                if (s[j] > m)
                    m = s[j];
            }
            double l = 0.0;
            for (int64_t j = 0; j < nk; ++j) {
                s[j] = exp(s[j] - m);
                l += s[j];
            }
            for (int64_t c = 0; c < dv; ++c) {
                double acc = 0.0;
                for (int64_t j = 0; j < nk; ++j)
                    acc += s[j] * bf16_to_double(V[(b * sk + j) * dv + c]);
                o[c] = acc / l;
            }
            if (lse)
                lse[b * sq + i] = m + log(l);
            free(s);
        }
    }
    return 0;
}
