/*
 * CPU oracle for the half-precision TN GEMM — TEST INFRASTRUCTURE ONLY.
 * Loaded only by tests/, __graft_entry__.smoke() and bench.py's CPU legs.
 *
 * Plain, slow, obviously correct: decode fp16 exactly to fp64, take the
 * k-ordered fp64 sum of products, apply alpha and beta in fp64, round once to
 * fp16 with round-to-nearest-even.  No blocking, no reordering.
 *
 * Sources (page title, section):
 *   - "CuTe C++ 简介01 / gemm_device 逐行解析", section 3 (appendix code): the
 *     TN inner product tCrC(m,n) += tCsA(m,k) * tCsB(n,k) and the epilogue
 *     tCgC(i) = alpha * tCrC(i) + beta * tCgC(i);
 *   - "cute(8) smem_gemm", section "代码实现": A is (M,K) and B is (N,K), both
 *     with stride (K,1); D is (M,N) with stride (N,1).
 *
 * Compile with -ffp-contract=off so no multiply-add is fused: the result is
 * then the same on every host.
 */
#include "gemm_tn_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stddef.h>

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double gto_half_to_double(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 10) & 0x1f;
    const int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        /* zero or subnormal: frac * 2^-24 */
        v = ldexp((double)frac, -24);
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        /* normal: (1024 + frac) * 2^(expo - 15 - 10) */
        v = ldexp((double)(1024 + frac), expo - 25);
    }
    return sign ? -v : v;
}

/*
 * Round a binary64 value to binary16, nearest, ties to even.
 * The value is scaled (exactly, by a power of two) so that one unit in the
 * last place of the target binade becomes 1.0, rounded to an integer with
 * rint() (default rounding mode = nearest-even), and the bits rebuilt.
 */
uint16_t gto_double_to_half(double x)
{
    if (isnan(x)) return 0x7e00;
    const uint16_t sign = signbit(x) ? 0x8000 : 0;
    const double a = fabs(x);
    if (isinf(a)) return sign | 0x7c00;
    if (a == 0.0) return sign;

    int e2;
    (void)frexp(a, &e2);          /* a = f * 2^e2, f in [0.5, 1) */
    const int E = e2 - 1;         /* a in [2^E, 2^(E+1)) */
    /* Exponent of one ulp: 2^(E-10) for normal binades, 2^-24 below 2^-14. */
    const int q = (E < -14) ? -24 : E - 10;
    if (q > 15 - 10 + 1) {
        /* a >= 2^17: far beyond the largest finite half (65504). */
        return sign | 0x7c00;
    }
    const double units = rint(ldexp(a, -q)); /* exact scaling, then RNE */
    long u = (long)units;
    uint32_t bits;
    if (q == -24) {
        /* subnormal range; u == 1024 is the smallest normal, same encoding. */
        bits = (uint32_t)u;
    } else {
        /* u in [1024, 2048]; u == 2048 carries into the next binade. */
        bits = ((uint32_t)(E + 15) << 10) + (uint32_t)(u - 1024);
    }
    if (bits >= 0x7c00) bits = 0x7c00; /* overflow to infinity */
    return (uint16_t)(sign | bits);
}

/* Exact decode table, filled once; entry h holds gto_half_to_double(h). */
static double g_decode[65536];
static pthread_once_t g_decode_once = PTHREAD_ONCE_INIT;

static void decode_table_fill(void)
{
    for (uint32_t h = 0; h < 65536u; ++h) g_decode[h] = gto_half_to_double((uint16_t)h);
}

static void decode_table_init(void)
{
    pthread_once(&g_decode_once, decode_table_fill);
}

/* One output element: alpha * sum_k A[m,k]*B[n,k] + beta * C[m,n], then RNE. */
static uint16_t one_entry(const uint16_t* a_row, const uint16_t* b_row, int64_t K,
                          double alpha, double beta, const uint16_t* c_elem)
{
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        acc += g_decode[a_row[k]] * g_decode[b_row[k]];
    }
    double v = alpha * acc;
    if (beta != 0.0) {
        v = v + beta * g_decode[*c_elem];
    }
    return gto_double_to_half(v);
}

void gto_gemm_tn_f16(const uint16_t* A, int64_t lda, int64_t strideA,
                     const uint16_t* B, int64_t ldb, int64_t strideB,
                     const uint16_t* C, int64_t ldc, int64_t strideC,
                     uint16_t* D, int64_t ldd, int64_t strideD,
                     int64_t M, int64_t N, int64_t K,
                     float alpha, float beta,
                     int64_t r_begin, int64_t r_end)
{
    decode_table_init();
    if (M <= 0 || N <= 0) return;
    const double al = (double)alpha;
    const double be = (double)beta;
    for (int64_t r = r_begin; r < r_end; ++r) {
        const int64_t b = r / M;
        const int64_t m = r % M;
        const uint16_t* a_row = A + b * strideA + m * lda;
        for (int64_t n = 0; n < N; ++n) {
            const uint16_t* b_row = B + b * strideB + n * ldb;
            const uint16_t* c_elem = (be != 0.0) ? (C + b * strideC + m * ldc + n) : NULL;
            D[b * strideD + m * ldd + n] = one_entry(a_row, b_row, K, al, be, c_elem);
        }
    }
}

void gto_gemm_tn_f16_entries(const uint16_t* A, int64_t lda, int64_t strideA,
                             const uint16_t* B, int64_t ldb, int64_t strideB,
                             const uint16_t* C, int64_t ldc, int64_t strideC,
                             int64_t K, float alpha, float beta,
                             const int64_t* b_idx, const int64_t* m_idx,
                             const int64_t* n_idx, int64_t count,
                             uint16_t* out)
{
    decode_table_init();
    const double al = (double)alpha;
    const double be = (double)beta;
    for (int64_t i = 0; i < count; ++i) {
        const int64_t b = b_idx[i], m = m_idx[i], n = n_idx[i];
        const uint16_t* a_row = A + b * strideA + m * lda;
        const uint16_t* b_row = B + b * strideB + n * ldb;
        const uint16_t* c_elem = (be != 0.0) ? (C + b * strideC + m * ldc + n) : NULL;
        out[i] = one_entry(a_row, b_row, K, al, be, c_elem);
    }
}

/* Generic strides: the k-ordered fp64 sum of A(m,k)*B(n,k), then alpha, beta, RNE. */
void gto_gemm_f16_strided(const uint16_t* A, int64_t a_rs, int64_t a_cs, int64_t strideA,
                          const uint16_t* B, int64_t b_rs, int64_t b_cs, int64_t strideB,
                          const uint16_t* C, int64_t ldc, int64_t strideC,
                          uint16_t* D, int64_t ldd, int64_t strideD,
                          int64_t M, int64_t N, int64_t K,
                          float alpha, float beta,
                          int64_t r_begin, int64_t r_end)
{
    decode_table_init();
    if (M <= 0 || N <= 0) return;
    const double al = (double)alpha;
    const double be = (double)beta;
    for (int64_t r = r_begin; r < r_end; ++r) {
        const int64_t b = r / M;
        const int64_t m = r % M;
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                acc += g_decode[A[b * strideA + m * a_rs + k * a_cs]] *
                       g_decode[B[b * strideB + n * b_rs + k * b_cs]];
            }
            double v = al * acc;
            if (be != 0.0) v = v + be * g_decode[C[b * strideC + m * ldc + n]];
            D[b * strideD + m * ldd + n] = gto_double_to_half(v);
        }
    }
}

void gto_transpose_u32(const uint32_t* X, int64_t ldx, uint32_t* Y, int64_t ldy, int64_t rows, int64_t cols)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) Y[c * ldy + r] = X[r * ldx + c];
}

void gto_transpose_u16(const uint16_t* X, int64_t ldx, uint16_t* Y, int64_t ldy, int64_t rows, int64_t cols)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) Y[c * ldy + r] = X[r * ldx + c];
}

/* alpha * (k-ordered fp64 dot of one query row with one key row) */
static double score(const uint16_t* q_row, const uint16_t* k_row, int64_t d, double alpha)
{
    double acc = 0.0;
    for (int64_t k = 0; k < d; ++k) acc += g_decode[q_row[k]] * g_decode[k_row[k]];
    return alpha * acc;
}

/* Two passes over the keys: the maximum, then the sum of exp(s_j - max). */
void gto_score_softmax_stats(const uint16_t* Q, int64_t ldq, int64_t strideQ,
                             const uint16_t* K, int64_t ldk, int64_t strideK,
                             int64_t M, int64_t N, int64_t d, float alpha,
                             double* row_max, double* row_sum,
                             int64_t r_begin, int64_t r_end)
{
    decode_table_init();
    if (M <= 0) return;
    const double al = (double)alpha;
    for (int64_t r = r_begin; r < r_end; ++r) {
        const int64_t b = r / M;
        const int64_t i = r % M;
        const uint16_t* q_row = Q + b * strideQ + i * ldq;
        const uint16_t* k_base = K + b * strideK;
        double m = -INFINITY;
        for (int64_t j = 0; j < N; ++j) {
            const double s = score(q_row, k_base + j * ldk, d, al);
            if (s > m) m = s;
        }
        double l = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            l += exp(score(q_row, k_base + j * ldk, d, al) - m);
        }
        row_max[r] = m;
        row_sum[r] = l;
    }
}
