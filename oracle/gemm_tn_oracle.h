/*
 * CPU oracle for the half-precision TN GEMM — TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
 * legs may load this code.  The product path (the CUDA library) never calls it
 * and shares no code, header, table or helper with it.
 *
 * What it computes (one definition, written out plainly):
 *
 *   D[b][m][n] = RNE_fp16( alpha * sum_{k<K} A[b][m][k] * B[b][n][k]
 *                          + beta * C[b][m][n] )
 *
 *   - the TN contraction of "CuTe C++ 简介01 … gemm_device", section 3
 *     (appendix code: the SIMT loop tCrC(m,n) += tCsA(m,k) * tCsB(n,k));
 *   - the epilogue C = alpha*A*B + beta*C of the same page (axpby, and the
 *     kernel signature in section 1);
 *   - A (M,K) and B (N,K) both K-contiguous, D (M,N) N-contiguous, as in
 *     "cute(8) smem_gemm", section "代码实现" (make_stride(K, Int<1>)).
 *
 * Readings taken where the pages are silent:
 *   - every fp16 operand is decoded exactly to fp64; products and the k-ordered
 *     sum are done in fp64; alpha and beta are fp32 values widened to fp64;
 *   - exactly one rounding to fp16 at the end, IEEE round-to-nearest-even,
 *     subnormals kept, overflow to +-inf, NaN stays NaN;
 *   - beta == 0 drops the C term entirely (C is not read, may be NULL);
 *   - K == 0 gives D = RNE(beta*C); M == 0 or N == 0 does nothing.
 *
 * Parity pins (tests/test_oracle_pins.py): exhaustive fp16 decode and encode
 * against numpy's IEEE conversions, exact rational brute force on tiny shapes,
 * identity / permutation matrices, the all-ones closed form, the transpose
 * invariant D(A,B)^T = D(B,A), small-integer exactness against integer matmul.
 */
#ifndef GEMM_TN_ORACLE_H
#define GEMM_TN_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exact binary16 -> binary64 decode (IEEE 754 binary16 bit layout). */
double gto_half_to_double(uint16_t h);

/* binary64 -> binary16, round to nearest, ties to even. */
uint16_t gto_double_to_half(double x);

/*
 * Batched TN GEMM over flattened output rows r in [r_begin, r_end), where
 * r = b*M + m.  Matrices are arrays of binary16 bit patterns; strides and
 * leading dimensions are in elements.  C may be NULL when beta == 0.
 */
void gto_gemm_tn_f16(const uint16_t* A, int64_t lda, int64_t strideA,
                     const uint16_t* B, int64_t ldb, int64_t strideB,
                     const uint16_t* C, int64_t ldc, int64_t strideC,
                     uint16_t* D, int64_t ldd, int64_t strideD,
                     int64_t M, int64_t N, int64_t K,
                     float alpha, float beta,
                     int64_t r_begin, int64_t r_end);

/*
 * The same definition evaluated at `count` chosen output positions
 * (b_idx[i], m_idx[i], n_idx[i]); results go to out[i].
 */
void gto_gemm_tn_f16_entries(const uint16_t* A, int64_t lda, int64_t strideA,
                             const uint16_t* B, int64_t ldb, int64_t strideB,
                             const uint16_t* C, int64_t ldc, int64_t strideC,
                             int64_t K, float alpha, float beta,
                             const int64_t* b_idx, const int64_t* m_idx,
                             const int64_t* n_idx, int64_t count,
                             uint16_t* out);

/*
 * The same definition with generic element strides, as the gemm_device page's
 * kernel takes them (dA, dB, dC: "CuTe C++ 简介01 / gemm_device 逐行解析",
 * section 1): A(m,k) = A[b*strideA + m*a_rs + k*a_cs], B(n,k) = B[b*strideB +
 * n*b_rs + k*b_cs]; C and D are row-major (ldc, ldd) as above.  Rows
 * r = b*M + m in [r_begin, r_end).
 */
void gto_gemm_f16_strided(const uint16_t* A, int64_t a_rs, int64_t a_cs, int64_t strideA,
                          const uint16_t* B, int64_t b_rs, int64_t b_cs, int64_t strideB,
                          const uint16_t* C, int64_t ldc, int64_t strideC,
                          uint16_t* D, int64_t ldd, int64_t strideD,
                          int64_t M, int64_t N, int64_t K,
                          float alpha, float beta,
                          int64_t r_begin, int64_t r_end);

/*
 * Matrix transpose y = x^T of the "10-mat-transpose-cute" page (each version
 * computes y[c][r] = x[r][c] for an M x N row-major x, predicated at the edges):
 * element bits are copied, 4-byte (fp32) or 2-byte (fp16) elements.
 */
void gto_transpose_u32(const uint32_t* X, int64_t ldx, uint32_t* Y, int64_t ldy, int64_t rows, int64_t cols);
void gto_transpose_u16(const uint16_t* X, int64_t ldx, uint16_t* Y, int64_t ldy, int64_t rows, int64_t cols);

/*
 * Softmax row statistics of the scaled score matrix, the step that follows the
 * score GEMM score = Q @ K.T of "为什么 cutlass_cute_tutorial_zh.md 中要用
 * retile_D" (section 1: Q is the MMA's A operand, K its B operand, head_dim
 * 64).  The pages stop at the score; the statistics are the textbook softmax
 * normaliser, for batch entry b and query row i:
 *
 *   s_j      = alpha * sum_{k<d} Q[b][i][k] * K[b][j][k]      (fp64, k order)
 *   m[b][i]  = max_{j<N} s_j
 *   l[b][i]  = sum_{j<N} exp(s_j - m[b][i])                     (fp64, j order)
 *
 * so that softmax(s)_j = exp(s_j - m) / l and logsumexp(s) = m + log(l).
 * Q is M x d (leading dimension ldq), K is N x d (ldk), batch strides strideQ,
 * strideK; outputs are indexed r = b*M + i for rows r in [r_begin, r_end).
 * N == 0 gives m = -inf and l = 0.  Inputs are finite.
 */
void gto_score_softmax_stats(const uint16_t* Q, int64_t ldq, int64_t strideQ,
                             const uint16_t* K, int64_t ldk, int64_t strideK,
                             int64_t M, int64_t N, int64_t d, float alpha,
                             double* row_max, double* row_sum,
                             int64_t r_begin, int64_t r_end);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_TN_ORACLE_H */
