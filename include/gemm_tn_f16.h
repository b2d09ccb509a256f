/*
 * gemm_tn_f16 — half-precision TN GEMM for one NVIDIA GB300 (sm_103a) GPU.
 *
 *     D[m][n] = alpha * sum_k A[m][k] * B[n][k] + beta * C[m][n]
 *
 * The operation is the GEMM of the "CuTe C++ 简介01 / gemm_device 逐行解析"
 * page: the TN inner product tCrC(m,n) += tCsA(m,k) * tCsB(n,k) and the
 * axpby epilogue C = alpha*A*B + beta*C (section 1, kernel signature;
 * section 3, appendix code), with A (M,K) and B (N,K) both K-contiguous and
 * D (M,N) N-contiguous as in "cute(8) smem_gemm", section "代码实现"
 * (make_stride(K, Int<1>) for A and B, make_stride(N, Int<1>) for D).
 * The batched form is the attention-score contraction score = Q . K^T of the
 * "为什么要用 retile_D" page (sections 1 and 3: Q is the A operand, K the B
 * operand, head_dim 64), one GEMM per batch entry.
 *
 * Numerics: A, B, C, D are IEEE binary16.  Products are accumulated in fp32
 * on the tensor cores (summation order unspecified); alpha*acc + beta*C is
 * formed in fp32 and rounded once to binary16, round-to-nearest-even,
 * subnormals kept, overflow to +-inf.
 *
 * Layout (all sizes and leading dimensions count ELEMENTS, not bytes):
 *   A: M rows of K halves, row m at A + m*lda,   lda >= max(K,1)
 *   B: N rows of K halves, row n at B + n*ldb,   ldb >= max(K,1)
 *   C: M rows of N halves, row m at C + m*ldc,   ldc >= max(N,1)  (if beta != 0)
 *   D: M rows of N halves, row m at D + m*ldd,   ldd >= max(N,1)
 *   batched: entry b of X starts at X + b*strideX (strides >= 0; a stride of
 *   0 broadcasts that operand; D's stride must keep entries disjoint).
 *
 * Ownership and memory: every pointer is DEVICE memory owned by the caller
 * and must stay valid until the work queued on `stream` has finished.  The
 * library keeps, per device, a small stream-ordered memory pool for its own
 * scratch (split-K partial sums, repacked copies of operands whose leading
 * dimension is not a multiple of 8); scratch is allocated and freed in stream
 * order, so concurrent calls on different streams never share it.
 * gemm_tn_f16_shutdown() returns the pool's memory.
 *
 * Alignment: every pointer must be 2-byte aligned.  Any leading dimension
 * and any 2-byte-aligned address is accepted; 16-byte aligned pointers with
 * leading dimensions (and batch strides) that are multiples of 8 take the
 * direct tensor-memory-accelerator path.  Otherwise A and B are first repacked to
 * aligned scratch copies, while C is read and D written by the epilogue in their
 * own rows, through the aligned 16-byte words that cover each row segment (only
 * D's own elements are ever written).
 *
 * Special cases: M == 0, N == 0 or batch == 0 does nothing and returns
 * GEMM_OK.  K == 0 gives D = beta*C (D = 0 when beta == 0).  When beta == 0,
 * C is never read and may be NULL (NaNs in C do not propagate).  D may alias
 * C exactly (same pointer, ldc == ldd, same batch stride); any other overlap
 * between D and A, B or C is undefined.
 *
 * Asynchrony and errors: calls enqueue work on `stream` and return without
 * waiting.  The returned status covers argument checks and the launch.  No
 * function ever exits or aborts the process.  Device-side waits are bounded:
 * a kernel whose pipeline stalls past its limit records GEMM_ERR_TIMEOUT in a
 * device error word and returns; read it with gemm_tn_f16_last_device_error().
 */
#ifndef GEMM_TN_F16_H
#define GEMM_TN_F16_H

#include <stdint.h>

#if defined(__GNUC__)
#define GEMM_TN_API __attribute__((visibility("default")))
#else
#define GEMM_TN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t is a pointer to this opaque type; NULL is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st* gemm_stream_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_VALUE = 1, /* bad size, leading dimension, stride or NULL pointer */
    GEMM_ERR_MISALIGNED = 2,    /* a pointer is not 2-byte aligned */
    GEMM_ERR_UNSUPPORTED = 3,   /* device is not sm_103 / sm_100 class, or sizes beyond limits */
    GEMM_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed (see gemm_tn_f16_last_cuda_error) */
    GEMM_ERR_TIMEOUT = 5,       /* a device-side wait ran past its limit (device error word) */
    GEMM_ERR_WORKSPACE = 6,     /* scratch memory could not be obtained */
    GEMM_ERR_BOUNDS = 7         /* checked build only: a kernel's own load or store fell outside the
                                   matrix it belongs to and was skipped (device error word) */
} gemm_status_t;

/*
 * D = alpha * A . B^T + beta * C for one problem.
 * A: const half[M][lda]; B: const half[N][ldb]; C: const half[M][ldc] or NULL
 * when beta == 0; D: half[M][ldd].  Sizes must be >= 0 and M, N, K < 2^31.
 * Returns GEMM_OK once the work is queued on `stream`.
 */
GEMM_TN_API gemm_status_t gemm_tn_f16(const void* A, int64_t lda,
                          const void* B, int64_t ldb,
                          const void* C, int64_t ldc,
                          void* D, int64_t ldd,
                          int64_t M, int64_t N, int64_t K,
                          float alpha, float beta,
                          gemm_stream_t stream);

/*
 * The same for `batch` independent problems of one shape:
 *   D_b = alpha * A_b . B_b^T + beta * C_b,  X_b = X + b*strideX (elements).
 * For the attention score S = Q . K^T: A = Q (seq_q x head_dim, lda = head_dim),
 * B = K (seq_k x head_dim), D = S (seq_q x seq_k), batch = batch*heads.
 */
GEMM_TN_API gemm_status_t gemm_tn_f16_batched(const void* A, int64_t lda, int64_t strideA,
                                  const void* B, int64_t ldb, int64_t strideB,
                                  const void* C, int64_t ldc, int64_t strideC,
                                  void* D, int64_t ldd, int64_t strideD,
                                  int64_t M, int64_t N, int64_t K, int64_t batch,
                                  float alpha, float beta,
                                  gemm_stream_t stream);

/*
 * Operand storage for gemm_f16.  The product is always D = alpha * A . B^T + beta * C
 * with A logically M x K and B logically N x K (TN is both K-major).
 *   GEMM_K_MAJOR : A stored M x lda with K contiguous (lda >= K); B stored N x ldb.
 *   GEMM_MN_MAJOR: A stored K x lda with M contiguous (lda >= M), i.e. A^T row-major;
 *                  B stored K x ldb with N contiguous (ldb >= N).
 */
typedef enum { GEMM_K_MAJOR = 0, GEMM_MN_MAJOR = 1 } gemm_major_t;

/*
 * The GEMM with either operand in either storage order -- the stride-generic form
 * of the "gemm_device 逐行解析" page, whose kernel takes A, B and C with arbitrary
 * strides dA, dB, dC (section 1).  Batched like gemm_tn_f16_batched (batch >= 1;
 * strideX between entries, 0 broadcasts A, B or C).  An MN-major operand is read by
 * the tensor core through an MN-major shared-memory layout; operands are never
 * swapped for small M in that case.  All other rules as gemm_tn_f16_batched;
 * GEMM_ERR_INVALID_VALUE for an unknown a_major / b_major.
 */
GEMM_TN_API gemm_status_t gemm_f16(int32_t a_major, int32_t b_major,
                                   const void* A, int64_t lda, int64_t strideA,
                                   const void* B, int64_t ldb, int64_t strideB,
                                   const void* C, int64_t ldc, int64_t strideC,
                                   void* D, int64_t ldd, int64_t strideD,
                                   int64_t M, int64_t N, int64_t K, int64_t batch,
                                   float alpha, float beta,
                                   gemm_stream_t stream);

/*
 * gemm_f16 with the products accumulated in fp16 on the tensor core, as the
 * "cute(8) smem_gemm" page's kernel does (GemmConfig: SM80_16x8x16_F16F16F16F16_TN).
 * About as fast as gemm_f16 (within a few percent either way on 8192^3) and far
 * less accurate (every 16-wide K step rounds the running sum to fp16); provided
 * for that page's semantics.
 * alpha and beta are applied in fp32 to the fp16 accumulator, then D is rounded.
 * Same arguments and rules as gemm_f16.
 */
GEMM_TN_API gemm_status_t gemm_f16_acc16(int32_t a_major, int32_t b_major,
                                         const void* A, int64_t lda, int64_t strideA,
                                         const void* B, int64_t ldb, int64_t strideB,
                                         const void* C, int64_t ldc, int64_t strideC,
                                         void* D, int64_t ldd, int64_t strideD,
                                         int64_t M, int64_t N, int64_t K, int64_t batch,
                                         float alpha, float beta,
                                         gemm_stream_t stream);

/*
 * gemm_tn_f16 with A, B, C and D in HOST memory: the same product, rules and
 * layouts, with the host <-> device traffic handled by the library.  B goes to the
 * device first; A, C and D travel in blocks of rows on two library streams, so that
 * one block's GEMM overlaps the next block's A and C coming in and the previous
 * block's D going out.  Only the matrix elements are copied (never the padding
 * between rows; D's padding in host memory is left untouched).  Page-locked host
 * memory (cudaHostAlloc / cudaHostRegister) lets the copies run asynchronously and
 * overlap; pageable memory works but the copies then block the calling thread.
 * Asynchronous on `stream`: the host buffers must stay valid and A, B, C unmodified
 * until the stream has passed the call, and D is complete only then (synchronize on
 * `stream` before reading it).  Device staging buffers come from the library's
 * stream-ordered pool (GEMM_ERR_WORKSPACE if that fails).  The pages move data to the
 * device before their kernels and show no such call.
 */
GEMM_TN_API gemm_status_t gemm_tn_f16_host(const void* A, int64_t lda, const void* B, int64_t ldb,
                                           const void* C, int64_t ldc, void* D, int64_t ldd,
                                           int64_t M, int64_t N, int64_t K, float alpha, float beta,
                                           gemm_stream_t stream);

/*
 * Fused score GEMM + scale + softmax statistics.  The score is the Q @ K.T of the
 * "为什么 cutlass_cute_tutorial_zh.md 中要用 retile_D" page (section 1: Q is the
 * MMA's A operand, K its B operand; head_dim 64 there); the pages stop at the
 * score, and this call continues with the softmax normaliser of each score row,
 * computed online so that the score matrix is never stored:
 *
 *   s_ij          = alpha * sum_{k<d} Q[b][i][k] * K[b][j][k]   (fp32 accumulate)
 *   row_max[b*M+i] = max_j s_ij
 *   row_sum[b*M+i] = sum_j exp(s_ij - row_max[b*M+i])
 *
 * so softmax(s_i)_j = exp(s_ij - row_max) / row_sum and logsumexp = row_max + log(row_sum).
 * Q: M x d per batch entry, row-major with leading dimension ldq >= d; K: N x d,
 * ldk >= d; strideQ / strideK between batch entries (0 broadcasts one operand).
 * row_max, row_sum: batch * M fp32 each, device memory, 4-byte aligned, written
 * only (they must not overlap each other or Q, K: GEMM_ERR_INVALID_VALUE).
 * d <= 256 (GEMM_ERR_UNSUPPORTED above).  Q and K need only 2-byte alignment:
 * operands whose rows are not 16-byte aligned are first copied to an aligned
 * scratch copy from the library's stream-ordered pool (GEMM_ERR_WORKSPACE if that
 * fails).  M == 0 or batch == 0 does nothing; N == 0 gives row_max = -inf,
 * row_sum = 0; d == 0 gives row_max = 0, row_sum = N.  Inputs are finite.
 * Asynchronous on `stream`; a device-side wait that times out is reported by
 * gemm_tn_f16_last_device_error().
 */
GEMM_TN_API gemm_status_t score_softmax_stats_f16(const void* Q, int64_t ldq, int64_t strideQ,
                                                  const void* K, int64_t ldk, int64_t strideK,
                                                  float* row_max, float* row_sum,
                                                  int64_t M, int64_t N, int64_t d, int64_t batch,
                                                  float alpha, gemm_stream_t stream);

/*
 * Matrix transpose Y = X^T of the "10-mat-transpose-cute" page (y[c][r] = x[r][c]
 * for a rows x cols row-major x; predicated at ragged edges): fp32 (the page's
 * type) and fp16 elements, bits copied unchanged.
 * X: rows x ldx (ldx >= cols), Y: cols x ldy (ldy >= rows), both device memory;
 * they must not overlap (GEMM_ERR_INVALID_VALUE), elements must be naturally
 * aligned (GEMM_ERR_MISALIGNED).  16-byte aligned matrices with leading dimensions
 * that are multiples of 16 bytes take the vectorised path.  Asynchronous on stream.
 */
GEMM_TN_API gemm_status_t transpose_f32(const void* X, int64_t ldx, void* Y, int64_t ldy,
                                        int64_t rows, int64_t cols, gemm_stream_t stream);
GEMM_TN_API gemm_status_t transpose_f16(const void* X, int64_t ldx, void* Y, int64_t ldy,
                                        int64_t rows, int64_t cols, gemm_stream_t stream);

/* Static English text for a status code; never NULL. */
GEMM_TN_API const char* gemm_status_string(gemm_status_t status);

/*
 * Synchronises the current device, then reads and clears the device error
 * word that bounded device-side waits write.  GEMM_OK when no kernel of this
 * library has reported a stall since the last call, GEMM_ERR_TIMEOUT if one
 * has, GEMM_ERR_CUDA if the synchronisation itself failed.
 */
GEMM_TN_API gemm_status_t gemm_tn_f16_last_device_error(void);

/* The CUDA error code (cudaError_t value) behind the last GEMM_ERR_CUDA of this thread. */
GEMM_TN_API int gemm_tn_f16_last_cuda_error(void);

/* Returns the library pool's memory to the driver for every device it was used on. */
GEMM_TN_API void gemm_tn_f16_shutdown(void);

/* Library version, major*10000 + minor*100 + patch. */
GEMM_TN_API int gemm_tn_f16_version(void);

/*
 * 1 for the checked build (libgemm_tn_f16_checked.so, compiled with device-side bounds
 * checks), 0 for the regular one.  In the checked build every load and store the
 * kernels issue themselves -- C and D rows or elements in the epilogues, rows read by
 * the row loader, the repack of misaligned operands, the split-K sum, the K == 0
 * scale -- is tested against the byte range of its matrix (derived from the pointer,
 * sizes, leading dimension and batch stride of the call); one outside is skipped and
 * reported by gemm_tn_f16_last_device_error() as GEMM_ERR_BOUNDS.  Tensor copies are
 * bounded by their tensor maps.  A debugging aid: the checks cost time.
 */
GEMM_TN_API int gemm_tn_f16_is_checked(void);

/*
 * Host-only planning (no CUDA call; safe without a GPU).  Describes the
 * kernel the library would launch for a problem on a device with `num_sms`
 * streaming multiprocessors.  `align_flags` bit i set means operand i
 * (0=A, 1=B, 2=C, 3=D) has a 16-byte aligned base pointer.
 */
typedef struct {
    int32_t kernel;          /* 0 none (empty problem), 1 scale-only (K == 0),
                                2 tensor-core tile kernel, 3 split-K (+ reduction),
                                4 small-problem kernel (one CTA per 128 x tile_n tile, every
                                  k-block loaded at once: K <= 512 with tile_n 64, K <= 384
                                  with tile_n 128; stages = k-blocks) */
    int32_t tile_m;          /* output rows per tile as seen by the tensor core (128 or 256) */
    int32_t tile_n;          /* output columns per tile as seen by the tensor core (16..256, or 432
                                or 512: two MMAs, N = 256 and N = tile_n - 256, side by side on
                                a CTA pair) */
    int32_t cta_pair;        /* 1: one CTA per tile; 2: CTA pair sharing one 256-row tile */
    int32_t swap_ab;         /* 1: computes D^T = B . A^T (small M) */
    int32_t splits;          /* K slices (1 = no split) */
    int32_t stages;          /* shared-memory pipeline depth */
    int32_t epi_tma;         /* 1: D written by tensor copies (C, if beta != 0, read by tensor copies when
                                its rows are 16-byte aligned, else by the epilogue's own aligned
                                loads); 0: D (and C) accessed by the epilogue's own loads and
                                stores, through aligned 16-byte words (D rows not 16-byte
                                aligned) or element by element (a forced predicated epilogue) */
    int32_t pack_a;          /* 1: A is first repacked to an aligned scratch copy */
    int32_t pack_b;          /* 1: B is first repacked */
    int64_t units;           /* work units (tiles x splits x batch) */
    int64_t grid;            /* CTAs launched */
    int64_t workspace_bytes; /* scratch taken from the pool for this call */
    int32_t stream_k;        /* 1: the last partial wave of tiles is spread over all CTA groups by k-block */
    int32_t sk_maxc;         /* stream-K: largest number of CTA groups contributing to one tile */
    int64_t dp_tiles;        /* tiles computed whole (data-parallel), before the stream-K tiles */
    int64_t sk_tiles;        /* tiles shared out by k-block */
    int32_t stage_cd;        /* always 0: no scratch copies of C or D are made (the epilogue reads
                                C and writes D in place at any alignment) */
    int32_t row_load;        /* bit 0 (A) / bit 1 (B): the operand's rows, which tensor copies cannot
                                address, are read by the kernel's own loader warps instead of
                                being repacked (GEMM_TN_OPT_ROW_LOADER; pack_a / pack_b stay 0) */
    int32_t k_cluster;       /* 1: each (swapped) tile's K is split between the two CTAs of a
                                cluster; the second half's fp32 partial goes through distributed
                                shared memory to the first CTA, which writes D (one launch, no
                                scratch; splits stays 1) */
    int32_t reserved;
} gemm_tn_plan_t;

GEMM_TN_API gemm_status_t gemm_tn_f16_plan(int64_t M, int64_t N, int64_t K, int64_t batch,
                               int64_t lda, int64_t ldb, int64_t ldc, int64_t ldd,
                               int64_t strideA, int64_t strideB, int64_t strideC, int64_t strideD,
                               float beta, uint32_t align_flags, int32_t num_sms,
                               gemm_tn_plan_t* plan);

/*
 * Process-wide tuning and test options (host only; take effect on the next call).
 *   GEMM_TN_OPT_WAIT_TIMEOUT_NS   limit of every device-side wait, in ns (default 2e9).
 *   GEMM_TN_OPT_SKIP_FIRST_LOAD   1: CTA 0 of each tensor-core launch skips its first operand
 *                                 load, so its MMA wait runs out and the kernel reports
 *                                 GEMM_ERR_TIMEOUT -- exercises the stall path without any
 *                                 fault.  Testing only; 0 restores normal operation.
 *   GEMM_TN_OPT_FORCE_BN          force the tile width: 128, 256, 432 or 512 (512: CTA pairs
 *                                 with a TMA epilogue only, else 256; 432: CTA pairs, K-major
 *                                 operands, beta == 0 and 16-byte aligned D rows only, else
 *                                 as 512), 0 = automatic.
 *   GEMM_TN_OPT_FORCE_PAIR        force 1 (single CTA) or 2 (CTA pair), 0 = automatic.
 *   GEMM_TN_OPT_FORCE_SPLITS      force the number of K slices, 0 = automatic: K slices, summed
 *                                 by a second kernel, when 128 x 128 tiles would occupy at
 *                                 most a quarter of the SMs and K has 32+ 64-wide blocks,
 *                                 or at most half with 128-255 blocks; for swapped small-M
 *                                 problems when two or more slices per tile fit and K has
 *                                 64+ blocks.  About SMs / tiles slices, up to 32, at least 8
 *                                 blocks each.  Not with GEMM_TN_OPT_STREAM_K != 0.
 *   GEMM_TN_OPT_FORCE_SWAP        force operand swapping off (-1) or on (1), 0 = automatic.
 *   GEMM_TN_OPT_FORCE_GENERIC_EPI 1: never use the TMA-store epilogue.
 *   GEMM_TN_OPT_FORCE_PACK        1: repack A and B through scratch even when aligned.
 *   GEMM_TN_OPT_STREAM_K          0 (default): spread the k-blocks of the tiles of a partial
 *                                 last wave over all CTA groups where that was measured to
 *                                 pay (narrow swapped tiles; or 128+ k-blocks per tile, or
 *                                 64 behind three whole waves, with at least 36 k-blocks of
 *                                 the last wave idle and at most 8 contributors per split
 *                                 tile); 1: whenever the tiles do not divide evenly;
 *                                 -1: never.
 *   GEMM_TN_OPT_GROUP_M           rasterisation group: consecutive work units walk this many
 *                                 tile rows column by column (1-64), 0 = automatic.
 *   GEMM_TN_OPT_SERPENTINE        1: every other wave of whole tiles walks K backwards, so it
 *                                 starts on the k-blocks the wave before it loaded last;
 *                                 -1: never; 0 (default): when the tiles span two or more
 *                                 waves and A and B together hold 128 MB or more.
 *   GEMM_TN_OPT_CHECK_TRIM_D      checked build, testing only: bytes (0-4096) taken off the end
 *                                 of D's range in the device-side checks, so that the last
 *                                 stores of a call are reported (GEMM_ERR_BOUNDS) and skipped.
 *                                 No effect in the regular build.
 *   GEMM_TN_OPT_K_CLUSTER         1: swapped small-M problems split K between the two CTAs
 *                                 of a cluster; -1: never; 0 (default): where two K slices and
 *                                 a separate sum would otherwise be planned.
 *   GEMM_TN_OPT_SMALL             small-problem kernel, which applies to K <= 512 / 384 for
 *                                 tiles 64 / 128 wide, K-major operands whose rows tensor
 *                                 copies address as they are and fp32 accumulation, and only
 *                                 while no option of the persistent kernel is forced:
 *                                 -1 never; 1 wherever it applies (tile width 64 when the
 *                                 64-wide tiles fit one wave, else 128); 64 / 128 wherever
 *                                 it applies, with that tile width; 0 (default): where the
 *                                 64-wide tiles fit one wave (batch x ceil(M/128) x
 *                                 ceil(N/64) <= SMs), with that width.
 *   GEMM_TN_OPT_ROW_LOADER        1: K-major operands whose rows tensor copies cannot address
 *                                 are read by the kernel's own loader warps (CTA-pair 256x256
 *                                 and single-CTA 128x128 tiles, unswapped, no K slices)
 *                                 instead of being repacked, so the call needs no scratch
 *                                 for them; several times slower than the repack.  0 (default):
 *                                 repack.
 * A forced setting that no compiled kernel supports for a problem is ignored.
 * Returns GEMM_ERR_INVALID_VALUE for an unknown option or an out-of-range value.
 */
enum {
    GEMM_TN_OPT_WAIT_TIMEOUT_NS = 1,
    GEMM_TN_OPT_SKIP_FIRST_LOAD = 2,
    GEMM_TN_OPT_FORCE_BN = 3,
    GEMM_TN_OPT_FORCE_PAIR = 4,
    GEMM_TN_OPT_FORCE_SPLITS = 5,
    GEMM_TN_OPT_FORCE_SWAP = 6,
    GEMM_TN_OPT_FORCE_GENERIC_EPI = 7,
    GEMM_TN_OPT_FORCE_PACK = 8,
    GEMM_TN_OPT_STREAM_K = 9,
    GEMM_TN_OPT_GROUP_M = 10,
    GEMM_TN_OPT_SERPENTINE = 11,
    GEMM_TN_OPT_ROW_LOADER = 12,
    GEMM_TN_OPT_CHECK_TRIM_D = 13,
    GEMM_TN_OPT_K_CLUSTER = 14,
    GEMM_TN_OPT_SMALL = 15
};
GEMM_TN_API gemm_status_t gemm_tn_f16_set_option(int32_t option, int64_t value);
GEMM_TN_API int64_t gemm_tn_f16_get_option(int32_t option);

/*
 * Split-K GEMM that allocates nothing.  (The pages have no counterpart: this is
 * a service of the library, not a step of the method.)
 *
 * Same operation, arguments and rules as gemm_tn_f16, plus `splits` (number of
 * K slices, 0 = automatic), computed by the split-K tensor-core kernel and its
 * reduction with the fp32 partial sums held in one device array built into the
 * library (GEMM_TN_STATIC_SCRATCH_BYTES per GPU that loads the library, kept
 * until the process exits).  It never calls cudaMalloc, cudaFree or any other
 * allocating routine.  It is meant for callers that must not allocate device
 * memory when they call the GEMM: an allocator or memory pool calling from its
 * own internals (re-entering cudaMalloc there can deadlock), or a service whose
 * device-memory budget is fixed at start-up and whose request path may not
 * allocate (cudaMalloc can synchronise the device and has no latency bound).
 *
 * Limits: splits*M*N*4 bytes must fit in GEMM_TN_STATIC_SCRATCH_BYTES (else
 * GEMM_ERR_WORKSPACE, nothing launched); A and B must be 16-byte aligned with
 * lda and ldb multiples of 8, since there is no scratch for a repacked copy
 * (else GEMM_ERR_MISALIGNED).
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before
 * any stream capture.  All calls on a device share the one array and leave
 * their partial sums in it: calls whose work can overlap on the GPU (for
 * example on two streams with no ordering between them) race and give wrong
 * results.  Nothing in the array needs to start at zero.
 */
#define GEMM_TN_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)
GEMM_TN_API gemm_status_t gemm_tn_f16_splitk_static(const void* A, int64_t lda,
                                                    const void* B, int64_t ldb,
                                                    const void* C, int64_t ldc,
                                                    void* D, int64_t ldd,
                                                    int64_t M, int64_t N, int64_t K,
                                                    float alpha, float beta, int32_t splits,
                                                    gemm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_TN_F16_H */
