// Declarations shared between the host API and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kparams.h"

namespace gtn {

// One compiled tensor-core kernel variant.
struct TcVariant {
    int bn;      // MMA N (columns of the accumulator tile)
    int pair;    // 1 = one CTA per 128-row tile, 2 = CTA pair per 256-row tile
    int stages;  // shared-memory ring depth
    int epi;     // EpiMode
    int sk;      // 1: compiled with the stream-K phase
    int index;   // position in the variant table (for per-device caches)
};

constexpr int kMaxVariants = 96;

// Looks up the compiled variant for (bn, pair, epi, sk); returns false if none exists.
bool find_tc_variant(int bn, int pair, int epi, int sk, TcVariant* out);

// Launches a tensor-core variant with a persistent grid of at most `max_ctas`
// CTAs (rounded to whole CTA pairs).  *grid_out receives the grid used.
cudaError_t launch_tc_variant(const TcVariant& v, const CUtensorMap& tmA, const CUtensorMap& tmB,
                              const CUtensorMap& tmC, const CUtensorMap& tmD, const KParams& p, int64_t max_ctas,
                              cudaStream_t stream, int64_t* grid_out);

// Largest number of CTAs of variant v that can be resident at once on the current device.
int64_t tc_variant_capacity(const TcVariant& v, int sms);

// Device address of the library's error word on the current device.
cudaError_t error_word_address(uint32_t** out);

// One operand to copy into a dense scratch copy whose leading dimension ldo is a multiple of 8.
struct RepackArgs {
    const void* src;
    int64_t ld_src, stride_src;
    void* dst;
    int64_t ldo, rows, K, batch;
    Extent src_ext, dst_ext;  // byte ranges of source and copy (checked build)
};
// Repacks up to two operands in one launch; `err` is the device error word (checked build).
cudaError_t launch_repack(const RepackArgs* ops, int count, int sms, cudaStream_t stream, uint32_t* err);
// Byte ranges of the partial sums, C and D for the checked build's bounds checks.
struct ReduceChecks {
    Extent w, c, d;
    uint32_t* err;
};
cudaError_t launch_splitk_reduce(const float* W, int32_t splits, int64_t M, int64_t N, int64_t batch, float alpha,
                                 float beta, const void* C, int64_t ldc, int64_t strideC, void* D, int64_t ldd,
                                 int64_t strideD, int sms, cudaStream_t stream, const ReduceChecks& chk);
cudaError_t launch_scale(int64_t M, int64_t N, int64_t batch, float beta, const void* C, int64_t ldc,
                         int64_t strideC, void* D, int64_t ldd, int64_t strideD, int sms, cudaStream_t stream,
                         const ReduceChecks& chk);

// Small-problem kernel (small_gemm.cu): one CTA per 128 x bn tile (bn = 64 or 128), grid
// (tiles_m, tiles_n, batch), every k-block of K loaded at once: at most
// small_max_kb(bn) of them (8 or 6, 192 KB of shared memory).  A and B are K-major and
// addressable by tensor copies (boxes of 64 K x 128 rows and 64 K x bn rows); C and D
// of any alignment.
constexpr int small_max_kb(int bn) { return bn == 64 ? 8 : 6; }
struct SmallParams {
    int32_t M, N;           // rows and columns of D per batch entry
    int32_t kb;             // ceil(K / 64), 1..small_max_kb(bn)
    int32_t zA, zB;         // 1: operand has a batch dimension in its tensor map
    float alpha, beta;
    const void* C;          // read when beta != 0
    int64_t ldc, strideC;
    void* D;
    int64_t ldd, strideD;
    uint32_t* err;          // device error word
    uint64_t timeout_ns;    // bound on every wait
    Extent ext_c, ext_d;    // byte ranges of C and D (checked build)
};
cudaError_t launch_small_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const SmallParams& p, int bn,
                              int64_t tiles_m, int64_t tiles_n, int64_t batch, cudaStream_t stream);

// Fused score + softmax statistics kernel (score_softmax.cu).
constexpr int kSoftmaxTileM = 128;  // query rows per work unit
// Keys per score tile of the compiled kernel (the row count of its key boxes).
int softmax_tile_n();
struct SoftmaxParams {
    int32_t M, N;           // query rows and keys per batch entry
    int32_t mblocks;        // ceil(M / kSoftmaxTileM)
    int32_t ntiles;         // ceil(N / softmax_tile_n())
    int64_t num_units;      // batch * mblocks
    float alpha;            // score scale
    float sc;               // alpha * log2(e)
    float* row_max;         // [batch * M]
    float* row_sum;         // [batch * M]
    uint32_t* err;          // device error word
    uint64_t timeout_ns;    // bound on every wait
    int32_t zq, zk;         // 1: operand has a batch dimension in its tensor map
};
// kq = number of 64-wide blocks of the head dimension (1, 2 or 4).
cudaError_t launch_score_softmax(const CUtensorMap& tmQ, const CUtensorMap& tmK, const SoftmaxParams& p, int kq,
                                 int sms, cudaStream_t stream);
// m[i] = mv, l[i] = lv for i < n.
cudaError_t launch_fill_stats(float* m, float* l, int64_t n, float mv, float lv, int sms, cudaStream_t stream);

}  // namespace gtn
