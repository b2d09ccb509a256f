// Memory-bound helper kernels around the tensor-core GEMM:
//   - repack: copies an operand whose rows do not start on 16-byte boundaries
//     (leading dimension not a multiple of 8 halves, or a misaligned base)
//     into a dense scratch copy with an aligned leading dimension, so the
//     tensor-core kernel can fetch it with TMA;
//   - split-K reduction: D = alpha * sum_s W[s] + beta * C, summing the fp32
//     partial sums of the K slices in slice order (deterministic);
//   - scale: the K == 0 case, D = beta * C (or 0).
// All are grid-stride loops with coalesced accesses along the contiguous
// dimension; grids are sized in multiples of the SM count by the caller.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace gtn {

// dst[b][r][0..ldo) = src[b][r][0..K) followed by zeros; ldo % 8 == 0 and dst 16-byte aligned.
// One thread writes one 16-byte group of 8 halves.
__global__ void repack_rows_kernel(const __half* __restrict__ src, int64_t ld_src, int64_t stride_src,
                                   __half* __restrict__ dst, int64_t ldo, int64_t rows, int64_t K,
                                   int64_t batch) {
    const int64_t groups_per_row = ldo / 8;
    const int64_t total = batch * rows * groups_per_row;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t g = i % groups_per_row;
        const int64_t rb = i / groups_per_row;  // b * rows + r
        const int64_t r = rb % rows;
        const int64_t b = rb / rows;
        const __half* s = src + b * stride_src + r * ld_src;
        const int64_t k0 = g * 8;
        alignas(16) __half v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = (k0 + j < K) ? s[k0 + j] : __ushort_as_half(0);
        *reinterpret_cast<uint4*>(dst + rb * ldo + k0) = *reinterpret_cast<const uint4*>(v);
    }
}

// D[b][m][n] = alpha * sum_{s<S} W[b][s][m][n] + beta * C[b][m][n]
__global__ void splitk_reduce_kernel(const float* __restrict__ W, int32_t splits, int64_t M, int64_t N,
                                     int64_t batch, float alpha, float beta, const __half* C, int64_t ldc,
                                     int64_t strideC, __half* D, int64_t ldd, int64_t strideD) {
    const int64_t mn = M * N;
    const int64_t total = batch * mn;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t b = i / mn;
        const int64_t e = i % mn;
        const int64_t m = e / N;
        const int64_t n = e % N;
        const float* w = W + b * splits * mn + e;
        float acc = 0.0f;
        for (int32_t s = 0; s < splits; ++s) acc += w[s * mn];
        float x = alpha * acc;
        if (beta != 0.0f) x = fmaf(beta, __half2float(C[b * strideC + m * ldc + n]), x);
        D[b * strideD + m * ldd + n] = __float2half_rn(x);
    }
}

// D = beta * C (beta != 0) or D = 0.
__global__ void scale_kernel(int64_t M, int64_t N, int64_t batch, float beta, const __half* C, int64_t ldc,
                             int64_t strideC, __half* D, int64_t ldd, int64_t strideD) {
    const int64_t mn = M * N;
    const int64_t total = batch * mn;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t b = i / mn;
        const int64_t e = i % mn;
        const int64_t m = e / N;
        const int64_t n = e % N;
        float x = 0.0f;
        if (beta != 0.0f) x = beta * __half2float(C[b * strideC + m * ldc + n]);
        D[b * strideD + m * ldd + n] = __float2half_rn(x);
    }
}

static int grid_for(int64_t total, int threads, int sms) {
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(sms) * 8;  // 8 resident 256-thread blocks per SM
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return static_cast<int>(blocks);
}

cudaError_t launch_repack(const void* src, int64_t ld_src, int64_t stride_src, void* dst, int64_t ldo, int64_t rows,
                          int64_t K, int64_t batch, int sms, cudaStream_t stream) {
    const int64_t total = batch * rows * (ldo / 8);
    repack_rows_kernel<<<grid_for(total, 256, sms), 256, 0, stream>>>(
        static_cast<const __half*>(src), ld_src, stride_src, static_cast<__half*>(dst), ldo, rows, K, batch);
    return cudaGetLastError();
}

cudaError_t launch_splitk_reduce(const float* W, int32_t splits, int64_t M, int64_t N, int64_t batch, float alpha,
                                 float beta, const void* C, int64_t ldc, int64_t strideC, void* D, int64_t ldd,
                                 int64_t strideD, int sms, cudaStream_t stream) {
    splitk_reduce_kernel<<<grid_for(batch * M * N, 256, sms), 256, 0, stream>>>(
        W, splits, M, N, batch, alpha, beta, static_cast<const __half*>(C), ldc, strideC, static_cast<__half*>(D),
        ldd, strideD);
    return cudaGetLastError();
}

cudaError_t launch_scale(int64_t M, int64_t N, int64_t batch, float beta, const void* C, int64_t ldc,
                         int64_t strideC, void* D, int64_t ldd, int64_t strideD, int sms, cudaStream_t stream) {
    scale_kernel<<<grid_for(batch * M * N, 256, sms), 256, 0, stream>>>(
        M, N, batch, beta, static_cast<const __half*>(C), ldc, strideC, static_cast<__half*>(D), ldd, strideD);
    return cudaGetLastError();
}

}  // namespace gtn
