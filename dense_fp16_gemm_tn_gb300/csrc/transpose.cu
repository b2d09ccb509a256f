// Matrix transpose y = x^T (y[c][r] = x[r][c]) for fp32 and fp16 matrices: the
// operation the "10-mat-transpose-cute" page optimises on an RTX 4090 (register,
// shared-memory, swizzled and vectorised versions; predicated edges).  On GB300 it
// is purely HBM-bound, so the design is about moving bytes:
//   - 64 x 64 tiles staged through shared memory padded by one 4-byte word per row
//     (reads down a column then hit distinct banks);
//   - 16-byte vector loads along x's rows and 16-byte vector stores along y's rows
//     when both matrices' rows are 16-byte aligned, scalar predicated accesses for
//     edge tiles or unaligned matrices;
//   - a persistent grid of 8 blocks per SM walking the tiles.
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_tn_f16.h"
#include "internal.h"

namespace gtn {
namespace {

constexpr int TILE = 64;
constexpr int THREADS = 256;

template <typename T>
struct Vec;
template <>
struct Vec<uint32_t> {
    static constexpr int N = 4;  // elements per 16-byte vector
};
template <>
struct Vec<uint16_t> {
    static constexpr int N = 8;
};

template <typename T, bool VEC>
__global__ void __launch_bounds__(THREADS) transpose_kernel(const T* __restrict__ X, int64_t ldx, T* __restrict__ Y,
                                                           int64_t ldy, int64_t rows, int64_t cols) {
    constexpr int PAD = 4 / sizeof(T);  // one 4-byte word per row
    __shared__ T tile[TILE][TILE + PAD];
    constexpr int V = VEC ? Vec<T>::N : 1;
    const int64_t tiles_c = (cols + TILE - 1) / TILE;
    const int64_t tiles = ((rows + TILE - 1) / TILE) * tiles_c;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t r0 = (t / tiles_c) * TILE;
        const int64_t c0 = (t % tiles_c) * TILE;
        const bool full = r0 + TILE <= rows && c0 + TILE <= cols;
        if (VEC && full) {
            // x rows: TILE/V vectors each
            for (int e = threadIdx.x; e < TILE * TILE / V; e += THREADS) {
                const int r = e / (TILE / V), cv = e % (TILE / V);
                const uint4 v = *reinterpret_cast<const uint4*>(X + (r0 + r) * ldx + c0 + cv * V);
                const T* pv = reinterpret_cast<const T*>(&v);
#pragma unroll
                for (int i = 0; i < V; ++i) tile[r][cv * V + i] = pv[i];
            }
        } else {
            for (int e = threadIdx.x; e < TILE * TILE; e += THREADS) {
                const int r = e / TILE, c = e % TILE;
                if (r0 + r < rows && c0 + c < cols) tile[r][c] = X[(r0 + r) * ldx + c0 + c];
            }
        }
        __syncthreads();
        if (VEC && full) {
            // y rows (= tile columns): TILE/V vectors each
            for (int e = threadIdx.x; e < TILE * TILE / V; e += THREADS) {
                const int c = e / (TILE / V), rv = e % (TILE / V);
                uint4 v;
                T* pv = reinterpret_cast<T*>(&v);
#pragma unroll
                for (int i = 0; i < V; ++i) pv[i] = tile[rv * V + i][c];
                *reinterpret_cast<uint4*>(Y + (c0 + c) * ldy + r0 + rv * V) = v;
            }
        } else {
            for (int e = threadIdx.x; e < TILE * TILE; e += THREADS) {
                const int c = e / TILE, r = e % TILE;
                if (r0 + r < rows && c0 + c < cols) Y[(c0 + c) * ldy + r0 + r] = tile[r][c];
            }
        }
        __syncthreads();
    }
}

template <typename T>
gemm_status_t transpose_impl(const void* Xv, int64_t ldx, void* Yv, int64_t ldy, int64_t rows, int64_t cols,
                             cudaStream_t stream) {
    if (rows < 0 || cols < 0) return GEMM_ERR_INVALID_VALUE;
    if (rows == 0 || cols == 0) return GEMM_OK;
    if (!Xv || !Yv || ldx < cols || ldy < rows) return GEMM_ERR_INVALID_VALUE;
    const uintptr_t xa = reinterpret_cast<uintptr_t>(Xv), ya = reinterpret_cast<uintptr_t>(Yv);
    if ((xa % sizeof(T)) || (ya % sizeof(T))) return GEMM_ERR_MISALIGNED;
    const uintptr_t xe = xa + sizeof(T) * static_cast<uintptr_t>((rows - 1) * ldx + cols);
    const uintptr_t ye = ya + sizeof(T) * static_cast<uintptr_t>((cols - 1) * ldy + rows);
    if (xa < ye && ya < xe) return GEMM_ERR_INVALID_VALUE;  // in place / overlapping is not supported
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return GEMM_ERR_CUDA;
    const int64_t tiles = ((rows + TILE - 1) / TILE) * ((cols + TILE - 1) / TILE);
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    const int grid = static_cast<int>(tiles < cap ? tiles : cap);
    constexpr int V = Vec<T>::N;
    const bool vec = (xa % 16 == 0) && (ya % 16 == 0) && (ldx % V == 0) && (ldy % V == 0);
    const T* X = static_cast<const T*>(Xv);
    T* Y = static_cast<T*>(Yv);
    if (vec) transpose_kernel<T, true><<<grid, THREADS, 0, stream>>>(X, ldx, Y, ldy, rows, cols);
    else transpose_kernel<T, false><<<grid, THREADS, 0, stream>>>(X, ldx, Y, ldy, rows, cols);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

}  // namespace
}  // namespace gtn

extern "C" GEMM_TN_API gemm_status_t transpose_f32(const void* X, int64_t ldx, void* Y, int64_t ldy, int64_t rows,
                                                   int64_t cols, gemm_stream_t stream) {
    return gtn::transpose_impl<uint32_t>(X, ldx, Y, ldy, rows, cols, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" GEMM_TN_API gemm_status_t transpose_f16(const void* X, int64_t ldx, void* Y, int64_t ldy, int64_t rows,
                                                   int64_t cols, gemm_stream_t stream) {
    return gtn::transpose_impl<uint16_t>(X, ldx, Y, ldy, rows, cols, reinterpret_cast<cudaStream_t>(stream));
}
