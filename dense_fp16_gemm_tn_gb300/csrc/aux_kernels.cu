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
#include "ptx.cuh"

namespace gtn {

struct RepackJob {
    const __half* src;
    int64_t ld_src, stride_src;
    __half* dst;
    int64_t ldo, rows, K, batch;
    Extent src_ext, dst_ext;
};

// The 16 bytes starting `shift` bytes (even, 0..14) into the 32-byte window w0..w7.
// `shift` is the same for every group of a row, so the switch does not diverge.
__device__ __forceinline__ uint4 window16(const uint32_t (&w)[8], uint32_t shift) {
    const bool half = (shift & 2u) != 0;
    auto f = [&](uint32_t lo, uint32_t hi) { return half ? __funnelshift_r(lo, hi, 16) : lo; };
    switch (shift >> 2) {
        case 0: return make_uint4(f(w[0], w[1]), f(w[1], w[2]), f(w[2], w[3]), f(w[3], w[4]));
        case 1: return make_uint4(f(w[1], w[2]), f(w[2], w[3]), f(w[3], w[4]), f(w[4], w[5]));
        case 2: return make_uint4(f(w[2], w[3]), f(w[3], w[4]), f(w[4], w[5]), f(w[5], w[6]));
        default: return make_uint4(f(w[3], w[4]), f(w[4], w[5]), f(w[5], w[6]), f(w[6], w[7]));
    }
}

// dst[b][r][0..ldo) = src[b][r][0..K) followed by zeros, for up to two operands in one
// launch; ldo % 8 == 0 and dst 16-byte aligned.  A lane writes 16-byte groups of 8
// halves.  Their source halves start at any 2-byte boundary: the lane loads the
// aligned 16-byte block holding the first one and, when the group straddles into the
// next block and that block holds a half of the row, that block too, then shifts
// the 32-byte window into place.  No load leaves the blocks that hold row data.
// A warp takes a span of 32 x kRepackGroups groups of one row at a time (the index
// arithmetic once per span); a lane takes kRepackGroups groups 32 apart, so a warp's
// stores cover 512 contiguous bytes and each lane has up to 2 x kRepackGroups loads
// in flight.
constexpr int kRepackGroups = 4;

constexpr int kMaxRepackJobs = 2;
struct RepackJobs {
    RepackJob j[kMaxRepackJobs];
    int64_t first_item[kMaxRepackJobs + 1];  // job i owns items [first_item[i], first_item[i + 1])
    uint32_t* err;                           // device error word (checked build)
};

__global__ void __launch_bounds__(256, 4) repack_rows_kernel(const RepackJobs jobs) {
    constexpr int32_t kSpan = 32 * kRepackGroups;  // groups of one work item
    // The GEMM that reads these copies may start its set-up now; it waits for this
    // grid's completion before its first load.
    griddep_launch_dependents();
    const int64_t items_total = jobs.first_item[kMaxRepackJobs];
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    // work item = (row, span of kSpan groups): a warp takes items w, w + nwarps, ...
    for (int64_t item = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; item < items_total;
         item += nwarps) {
        const int ji = item >= jobs.first_item[2] ? 2 : item >= jobs.first_item[1] ? 1 : 0;
        const RepackJob& jb = jobs.j[ji];
        const int64_t it = item - jobs.first_item[ji];
        const int64_t cpr = (jb.ldo / 8 + kSpan - 1) / kSpan;
        const int64_t rb = it / cpr;  // b * rows + r
        const int32_t span0 = static_cast<int32_t>(it - rb * cpr) * kSpan;
        const int64_t bi = jb.batch > 1 ? rb / jb.rows : 0;
        const int64_t r = rb - bi * jb.rows;
        const __half* src_row = jb.src + bi * jb.stride_src + r * jb.ld_src;
        __half* dst_row = jb.dst + rb * jb.ldo;
        const int32_t groups = static_cast<int32_t>(jb.ldo / 8);
        const int32_t K = static_cast<int32_t>(jb.K);
        const uint32_t shift = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(src_row) & 15u);  // bytes, even
        const uint4* row_blk = reinterpret_cast<const uint4*>(reinterpret_cast<uintptr_t>(src_row) - shift);
        // a group's window reaches into the following block when element k0 + (16 - shift) / 2 < K
        const int32_t reach = static_cast<int32_t>((16u - shift) / 2u);
        {
            const int32_t g0 = span0;
            uint32_t w[kRepackGroups][8];
#pragma unroll
            for (int u = 0; u < kRepackGroups; ++u) {
                const int32_t g = g0 + u * 32 + lane;
                const int32_t k0 = g * 8;
#pragma unroll
                for (int t = 0; t < 8; ++t) w[u][t] = 0;
                bool load_ok = g < groups && k0 < K;
                if constexpr (kChecked) {
                    // the halves of the row this group uses must lie inside the source matrix
                    if (load_ok) {
                        const uint64_t a = reinterpret_cast<uintptr_t>(src_row + k0);
                        const uint64_t b = reinterpret_cast<uintptr_t>(src_row + (k0 + 8 < K ? k0 + 8 : K));
                        load_ok = in_extent(a, b, jb.src_ext, jobs.err, CHK_REPACK_SRC);
                    }
                }
                if (load_ok) {
                    const uint4 v0 = __ldg(row_blk + g);
                    w[u][0] = v0.x; w[u][1] = v0.y; w[u][2] = v0.z; w[u][3] = v0.w;
                    if (shift != 0 && k0 + reach < K) {
                        const uint4 v1 = __ldg(row_blk + g + 1);
                        w[u][4] = v1.x; w[u][5] = v1.y; w[u][6] = v1.z; w[u][7] = v1.w;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kRepackGroups; ++u) {
                const int32_t g = g0 + u * 32 + lane;
                if (g >= groups) break;
                const int32_t k0 = g * 8;
                uint4 out = make_uint4(0, 0, 0, 0);
                if (k0 < K) {
                    out = window16(w[u], shift);
                    // zero the halves past the end of the row
                    const int32_t valid = K - k0;
                    if (valid < 8) {
                        uint32_t o[4] = {out.x, out.y, out.z, out.w};
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            if (2 * t >= valid) o[t] = 0;
                            else if (2 * t + 1 >= valid) o[t] &= 0xFFFFu;
                        }
                        out = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
                if (chk_elem(reinterpret_cast<const uint4*>(dst_row + k0), jb.dst_ext, jobs.err, CHK_REPACK_DST))
                    *reinterpret_cast<uint4*>(dst_row + k0) = out;
            }
        }
    }
}

// D[b][m][n] = alpha * sum_{s<S} W[b][s][m][n] + beta * C[b][m][n], four consecutive n per
// thread (N % 4 == 0): 16-byte loads of the partials, up to eight slices' loads in flight,
// added in slice order.
__global__ void splitk_reduce4_kernel(const float* __restrict__ W, int32_t splits, int64_t M, int64_t N,
                                      int64_t batch, float alpha, float beta, const __half* C, int64_t ldc,
                                      int64_t strideC, __half* D, int64_t ldd, int64_t strideD,
                                      const ReduceChecks chk) {
    griddep_wait();  // launched as a dependent of the GEMM that writes W: its partials are visible
    const int64_t mn = M * N;
    const int64_t total = batch * mn / 4;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t e4 = i * 4;
        const int64_t b = e4 / mn;
        const int64_t e = e4 - b * mn;
        const int64_t m = e / N;
        const int64_t n = e - m * N;
        const float4* w = reinterpret_cast<const float4*>(W + b * splits * mn + e);
        const int64_t step = mn / 4;
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int32_t s0 = 0; s0 < splits; s0 += 8) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (s0 + u < splits && chk_elem(w + (s0 + u) * step, chk.w, chk.err, CHK_REDUCE_W))
                    v[u] = __ldcs(w + (s0 + u) * step);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (s0 + u < splits) {
                    acc[0] += v[u].x;
                    acc[1] += v[u].y;
                    acc[2] += v[u].z;
                    acc[3] += v[u].w;
                }
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float x = alpha * acc[q];
            const __half* ca = C + b * strideC + m * ldc + n + q;
            if (beta != 0.0f && chk_elem(ca, chk.c, chk.err, CHK_REDUCE_C)) x = fmaf(beta, __half2float(*ca), x);
            __half* da = D + b * strideD + m * ldd + n + q;
            if (chk_elem(da, chk.d, chk.err, CHK_REDUCE_D)) *da = __float2half_rn(x);
        }
    }
}

// D[b][m][n] = alpha * sum_{s<S} W[b][s][m][n] + beta * C[b][m][n]
__global__ void splitk_reduce_kernel(const float* __restrict__ W, int32_t splits, int64_t M, int64_t N,
                                     int64_t batch, float alpha, float beta, const __half* C, int64_t ldc,
                                     int64_t strideC, __half* D, int64_t ldd, int64_t strideD,
                                     const ReduceChecks chk) {
    griddep_wait();  // launched as a dependent of the GEMM that writes W: its partials are visible
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
        for (int32_t s = 0; s < splits; ++s)
            if (chk_elem(w + s * mn, chk.w, chk.err, CHK_REDUCE_W)) acc += w[s * mn];
        float x = alpha * acc;
        const __half* ca = C + b * strideC + m * ldc + n;
        if (beta != 0.0f && chk_elem(ca, chk.c, chk.err, CHK_REDUCE_C)) x = fmaf(beta, __half2float(*ca), x);
        __half* da = D + b * strideD + m * ldd + n;
        if (chk_elem(da, chk.d, chk.err, CHK_REDUCE_D)) *da = __float2half_rn(x);
    }
}

// D = beta * C (beta != 0) or D = 0.
__global__ void scale_kernel(int64_t M, int64_t N, int64_t batch, float beta, const __half* C, int64_t ldc,
                             int64_t strideC, __half* D, int64_t ldd, int64_t strideD, const ReduceChecks chk) {
    const int64_t mn = M * N;
    const int64_t total = batch * mn;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t b = i / mn;
        const int64_t e = i % mn;
        const int64_t m = e / N;
        const int64_t n = e % N;
        float x = 0.0f;
        const __half* ca = C + b * strideC + m * ldc + n;
        if (beta != 0.0f && chk_elem(ca, chk.c, chk.err, CHK_REDUCE_C)) x = beta * __half2float(*ca);
        __half* da = D + b * strideD + m * ldd + n;
        if (chk_elem(da, chk.d, chk.err, CHK_REDUCE_D)) *da = __float2half_rn(x);
    }
}

static int grid_for(int64_t total, int threads, int sms) {
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(sms) * 8;  // 8 resident 256-thread blocks per SM
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return static_cast<int>(blocks);
}

cudaError_t launch_repack(const RepackArgs* ops, int count, int sms, cudaStream_t stream, uint32_t* err) {
    if (count > kMaxRepackJobs) return cudaErrorInvalidValue;
    RepackJobs jobs = {};
    jobs.err = err;
    constexpr int64_t kSpan = 32 * kRepackGroups;
    int64_t items = 0;
    for (int i = 0; i < kMaxRepackJobs; ++i) {
        jobs.first_item[i] = items;
        if (i < count) {
            const RepackArgs& o = ops[i];
            jobs.j[i] = {static_cast<const __half*>(o.src), o.ld_src, o.stride_src, static_cast<__half*>(o.dst),
                         o.ldo, o.rows, o.K, o.batch, o.src_ext, o.dst_ext};
            items += o.batch * o.rows * ((o.ldo / 8 + kSpan - 1) / kSpan);
        }
    }
    jobs.first_item[kMaxRepackJobs] = items;
    if (items == 0) return cudaSuccess;
    // a warp per span: 256-thread blocks, up to 4 blocks per SM (all resident)
    const int64_t want = (items + 7) / 8;
    int64_t blocks = want < static_cast<int64_t>(sms) * 4 ? want : static_cast<int64_t>(sms) * 4;
    repack_rows_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(jobs);
    return cudaGetLastError();
}

cudaError_t launch_splitk_reduce(const float* W, int32_t splits, int64_t M, int64_t N, int64_t batch, float alpha,
                                 float beta, const void* C, int64_t ldc, int64_t strideC, void* D, int64_t ldd,
                                 int64_t strideD, int sms, cudaStream_t stream, const ReduceChecks& chk) {
    // A programmatic dependent of the GEMM before it on the stream: scheduled while that
    // GEMM runs, it waits for the GEMM's completion before reading the partials.
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (N % 4 == 0) {
        cfg.gridDim = dim3(static_cast<unsigned>(grid_for(batch * M * N / 4, 256, sms)), 1, 1);
        return cudaLaunchKernelEx(&cfg, splitk_reduce4_kernel, W, splits, M, N, batch, alpha, beta,
                                  static_cast<const __half*>(C), ldc, strideC, static_cast<__half*>(D), ldd, strideD,
                                  chk);
    }
    cfg.gridDim = dim3(static_cast<unsigned>(grid_for(batch * M * N, 256, sms)), 1, 1);
    return cudaLaunchKernelEx(&cfg, splitk_reduce_kernel, W, splits, M, N, batch, alpha, beta,
                              static_cast<const __half*>(C), ldc, strideC, static_cast<__half*>(D), ldd, strideD, chk);
}

cudaError_t launch_scale(int64_t M, int64_t N, int64_t batch, float beta, const void* C, int64_t ldc,
                         int64_t strideC, void* D, int64_t ldd, int64_t strideD, int sms, cudaStream_t stream,
                         const ReduceChecks& chk) {
    scale_kernel<<<grid_for(batch * M * N, 256, sms), 256, 0, stream>>>(
        M, N, batch, beta, static_cast<const __half*>(C), ldc, strideC, static_cast<__half*>(D), ldd, strideD, chk);
    return cudaGetLastError();
}

}  // namespace gtn
