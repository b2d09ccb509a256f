// Small problems (K of at most 512 / 384 for tiles 64 / 128 wide, and at most one wave of
// tiles): one CTA per 128 x BN tile of D, no persistent scheduling.  Thread 0
// initialises one barrier per k-block and
// issues every k-block's tensor copies at once, before anything else of the set-up,
// so the loads are in flight while tensor memory is allocated; it then issues the
// tile's MMAs (128 x BN x 16, fp16 in, fp32 accumulate) into tensor memory as each
// k-block lands.  The four warps read their 32 accumulator rows each and write
// D = RNE(alpha * acc + beta * C) straight from registers, 16 bytes at a time where a
// row's elements are 16-byte aligned and in bounds, element by element elsewhere.
// The persistent kernel's set-up (ring barriers, tile scheduling with 64-bit
// divisions, staging buffers, TMA stores) costs a single-tile launch more than its
// main loop; here the work is the same contraction as the gemm_device page's
// section 3 (each D element the K-long inner product of a row of A and a row of B,
// then the axpby epilogue).
#include <cuda_fp16.h>

#include <mutex>

#include "checked.h"
#include "internal.h"
#include "ptx.cuh"

namespace gtn {
namespace {

constexpr int kSmallThreads = 128;

template <int BN>
struct SmallCfg {
    static constexpr int A_BYTES = 128 * 128;  // 128 rows x 64 halves, 128-byte swizzle
    static constexpr int B_BYTES = BN * 128;   // BN rows x 64 halves
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int MAX_KB = small_max_kb(BN);           // every k-block resident at once
    static constexpr int OFF_BAR = MAX_KB * STAGE;            // MAX_KB full barriers + done
    static constexpr int OFF_SLOT = OFF_BAR + 8 * (MAX_KB + 1);
    static constexpr int OFF_ABORT = OFF_SLOT + 8;
    static constexpr int SMEM_BYTES = OFF_ABORT + 8 + 1024;  // + slack to align the base to 1024
    static constexpr uint32_t TMEM_COLS = BN;                 // a power of two >= 32
    static_assert(BN == 64 || BN == 128, "tile widths of the small-problem kernel");
    static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "swizzled tiles start on 1024-byte boundaries");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory of one CTA");
};

// Bounded wait on a barrier phase; on timeout records 0x500 | who and raises the CTA's
// abort flag.  Returns false on timeout or when another thread has aborted.
__device__ __forceinline__ bool small_wait(uint32_t bar, uint32_t parity, const SmallParams& p,
                                           volatile int* abort_flag, uint32_t who) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait_ns(bar, parity, 32)) return true;
        if ((i & 15u) == 0) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > p.timeout_ns) {
                atomicCAS(p.err, 0u, 0x500u | who);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

template <int BN>
__global__ void __launch_bounds__(kSmallThreads, 1)
gemm_small_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const SmallParams p) {
    using Cfg = SmallCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + Cfg::OFF_BAR;
    const uint32_t done_bar = bar0 + 8u * Cfg::MAX_KB;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_SLOT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_ABORT);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int32_t tm = static_cast<int32_t>(blockIdx.x), tn = static_cast<int32_t>(blockIdx.y);
    const int32_t b = static_cast<int32_t>(blockIdx.z);
    const int nkb = p.kb;

    if (threadIdx.x == 0) {
        for (int k = 0; k < nkb; ++k) mbar_init(bar0 + 8u * k, 1);
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
        for (int k = 0; k < nkb; ++k) {
            const uint32_t fb = bar0 + 8u * k;
            const uint32_t dst = sbase + static_cast<uint32_t>(k * Cfg::STAGE);
            mbar_arrive_expect_tx(fb, Cfg::STAGE);
            tma_load_3d(dst, &tmA, fb, k * 64, tm * 128, p.zA ? b : 0);
            tma_load_3d(dst + Cfg::A_BYTES, &tmB, fb, k * 64, tn * BN, p.zB ? b : 0);
        }
    }
    if (warp == 1) tmem_alloc<1>(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (threadIdx.x == 0) {
        // K-major tiles: each 16-wide K step is 32 bytes further along the 128-byte rows.
        constexpr uint32_t IDESC = idesc_f16_f32(128, BN);
        bool ok = true;
        for (int k = 0; k < nkb; ++k) {
            if (!small_wait(bar0 + 8u * k, 0, p, abort_flag, 0x11)) {
                ok = false;
                break;
            }
            const uint32_t st = sbase + static_cast<uint32_t>(k * Cfg::STAGE);
            const uint64_t ad = smem_desc_sw128(st), bd = smem_desc_sw128(st + Cfg::A_BYTES);
#pragma unroll
            for (int j = 0; j < 4; ++j) mma_f16<1>(tmem, ad + 2u * j, bd + 2u * j, IDESC, (k > 0 || j > 0) ? 1u : 0u);
        }
        if (ok) mma_commit(done_bar);
    }

    // C of this thread's row, read while the loads and MMAs run (beta != 0): a load per
    // 8-column group, all in flight together, 16 bytes where the group is whole and aligned.
    const int64_t row = static_cast<int64_t>(tm) * 128 + warp * 32 + lane;
    const bool live = row < p.M;
    const bool use_c = p.beta != 0.0f;
    uint4 cw[BN / 8];
#pragma unroll
    for (int g = 0; g < BN / 8; ++g) cw[g] = make_uint4(0u, 0u, 0u, 0u);
    if (use_c && live) {
        const __half* Crow = static_cast<const __half*>(p.C) + static_cast<int64_t>(b) * p.strideC + row * p.ldc;
#pragma unroll
        for (int g = 0; g < BN / 8; ++g) {
            const int64_t col = static_cast<int64_t>(tn) * BN + 8 * g;
            if (col >= p.N) break;
            const __half* ca = Crow + col;
            if (col + 8 <= p.N && (reinterpret_cast<uintptr_t>(ca) & 15u) == 0) {
                if (!kChecked || in_extent(reinterpret_cast<uintptr_t>(ca), reinterpret_cast<uintptr_t>(ca + 8),
                                           p.ext_c, p.err, CHK_EPI_C_ELEM))
                    cw[g] = *reinterpret_cast<const uint4*>(ca);
            } else {
                __half* ch = reinterpret_cast<__half*>(&cw[g]);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (col + j < p.N && chk_elem(ca + j, p.ext_c, p.err, CHK_EPI_C_ELEM)) ch[j] = ca[j];
            }
        }
    }

    int got = 1;
    if (lane == 0) got = small_wait(done_bar, 0, p, abort_flag, 0x12) ? 1 : 0;
    got = __shfl_sync(0xffffffffu, got, 0);
    if (got) {
        tc_fence_after();
        __half* Drow = static_cast<__half*>(p.D) + static_cast<int64_t>(b) * p.strideD + row * p.ldd;
        const uint32_t t_row = tmem + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32), v);
            tmem_ld_wait();
            if (!live) continue;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const int64_t col = static_cast<int64_t>(tn) * BN + c * 32 + 8 * g;
                if (col >= p.N) break;
                float x[8];
                const __half* ch = reinterpret_cast<const __half*>(&cw[c * 4 + g]);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    x[j] = p.alpha * __uint_as_float(v[8 * g + j]);
                    if (use_c) x[j] = fmaf(p.beta, __half2float(ch[j]), x[j]);
                }
                __half* da = Drow + col;
                if (col + 8 <= p.N && (reinterpret_cast<uintptr_t>(da) & 15u) == 0) {
                    if (!kChecked || in_extent(reinterpret_cast<uintptr_t>(da), reinterpret_cast<uintptr_t>(da + 8),
                                               p.ext_d, p.err, CHK_EPI_D_ELEM))
                        *reinterpret_cast<uint4*>(da) =
                            make_uint4(pack2(x[0], x[1]), pack2(x[2], x[3]), pack2(x[4], x[5]), pack2(x[6], x[7]));
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (col + j < p.N && chk_elem(da + j, p.ext_d, p.err, CHK_EPI_D_ELEM))
                            da[j] = __float2half_rn(x[j]);
                }
            }
        }
    }

    __syncwarp();
    if (*abort_flag) {  // let tensor copies and MMAs still in flight land before the memory goes
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 2000000ull) {
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc<1>(tmem, Cfg::TMEM_COLS);
}

template <int BN>
cudaError_t launch_bn(const CUtensorMap& tmA, const CUtensorMap& tmB, const SmallParams& p, int64_t tiles_m,
                      int64_t tiles_n, int64_t batch, cudaStream_t stream) {
    using Cfg = SmallCfg<BN>;
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 0 || dev >= 64 || !done[dev]) {
            e = cudaFuncSetAttribute(gemm_small_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) done[dev] = true;
        }
    }
    const dim3 grid(static_cast<unsigned>(tiles_m), static_cast<unsigned>(tiles_n), static_cast<unsigned>(batch));
    gemm_small_kernel<BN><<<grid, kSmallThreads, Cfg::SMEM_BYTES, stream>>>(tmA, tmB, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_small_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const SmallParams& p, int bn,
                              int64_t tiles_m, int64_t tiles_n, int64_t batch, cudaStream_t stream) {
    if (p.kb < 1 || p.kb > small_max_kb(bn) || tiles_m < 1 || tiles_n < 1 || batch < 1 || tiles_m > 0x7fffffff ||
        tiles_n > 65535 || batch > 65535)
        return cudaErrorInvalidValue;
    if (bn == 64) return launch_bn<64>(tmA, tmB, p, tiles_m, tiles_n, batch, stream);
    if (bn == 128) return launch_bn<128>(tmA, tmB, p, tiles_m, tiles_n, batch, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gtn
