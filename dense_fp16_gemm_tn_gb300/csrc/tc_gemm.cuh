// Persistent, warp-specialised TN GEMM on the sm_100-family tensor cores.
//
//   D[m][n] = alpha * sum_k A[m][k] * B[n][k] + beta * C[m][n]     (per batch entry)
//
// This is the contraction of the "gemm_device 逐行解析" page (section 3: the
// TN inner product tCrC(m,n) += tCsA(m,k)*tCsB(n,k) and the axpby epilogue),
// laid out as in "cute(8) smem_gemm" (section 代码实现: A (M,K) and B (N,K)
// K-contiguous, D (M,N) N-contiguous).  That page's design (cp.async
// global->shared copies, ldmatrix shared->register copies re-tiled with
// retile_D, mma.sync 16x8x16 over a two-level K loop, Swizzle<3,3,3>) targets
// sm_80; here every step is redone for sm_103a:
//
//   warp 0      TMA producer: one thread streams 128x64 A and BNx64 B k-blocks
//               (128-byte swizzle, the layout the tensor core reads) into a
//               STAGES-deep shared-memory ring; `full`/`empty` mbarriers gate
//               each slot (the multi-stage ring the smem_gemm page calls "09").
//   warp 1      MMA issuer: one thread issues tcgen05.mma (M=128 or 256 for a
//               CTA pair, N=BN, K=16, fp16 x fp16 -> fp32) straight from the
//               shared-memory descriptors into a tensor-memory accumulator.
//               There is no shared->register step: the tensor core reads its
//               operands from shared memory itself.
//   warps 2-5   epilogue: tcgen05.ld tensor memory -> registers, alpha/beta in
//               fp32, one round-to-nearest-even to fp16, then TMA stores (or
//               predicated stores for ragged / misaligned outputs).
//
// Two accumulators in tensor memory let the epilogue of one tile overlap the
// main loop of the next.  The grid is persistent: CTA (or CTA pair) i takes
// work units i, i+G, i+2G, ... in an order grouped along M so that tiles
// running at the same time share A and B rows in L2.  A work unit is one
// output tile of one batch entry and, for split-K, one slice of K.
//
// Tails: TMA loads zero-fill rows/columns past M, N and K, and TMA stores
// clip at the tensor bounds, so ragged shapes need no masks on the fast path;
// the predicated epilogues mask element by element.
//
// Every mbarrier wait is bounded: past `timeout_ns` the waiting thread records
// an error word, raises a CTA-wide abort flag and returns; the kernel then lets
// in-flight copies and MMAs drain, frees its tensor memory and exits normally.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>

#include "kparams.h"
#include "ptx.cuh"

namespace gtn {

template <int BN, int PAIR, int STAGES, int EPI>
struct TileCfg {
    static constexpr int BM = 128;               // accumulator rows per CTA (tensor-memory lanes)
    static constexpr int BK = 64;                // halves per 128-byte swizzled row
    static constexpr int BN_LOCAL = BN / PAIR;   // B rows each CTA of a pair loads
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN_LOCAL * BK * 2;
    static constexpr uint32_t STAGE_TX = uint32_t(A_BYTES + B_BYTES) * PAIR;
    static constexpr int EPI_WARPS = 4;
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    static constexpr int TMEM_COLS = (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64 : (2 * BN <= 128) ? 128
                                   : (2 * BN <= 256) ? 256 : 512;
    static constexpr int EPI_WARP_BYTES =
        (EPI == EPI_TMA) ? 2 * 32 * 128 : (EPI == EPI_GENERIC || EPI == EPI_PARTIAL) ? 32 * 33 * 4 : 0;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_EPI = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_BAR = OFF_EPI + ((EPI_WARPS * EPI_WARP_BYTES + 1023) / 1024) * 1024;
    static constexpr int NUM_BARS = 2 * STAGES + 4;
    static constexpr int OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_ABORT = OFF_TMEM_SLOT + 4;
    static constexpr int SMEM_BYTES = OFF_ABORT + 4 + 1024;  // + slack to align the base to 1024

    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "tcgen05 M=128 needs N in [16,256], N%16==0");
    static_assert(BN_LOCAL % 8 == 0, "B tile must hold whole 8-row swizzle atoms");
    static_assert(B_BYTES % 1024 == 0 && A_BYTES % 1024 == 0, "tiles must stay 1024-byte aligned");
    static_assert(EPI != EPI_TMA || BN % 64 == 0, "TMA epilogue stores 64-column chunks");
    static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB of shared memory per CTA");
    static_assert(PAIR == 1 || PAIR == 2, "CTA pair or single CTA");
};

struct Unit {
    int32_t b, tm, tn, kb0, kb1, split;
};

__device__ __forceinline__ Unit decode_unit(const KParams& p, int64_t u) {
    Unit w;
    w.split = static_cast<int32_t>(u % p.splits);
    const int64_t t = u / p.splits;
    const int64_t per_batch = static_cast<int64_t>(p.tiles_m) * p.tiles_n;
    w.b = static_cast<int32_t>(t / per_batch);
    const int64_t r = t % per_batch;
    const int64_t span = static_cast<int64_t>(p.group_m) * p.tiles_n;
    const int32_t first = static_cast<int32_t>(r / span) * p.group_m;
    const int32_t gm = min(p.group_m, p.tiles_m - first);
    const int64_t rr = r % span;
    w.tm = first + static_cast<int32_t>(rr % gm);
    w.tn = static_cast<int32_t>(rr / gm);
    w.kb0 = static_cast<int32_t>((static_cast<int64_t>(w.split) * p.kb_total) / p.splits);
    w.kb1 = static_cast<int32_t>((static_cast<int64_t>(w.split + 1) * p.kb_total) / p.splits);
    return w;
}

// Slow path of a bounded wait.  Returns false (and raises the abort flag) when
// the wait gave up; records the first failure in the device error word.
static __device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, uint32_t* err, uint64_t timeout_ns,
                                       volatile int* abort_flag, uint32_t who) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 15u) == 0) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > timeout_ns) {
                atomicCAS(err, 0u, 0x500u | who);  // 5 = timeout status, low byte = which wait
                *abort_flag = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, uint32_t* err, uint64_t timeout_ns,
                                             volatile int* abort_flag, uint32_t who) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, err, timeout_ns, abort_flag, who);
}

__device__ __forceinline__ void spin_ns(uint64_t ns) {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < ns) {
    }
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

template <int BN, int PAIR, int STAGES, int EPI>
__global__ void __launch_bounds__(TileCfg<BN, PAIR, STAGES, EPI>::THREADS, 1)
gemm_tn_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmD, const KParams p) {
    using Cfg = TileCfg<BN, PAIR, STAGES, EPI>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sA = sbase + Cfg::OFF_A;
    const uint32_t sB = sbase + Cfg::OFF_B;
    const uint32_t bar0 = sbase + Cfg::OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_TMEM_SLOT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_ABORT);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = (PAIR == 2) ? cluster_cta_rank() : 0u;
    const int64_t cluster_id = blockIdx.x / PAIR;
    const int64_t nclusters = gridDim.x / PAIR;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), Cfg::EPI_WARPS * PAIR);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        if constexpr (EPI == EPI_TMA) prefetch_tensormap(&tmD);
    }
    if (warp == 1) tmem_alloc<PAIR>(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tc_fence_before();
    if constexpr (PAIR == 2) cluster_sync(); else __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            bool first = true;
            for (int64_t u = cluster_id; u < p.num_units && ok; u += nclusters) {
                const Unit w = decode_unit(p, u);
                const int32_t rowA = w.tm * (Cfg::BM * PAIR) + Cfg::BM * static_cast<int32_t>(rank);
                const int32_t rowB = w.tn * BN + Cfg::BN_LOCAL * static_cast<int32_t>(rank);
                for (int32_t kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!wait_bounded(empty_bar(stage), phase ^ 1u, p.err, p.timeout_ns, abort_flag, 1)) {
                        ok = false;
                        break;
                    }
                    const bool skip = first && p.debug_skip_first_load && blockIdx.x == 0;
                    first = false;
                    if (!skip) {
                        const uint32_t fb = full_bar(stage);
                        if (rank == 0) mbar_arrive_expect_tx(fb, Cfg::STAGE_TX);
                        const uint32_t dA = sA + stage * Cfg::A_BYTES;
                        const uint32_t dB = sB + stage * Cfg::B_BYTES;
                        if constexpr (PAIR == 1) {
                            tma_load_3d(dA, &tmA, fb, kb * Cfg::BK, rowA, w.b * p.zA);
                            tma_load_3d(dB, &tmB, fb, kb * Cfg::BK, rowB, w.b * p.zB);
                        } else {
                            const uint32_t fl = map_to_cta(fb, 0);
                            tma_load_3d_pair(dA, &tmA, fl, kb * Cfg::BK, rowA, w.b * p.zA);
                            tma_load_3d_pair(dB, &tmB, fl, kb * Cfg::BK, rowB, w.b * p.zB);
                        }
                    }
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            // Drain: wait until the MMA has released every slot, so that no
            // tcgen05.commit arrives on this CTA's barriers after it exits.
            for (int i = 0; i < STAGES && ok; ++i) {
                if (!wait_bounded(empty_bar(stage), phase ^ 1u, p.err, p.timeout_ns, abort_flag, 2)) break;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader CTA only)
        if (rank == 0 && lane == 0) {
            constexpr uint32_t IDESC = idesc_f16_f32(Cfg::BM * PAIR, BN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int64_t u = cluster_id; u < p.num_units && ok; u += nclusters) {
                const Unit w = decode_unit(p, u);
                if (!wait_bounded(tempty_bar(acc), acc_phase ^ 1u, p.err, p.timeout_ns, abort_flag, 3)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int32_t kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!wait_bounded(full_bar(stage), phase, p.err, p.timeout_ns, abort_flag, 4)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t adesc = smem_desc_sw128(sA + stage * Cfg::A_BYTES);
                    const uint64_t bdesc = smem_desc_sw128(sB + stage * Cfg::B_BYTES);
#pragma unroll
                    for (int k = 0; k < Cfg::BK / 16; ++k) {
                        // +32 bytes per 16-wide K step inside the 128-byte swizzled row
                        mma_f16<PAIR>(d_tmem, adesc + 2u * k, bdesc + 2u * k, IDESC,
                                      (kb > w.kb0 || k > 0) ? 1u : 0u);
                    }
                    if constexpr (PAIR == 1) mma_commit(empty_bar(stage));
                    else mma_commit_pair(empty_bar(stage), 0x3);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                if constexpr (PAIR == 1) mma_commit(tfull_bar(acc));
                else mma_commit_pair(tfull_bar(acc), 0x3);
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int ew = warp - 2;
        const int quarter = warp & 3;  // tensor-memory lanes 32*quarter .. +31 are this warp's
        uint8_t* ebuf = smem + Cfg::OFF_EPI + ew * Cfg::EPI_WARP_BYTES;
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t chunk_count = 0;
        const bool use_c = (EPI == EPI_GENERIC || EPI == EPI_SWAP) && p.beta != 0.0f;
        for (int64_t u = cluster_id; u < p.num_units; u += nclusters) {
            const Unit w = decode_unit(p, u);
            // First accumulator row / column of this warp, in the tensor-core view.
            const int64_t arow0 = static_cast<int64_t>(w.tm) * (Cfg::BM * PAIR) + Cfg::BM * rank + quarter * 32;
            const int64_t acol0 = static_cast<int64_t>(w.tn) * BN;
            // Predicated epilogue: C of the first 32-column chunk is fetched before the
            // accumulator is ready, so its memory latency overlaps the main loop.
            __half cnext[32];
            auto load_c_chunk = [&](int c, __half (&dst)[32]) {
                const int64_t col = acol0 + c * 32 + lane;
                const bool col_ok = col < p.N;
                const __half* src = static_cast<const __half*>(p.C) + static_cast<int64_t>(w.b) * p.strideC + col;
#pragma unroll
                for (int r = 0; r < 32; ++r)
                    dst[r] = (col_ok && arow0 + r < p.M) ? src[(arow0 + r) * p.ldc] : __ushort_as_half(0);
            };
            if constexpr (EPI == EPI_GENERIC) {
                if (use_c) load_c_chunk(0, cnext);
            }
            int ok = 1;
            if (lane == 0) ok = wait_bounded(tfull_bar(acc), acc_phase, p.err, p.timeout_ns, abort_flag, 5) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * BN);

            if constexpr (EPI == EPI_TMA) {
#pragma unroll 1
                for (int c = 0; c < BN / 64; ++c) {
                    uint32_t v0[32], v1[32];
                    tmem_ld_32x32b_x32(t_row + c * 64, v0);
                    tmem_ld_32x32b_x32(t_row + c * 64 + 32, v1);
                    tmem_ld_wait();
                    const uint32_t buf = chunk_count & 1u;
                    if (lane == 0) bulk_wait_group_read<1>();
                    __syncwarp();
                    const uint32_t sb = smem_u32(ebuf) + buf * 4096u;
                    const uint32_t row_addr = sb + lane * 128u;
                    const float al = p.alpha;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        st_shared_v4(row_addr + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4),
                                     pack_half2(al * __uint_as_float(v0[8 * j + 0]), al * __uint_as_float(v0[8 * j + 1])),
                                     pack_half2(al * __uint_as_float(v0[8 * j + 2]), al * __uint_as_float(v0[8 * j + 3])),
                                     pack_half2(al * __uint_as_float(v0[8 * j + 4]), al * __uint_as_float(v0[8 * j + 5])),
                                     pack_half2(al * __uint_as_float(v0[8 * j + 6]), al * __uint_as_float(v0[8 * j + 7])));
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        st_shared_v4(row_addr + ((static_cast<uint32_t>(j + 4) ^ (lane & 7u)) << 4),
                                     pack_half2(al * __uint_as_float(v1[8 * j + 0]), al * __uint_as_float(v1[8 * j + 1])),
                                     pack_half2(al * __uint_as_float(v1[8 * j + 2]), al * __uint_as_float(v1[8 * j + 3])),
                                     pack_half2(al * __uint_as_float(v1[8 * j + 4]), al * __uint_as_float(v1[8 * j + 5])),
                                     pack_half2(al * __uint_as_float(v1[8 * j + 6]), al * __uint_as_float(v1[8 * j + 7])));
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&tmD, sb, static_cast<int32_t>(acol0 + c * 64), static_cast<int32_t>(arow0),
                                     w.b * p.zD);
                        bulk_commit_group();
                    }
                    ++chunk_count;
                }
            } else if constexpr (EPI == EPI_GENERIC || EPI == EPI_PARTIAL) {
                // Transpose each 32x32 block through padded shared memory so that a warp
                // reads C and writes D along rows (coalesced), whatever the alignment.
                float* T = reinterpret_cast<float*>(ebuf);
                __half* Dp = static_cast<__half*>(p.D);
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    __half ccur[32];
                    if constexpr (EPI == EPI_GENERIC) {
                        if (use_c) {
#pragma unroll
                            for (int r = 0; r < 32; ++r) ccur[r] = cnext[r];
                            // Loads for the next chunk are issued before this chunk's stores
                            // (different columns, so an aliased C == D stays correct).
                            if (c + 1 < BN / 32) load_c_chunk(c + 1, cnext);
                        }
                    }
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(t_row + c * 32, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) T[lane * 33 + j] = __uint_as_float(v[j]);
                    __syncwarp();
                    const int64_t col = acol0 + c * 32 + lane;
                    if (col < p.N) {
                        if constexpr (EPI == EPI_GENERIC) {
                            __half* dst = Dp + static_cast<int64_t>(w.b) * p.strideD + col;
#pragma unroll
                            for (int r = 0; r < 32; ++r) {
                                const int64_t row = arow0 + r;
                                if (row < p.M) {
                                    float x = p.alpha * T[r * 33 + lane];
                                    if (use_c) x = fmaf(p.beta, __half2float(ccur[r]), x);
                                    dst[row * p.ldd] = __float2half_rn(x);
                                }
                            }
                        } else {
                            float* Wp = p.W + (static_cast<int64_t>(w.b) * p.splits + w.split) * p.M * p.N + col;
#pragma unroll 8
                            for (int r = 0; r < 32; ++r) {
                                const int64_t row = arow0 + r;
                                if (row < p.M) Wp[row * p.N] = T[r * 33 + lane];
                            }
                        }
                    }
                    __syncwarp();
                }
            } else {
                // Swapped operands: accumulator row = problem column n, accumulator column = problem row m.
                const int64_t n = arow0 + lane;
                __half* Dp = static_cast<__half*>(p.D);
                const __half* Cp = static_cast<const __half*>(p.C);
#pragma unroll 1
                for (int c = 0; c < BN / 16; ++c) {
                    uint32_t v[16];
                    tmem_ld_32x32b_x16(t_row + c * 16, v);
                    tmem_ld_wait();
                    if (n < p.N) {
                        if constexpr (EPI == EPI_SWAP) {
                            // all C loads of the chunk first, then the stores
                            __half cv[16];
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const int64_t m = acol0 + c * 16 + j;
                                cv[j] = (use_c && m < p.M)
                                            ? Cp[static_cast<int64_t>(w.b) * p.strideC + m * p.ldc + n]
                                            : __ushort_as_half(0);
                            }
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const int64_t m = acol0 + c * 16 + j;
                                if (m < p.M) {
                                    float x = p.alpha * __uint_as_float(v[j]);
                                    if (use_c) x = fmaf(p.beta, __half2float(cv[j]), x);
                                    Dp[static_cast<int64_t>(w.b) * p.strideD + m * p.ldd + n] = __float2half_rn(x);
                                }
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const int64_t m = acol0 + c * 16 + j;
                                if (m < p.M)
                                    p.W[((static_cast<int64_t>(w.b) * p.splits + w.split) * p.M + m) * p.N + n] =
                                        __uint_as_float(v[j]);
                            }
                        }
                    }
                }
            }
            // This warp is done reading the accumulator: hand it back to the MMA issuer.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR == 1) mbar_arrive(tempty_bar(acc));
                else mbar_arrive_cluster(map_to_cta(tempty_bar(acc), 0));
            }
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
        if constexpr (EPI == EPI_TMA) {
            if (lane == 0) bulk_wait_group<0>();
            __syncwarp();
        }
    }

    // ---------------------------------------------------------------- teardown
    __syncwarp();
    if (*abort_flag) spin_ns(2000000ull);  // let in-flight TMA loads and MMAs land
    tc_fence_before();
    if constexpr (PAIR == 2) cluster_sync(); else __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc<PAIR>(tmem_base, Cfg::TMEM_COLS);
}

}  // namespace gtn
