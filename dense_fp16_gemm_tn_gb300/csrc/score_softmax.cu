// Fused score GEMM + scale + online softmax statistics:
//
//   s_ij = alpha * sum_k Q[b][i][k] * K[b][j][k]
//   m_i  = max_j s_ij,   l_i = sum_j exp(s_ij - m_i)
//
// The score step is the Q @ K.T of "为什么 cutlass_cute_tutorial_zh.md 中要用
// retile_D" (section 1: Q is the MMA's A operand, K its B operand); the
// statistics are the running maximum and normaliser that online softmax keeps
// per query row.  Only m and l leave the chip: the batch x M x N score matrix
// is never written to memory.
//
// One CTA per SM, persistent over units (batch entry, 128-row query block);
// units are taken in batch-major order so that the CTAs running at the same
// time share a few heads' keys through L2.  Warp roles:
//   warp 0      TMA producer: the unit's Q block (d / 64 boxes of 128 x 64, two
//               buffers) and a ring of key boxes (256 keys x 64 halves);
//   warp 1      tcgen05.mma issuer: S tile (128 x 256, fp32) into one of two
//               tensor-memory buffers (2 x 256 columns);
//   warps 2-9   softmax: warp w reads tensor-memory lanes 32*(w%4).. (one query
//               row per thread) of every other S tile (the tiles of buffer
//               (w-2)/4), so the two warps sharing a lane quarter alternate between
//               loading and folding; each keeps the row's running extreme of the
//               raw scores and the sum of 2^(t - t_max) in base-2 units
//               (t = s * log2 e), rescaling the sum when the maximum grows; the two
//               partial states of a row are merged through shared memory at the
//               end of the unit.
// Every wait is bounded (same error word and abort protocol as the GEMM).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace gtn {
namespace {

constexpr int SM_BM = kSoftmaxTileM;  // query rows per unit
constexpr int SM_BN = 256;            // keys per S tile
constexpr int SM_BK = 64;          // halves per box row (128 bytes)
constexpr int SM_EPI_WARPS = 8;
constexpr int SM_THREADS = 32 * (2 + SM_EPI_WARPS);
constexpr uint32_t SM_Q_BOX = SM_BM * SM_BK * 2;   // 16 KB
constexpr uint32_t SM_K_BOX = SM_BN * SM_BK * 2;   // 32 KB
constexpr uint32_t SM_TMEM_COLS = 2 * SM_BN;       // two S buffers

template <int KQ>
struct SmCfg {
    static constexpr int QBUF = 2;
    static constexpr uint32_t Q_BYTES = KQ * SM_Q_BOX;  // one query block, all of d
    static constexpr int STAGES_RAW = static_cast<int>((220u * 1024u - QBUF * Q_BYTES) / SM_K_BOX);
    static constexpr int STAGES = STAGES_RAW > 6 ? 6 : STAGES_RAW;
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + QBUF * Q_BYTES;
    static constexpr uint32_t OFF_MERGE = OFF_K + STAGES * SM_K_BOX;        // [2][128] float2
    static constexpr uint32_t OFF_BAR = OFF_MERGE + 2 * SM_BM * 8;
    static constexpr int NUM_BARS = 2 * STAGES + 2 + 2 + 2 + 2 + 2 + 2;
    static constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + 8 * NUM_BARS;
    static constexpr uint32_t OFF_ABORT = OFF_TMEM_SLOT + 8;
    static constexpr uint32_t SMEM = OFF_ABORT + 8 + 1024;  // + alignment slack
    static_assert(STAGES >= 2, "key ring too shallow");
    static_assert(SM_BM == 128 && SM_BN == 256, "one tensor-memory lane per query row; two 128-column halves");
    static_assert(SMEM <= 232448, "shared memory budget");
};

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float min3f(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Waits for the outstanding tcgen05.ld of this thread; the registers are passed
// through so that no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
          "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
          "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
          "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
        :
        : "memory");
}

// Waits here sit on the critical path of a tight producer/consumer chain: a short
// suspension bound lets a waiter see a completed phase promptly.
constexpr uint32_t kSuspendNs = 32;

static __device__ __noinline__ bool sm_wait_slow(uint32_t bar, uint32_t parity, uint32_t* err, uint64_t timeout_ns,
                                                 volatile int* abort_flag, uint32_t who) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait_ns(bar, parity, kSuspendNs)) return true;
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

__device__ __forceinline__ void sm_spin_ns(uint64_t ns) {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < ns) {
    }
}

__device__ __forceinline__ bool sm_wait(uint32_t bar, uint32_t parity, uint32_t* err, uint64_t timeout_ns,
                                        volatile int* abort_flag, uint32_t who) {
    if (mbar_try_wait_ns(bar, parity, kSuspendNs)) return true;
    return sm_wait_slow(bar, parity, err, timeout_ns, abort_flag, who);
}

// Running state of one query row over the columns one warp has folded: the
// extreme (maximum for alpha >= 0, minimum for alpha < 0) of the raw fp32 scores,
// and the sum of 2^(t - ref), t = score * sc with sc = alpha * log2(e), where the
// reference ref is the base-2 running maximum ext * sc.
struct RowState {
    float ext;  // raw score extreme (+-inf before the first column)
    float ref;  // ext * sc (-inf before the first column)
    float l;    // sum of 2^(t_j - ref)
};

__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }

// Folds 32 consecutive scores (the first `valid` of them real columns) into the state.
template <bool NEG, bool MASKED>
__device__ __forceinline__ void fold_chunk(const uint32_t (&r)[32], int valid, float sc, RowState& st) {
    float v[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        v[k] = __uint_as_float(r[k]);
        if (MASKED && k >= valid) v[k] = NEG ? __int_as_float(0x7f800000) : __int_as_float(0xff800000);
    }
    // extreme of the chunk: a tree of 3-input min / max
    float a[11];
#pragma unroll
    for (int k = 0; k < 10; ++k) a[k] = NEG ? min3f(v[3 * k], v[3 * k + 1], v[3 * k + 2])
                                           : max3f(v[3 * k], v[3 * k + 1], v[3 * k + 2]);
    a[10] = NEG ? fminf(v[30], v[31]) : fmaxf(v[30], v[31]);
    float b0 = NEG ? min3f(a[0], a[1], a[2]) : max3f(a[0], a[1], a[2]);
    float b1 = NEG ? min3f(a[3], a[4], a[5]) : max3f(a[3], a[4], a[5]);
    float b2 = NEG ? min3f(a[6], a[7], a[8]) : max3f(a[6], a[7], a[8]);
    float b3 = NEG ? min3f(a[9], a[10], st.ext) : max3f(a[9], a[10], st.ext);
    const float e2 = NEG ? fminf(fminf(b0, b1), fminf(b2, b3)) : fmaxf(fmaxf(b0, b1), fmaxf(b2, b3));
    const float mt2 = e2 * sc;
    // move the reference to the running maximum, rescaling the sum (2^(-inf) = 0
    // clears the empty start)
    const float f = ex2_approx(st.ref - mt2);
    st.l = (mt2 == st.ref) ? st.l : st.l * f;
    st.ref = mt2;
    st.ext = e2;
    const float2 sc2 = f2(sc), nm2 = f2(-mt2);
    float2 s0 = f2(0.f), s1 = f2(0.f);
#pragma unroll
    for (int k = 0; k < 32; k += 2) {
        // exponent arguments t - t_max, two columns per instruction
        float2 x = __ffma2_rn(make_float2(v[k], v[k + 1]), sc2, nm2);
        float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
        if (MASKED) {
            if (k >= valid) e.x = 0.f;
            if (k + 1 >= valid) e.y = 0.f;
        }
        if ((k >> 1) & 1) s1 = __fadd2_rn(s1, e);
        else s0 = __fadd2_rn(s0, e);
    }
    const float2 s = __fadd2_rn(s0, s1);
    st.l += s.x + s.y;
}

// Orders later uses of the registers after the preceding tcgen05.wait::ld.
__device__ __forceinline__ void regs_after_wait(uint32_t (&r)[32]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// The 128 columns of one half tile, one tensor-memory lane (query row) per thread.
__device__ __forceinline__ void load_half(uint32_t taddr, uint32_t (&r)[4][32]) {
    tmem_ld_32x32b_x32(taddr, r[0]);
    tmem_ld_32x32b_x32(taddr + 32u, r[1]);
    tmem_ld_32x32b_x32(taddr + 64u, r[2]);
    tmem_ld_32x32b_x32(taddr + 96u, r[3]);
    tmem_ld_wait_regs(r[0]);
    regs_after_wait(r[1]);
    regs_after_wait(r[2]);
    regs_after_wait(r[3]);
}

// sum over the 128 columns of 2^(score * sc - ref), in four packed partial sums
__device__ __forceinline__ float2 sum_exp2_128(const uint32_t (&r)[4][32], float sc, float ref) {
    const float2 sc2 = f2(sc), nm2 = f2(-ref);
    float2 s[4] = {f2(0.f), f2(0.f), f2(0.f), f2(0.f)};
#pragma unroll
    for (int k = 0; k < 128; k += 2) {
        const float2 x = __ffma2_rn(make_float2(__uint_as_float(r[k >> 5][k & 31]),
                                                __uint_as_float(r[k >> 5][(k + 1) & 31])), sc2, nm2);
        const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
        s[(k >> 1) & 3] = __fadd2_rn(s[(k >> 1) & 3], e);
    }
    return __fadd2_rn(__fadd2_rn(s[0], s[1]), __fadd2_rn(s[2], s[3]));
}

// Folds a full half tile (128 real columns) into the state: one extreme over the
// 128 scores, the reference moved to the new running maximum (the sum rescaled),
// then 128 exponentials.
template <bool NEG>
__device__ __forceinline__ void fold_full_half(const uint32_t (&r)[4][32], float sc, RowState& st) {
    float a[43];
#pragma unroll
    for (int i = 0; i < 42; ++i) {
        const int k = 3 * i;
        const float x0 = __uint_as_float(r[k >> 5][k & 31]);
        const float x1 = __uint_as_float(r[(k + 1) >> 5][(k + 1) & 31]);
        const float x2 = __uint_as_float(r[(k + 2) >> 5][(k + 2) & 31]);
        a[i] = NEG ? min3f(x0, x1, x2) : max3f(x0, x1, x2);
    }
    a[42] = NEG ? min3f(__uint_as_float(r[3][30]), __uint_as_float(r[3][31]), st.ext)
                : max3f(__uint_as_float(r[3][30]), __uint_as_float(r[3][31]), st.ext);
    float b[15];
#pragma unroll
    for (int i = 0; i < 14; ++i) b[i] = NEG ? min3f(a[3 * i], a[3 * i + 1], a[3 * i + 2])
                                           : max3f(a[3 * i], a[3 * i + 1], a[3 * i + 2]);
    b[14] = a[42];
    float c[5];
#pragma unroll
    for (int i = 0; i < 5; ++i) c[i] = NEG ? min3f(b[3 * i], b[3 * i + 1], b[3 * i + 2])
                                          : max3f(b[3 * i], b[3 * i + 1], b[3 * i + 2]);
    const float e2 = NEG ? fminf(min3f(c[0], c[1], c[2]), fminf(c[3], c[4]))
                         : fmaxf(max3f(c[0], c[1], c[2]), fmaxf(c[3], c[4]));
    const float mt = e2 * sc;
    const float f = ex2_approx(st.ref - mt);  // 2^(-inf) = 0 on the row's first columns
    st.l = (mt == st.ref) ? st.l : st.l * f;
    st.ref = mt;
    st.ext = e2;
    const float2 s = sum_exp2_128(r, sc, mt);
    st.l += s.x + s.y;
}

// Folds a partial half tile (the ragged last tile: 0 < valid < 128 real columns,
// warp-uniform) chunk by chunk, masking the columns past the last key.
template <bool NEG>
__device__ __forceinline__ void fold_partial_half(uint32_t taddr, int valid, float sc, RowState& st) {
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        const int vc = valid - 32 * c;
        if (vc <= 0) break;
        uint32_t r[32];
        tmem_ld_32x32b_x32(taddr + 32u * c, r);
        tmem_ld_wait_regs(r);
        if (vc >= 32) fold_chunk<NEG, false>(r, 32, sc, st);
        else fold_chunk<NEG, true>(r, vc, sc, st);
    }
}

template <int KQ>
__global__ void __launch_bounds__(SM_THREADS, 1)
score_softmax_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const SoftmaxParams p) {
    using Cfg = SmCfg<KQ>;
    constexpr int S = Cfg::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + Cfg::OFF_Q;
    const uint32_t sK = sbase + Cfg::OFF_K;
    const uint32_t bar0 = sbase + Cfg::OFF_BAR;
    auto kfull = [&](int s) { return bar0 + 8u * s; };
    auto kempty = [&](int s) { return bar0 + 8u * (S + s); };
    auto qfull = [&](int b) { return bar0 + 8u * (2 * S + b); };
    auto qempty = [&](int b) { return bar0 + 8u * (2 * S + 2 + b); };
    auto tfull = [&](int b) { return bar0 + 8u * (2 * S + 4 + b); };
    auto tempty = [&](int b) { return bar0 + 8u * (2 * S + 6 + b); };
    auto mfull = [&](int b) { return bar0 + 8u * (2 * S + 8 + b); };
    auto mempty = [&](int b) { return bar0 + 8u * (2 * S + 10 + b); };
    float2* merge = reinterpret_cast<float2*>(smem + Cfg::OFF_MERGE);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_TMEM_SLOT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_ABORT);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(kfull(s), 1);
            mbar_init(kempty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(qfull(b), 1);
            mbar_init(qempty(b), 1);
            mbar_init(tfull(b), 1);
            mbar_init(tempty(b), SM_EPI_WARPS / 2);
            mbar_init(mfull(b), 4 * 32);
            mbar_init(mempty(b), 4 * 32);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmQ);
        prefetch_tensormap(&tmK);
    }
    if (warp == 1) tmem_alloc<1>(smem_u32(tmem_slot), SM_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int64_t G = gridDim.x;
    const int32_t ntiles = p.ntiles;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t ui = 0;
            bool ok = true;
            for (int64_t u = blockIdx.x; ok && u < p.num_units; u += G, ++ui) {
                const int32_t b = static_cast<int32_t>(u / p.mblocks);
                const int32_t mb = static_cast<int32_t>(u % p.mblocks);
                const int qb = static_cast<int>(ui & 1u);
                if (!sm_wait(qempty(qb), ((ui >> 1) & 1u) ^ 1u, p.err, p.timeout_ns, abort_flag, 0x20)) break;
                mbar_arrive_expect_tx(qfull(qb), Cfg::Q_BYTES);
                for (int kb = 0; kb < KQ; ++kb)
                    tma_load_3d(sQ + qb * Cfg::Q_BYTES + kb * SM_Q_BOX, &tmQ, qfull(qb), kb * SM_BK, mb * SM_BM,
                                b * p.zq);
                for (int32_t t = 0; ok && t < ntiles; ++t) {
                    for (int kb = 0; kb < KQ; ++kb) {
                        if (!sm_wait(kempty(stage), phase ^ 1u, p.err, p.timeout_ns, abort_flag, 0x21)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(kfull(stage), SM_K_BOX);
                        tma_load_3d(sK + stage * SM_K_BOX, &tmK, kfull(stage), kb * SM_BK, t * SM_BN, b * p.zk);
                        if (++stage == S) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32(SM_BM, SM_BN);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t abuf = 0, aphase = 0;
            uint32_t ui = 0;
            bool ok = true;
            for (int64_t u = blockIdx.x; ok && u < p.num_units; u += G, ++ui) {
                const int qb = static_cast<int>(ui & 1u);
                if (!sm_wait(qfull(qb), (ui >> 1) & 1u, p.err, p.timeout_ns, abort_flag, 0x22)) break;
                tc_fence_after();
                for (int32_t t = 0; ok && t < ntiles; ++t) {
                    if (!sm_wait(tempty(static_cast<int>(abuf)), aphase ^ 1u, p.err, p.timeout_ns, abort_flag, 0x23)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + abuf * SM_BN;
                    for (int kb = 0; kb < KQ; ++kb) {
                        if (!sm_wait(kfull(stage), phase, p.err, p.timeout_ns, abort_flag, 0x24)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t qa = sQ + qb * Cfg::Q_BYTES + kb * SM_Q_BOX;
                        const uint32_t ka = sK + stage * SM_K_BOX;
#pragma unroll
                        for (int k = 0; k < SM_BK / 16; ++k)
                            mma_f16<1>(d_tmem, smem_desc_sw128(qa + 32u * k), smem_desc_sw128(ka + 32u * k), idesc,
                                       (kb | k) != 0 ? 1u : 0u);
                        mma_commit(kempty(stage));
                        if (++stage == S) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    mma_commit(tfull(static_cast<int>(abuf)));
                    abuf ^= 1u;
                    if (abuf == 0) aphase ^= 1u;
                }
                if (ok) mma_commit(qempty(qb));
            }
        }
    } else {
        // ------------------------------------------------------------ softmax warps
        const int q = warp & 3;             // tensor-memory lane quarter
        const int h = (warp - 2) >> 2;      // this warp folds the S tiles held in buffer h
        const bool neg = p.sc < 0.f;
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(h * SM_BN);
        uint32_t tphase = 0;                // phase of tfull(h)
        uint64_t g = 0;                     // S tiles of this CTA before the current unit
        uint32_t ui = 0;
        bool ok = true;
        for (int64_t u = blockIdx.x; ok && u < p.num_units; u += G, ++ui) {
            const int32_t b = static_cast<int32_t>(u / p.mblocks);
            const int32_t mb = static_cast<int32_t>(u % p.mblocks);
            RowState st;
            st.ext = neg ? __int_as_float(0x7f800000) : __int_as_float(0xff800000);
            st.ref = __int_as_float(0xff800000);
            st.l = 0.f;
            // tiles alternate between the two buffers across the CTA's whole tile sequence;
            // the two warps of a lane quarter take every other tile, so that one folds
            // while the other loads
            for (int32_t t = static_cast<int32_t>((g & 1u) ^ static_cast<uint32_t>(h)); t < ntiles; t += 2) {
                uint32_t got = 0;
                if (lane == 0)
                    got = sm_wait(tfull(h), tphase, p.err, p.timeout_ns, abort_flag, 0x25) ? 1u : 0u;
                got = __shfl_sync(0xffffffffu, got, 0);
                if (!got) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                auto release = [&]() {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(tempty(h));
                };
                const int valid = p.N - t * SM_BN;  // real columns in this tile
                if (valid >= SM_BN) {
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t r[4][32];
                        load_half(tbase + static_cast<uint32_t>(hh * (SM_BN / 2)), r);
                        if (hh == 1) release();  // the MMA may refill the buffer during the fold
                        if (neg) fold_full_half<true>(r, p.sc, st);
                        else fold_full_half<false>(r, p.sc, st);
                    }
                } else {
                    const int v0 = valid < SM_BN / 2 ? valid : SM_BN / 2;
                    if (neg) {
                        fold_partial_half<true>(tbase, v0, p.sc, st);
                        fold_partial_half<true>(tbase + SM_BN / 2, valid - v0, p.sc, st);
                    } else {
                        fold_partial_half<false>(tbase, v0, p.sc, st);
                        fold_partial_half<false>(tbase + SM_BN / 2, valid - v0, p.sc, st);
                    }
                    release();
                }
                tphase ^= 1u;
            }
            g += static_cast<uint64_t>(ntiles);
            if (!ok) break;
            // merge the two partial states of each row
            const int mbuf = static_cast<int>(ui & 1u);
            const uint32_t mpar = (ui >> 1) & 1u;
            const int row_local = 32 * q + lane;
            if (h == 1) {
                if (!sm_wait(mempty(mbuf), mpar ^ 1u, p.err, p.timeout_ns, abort_flag, 0x26)) break;
                merge[mbuf * SM_BM + row_local] = make_float2(st.ext, st.l);
                mbar_arrive(mfull(mbuf));
            } else {
                if (!sm_wait(mfull(mbuf), mpar, p.err, p.timeout_ns, abort_flag, 0x27)) break;
                const float2 o = merge[mbuf * SM_BM + row_local];
                mbar_arrive(mempty(mbuf));
                const float e = neg ? fminf(st.ext, o.x) : fmaxf(st.ext, o.x);
                const float mt = e * p.sc;
                // a half with no real column has l == 0 and contributes nothing
                const float l0 = st.l > 0.f ? st.l * ex2_approx(st.ext * p.sc - mt) : 0.f;
                const float l1 = o.y > 0.f ? o.y * ex2_approx(o.x * p.sc - mt) : 0.f;
                const int64_t row = static_cast<int64_t>(mb) * SM_BM + row_local;
                if (row < p.M) {
                    const int64_t r = static_cast<int64_t>(b) * p.M + row;
                    p.row_max[r] = p.alpha * e;
                    p.row_sum[r] = l0 + l1;
                }
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    __syncwarp();
    if (*abort_flag) sm_spin_ns(2000000ull);  // let in-flight TMA loads and MMAs land
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc<1>(tmem_base, SM_TMEM_COLS);
}

template <int KQ>
cudaError_t launch_kq(const CUtensorMap& tmQ, const CUtensorMap& tmK, const SoftmaxParams& p, int sms,
                      cudaStream_t stream) {
    using Cfg = SmCfg<KQ>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        e = cudaFuncSetAttribute(score_softmax_kernel<KQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(Cfg::SMEM));
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const int64_t grid = p.num_units < sms ? p.num_units : sms;
    score_softmax_kernel<KQ><<<static_cast<unsigned>(grid), SM_THREADS, Cfg::SMEM, stream>>>(tmQ, tmK, p);
    return cudaGetLastError();
}

__global__ void fill_stats_kernel(float* m, float* l, int64_t n, float mv, float lv) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        m[i] = mv;
        l[i] = lv;
    }
}

}  // namespace

cudaError_t launch_score_softmax(const CUtensorMap& tmQ, const CUtensorMap& tmK, const SoftmaxParams& p, int kq,
                                 int sms, cudaStream_t stream) {
    switch (kq) {
        case 1: return launch_kq<1>(tmQ, tmK, p, sms, stream);
        case 2: return launch_kq<2>(tmQ, tmK, p, sms, stream);
        case 4: return launch_kq<4>(tmQ, tmK, p, sms, stream);
    }
    return cudaErrorInvalidValue;
}

int softmax_tile_n() { return SM_BN; }

cudaError_t launch_fill_stats(float* m, float* l, int64_t n, float mv, float lv, int sms, cudaStream_t stream) {
    int64_t blocks = (n + 255) / 256;
    if (blocks > 4 * static_cast<int64_t>(sms)) blocks = 4 * static_cast<int64_t>(sms);
    if (blocks < 1) blocks = 1;
    fill_stats_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(m, l, n, mv, lv);
    return cudaGetLastError();
}

}  // namespace gtn
