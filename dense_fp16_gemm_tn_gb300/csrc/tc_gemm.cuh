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
//               CTA pair, N=BN, or two N=256 MMAs side by side for 512-column
//               pair tiles, K=16, fp16 x fp16 -> fp32) straight from the
//               shared-memory descriptors into a tensor-memory accumulator.
//               There is no shared->register step: the tensor core reads its
//               operands from shared memory itself.
//   warps 2-5   epilogue: tcgen05.ld tensor memory -> registers, alpha/beta in
//               fp32, one round-to-nearest-even to fp16, then TMA stores; for a
//               D whose rows TMA cannot address, each thread writes its row
//               through the aligned 16-byte words that cover it (rowio.h); a
//               predicated element-wise epilogue remains for forced use and
//               fp16 accumulators.
//
// Two accumulators in tensor memory let the epilogue of one tile overlap the
// main loop of the next.  A 512-column tile fills tensor memory with one
// accumulator: the epilogue hands its first half back as soon as it has read
// it, and the MMA starts the next tile's first k-block on that half while the
// second half is still being read.  The grid is persistent: CTA (or CTA pair) i takes
// work units i, i+G, i+2G, ... in an order grouped along M so that tiles
// running at the same time share A and B rows in L2.  A work unit is one
// output tile of one batch entry and, for split-K, one slice of K.
//
// Tails: TMA loads zero-fill rows/columns past M, N and K, and TMA stores
// clip at the tensor bounds, so ragged shapes need no masks on the fast path;
// the row-word epilogue writes only a row's real elements, the predicated ones
// mask element by element.
//
// Stream-K: when the tiles do not divide evenly over the CTA groups, the last
// partial wave is not run tile by tile; its k-block iterations are spread
// evenly over all groups instead.  A group that computes part of a tile writes
// its fp32 partial accumulator to scratch and counts itself in (per epilogue
// warp, i.e. per 32 rows); the last group to arrive for those rows sums all
// partials in group order (deterministic) and runs the epilogue.  No group, and
// no warp, ever waits for another.
//
// Every mbarrier wait is bounded: past `timeout_ns` the waiting thread records
// an error word, raises a CTA-wide abort flag and returns; the kernel then lets
// in-flight copies and MMAs drain, frees its tensor memory and exits normally.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>
#include <type_traits>

#include "kparams.h"
#include "ptx.cuh"
#include "rowio.h"

namespace gtn {

template <int BN, int PAIR, int STAGES, int EPIX>
struct TileCfg {
    static constexpr int EPI = epi_mode(EPIX);   // epilogue mode
    static constexpr bool RL = epi_rl(EPIX);     // row-loader warps for operands TMA cannot address
    static constexpr bool CK = epi_ck(EPIX);     // K halves on the two CTAs of a cluster (swapped tiles)
    static constexpr bool H2 = epi_h2(EPIX);     // one epilogue warpgroup per part of a wide accumulator
    static constexpr bool SQ = epi_sq(EPIX);     // four TMA-store staging buffers per epilogue warp
    static constexpr int NBUF = SQ ? 4 : 2;      // staging buffers of 32 x 64 halves per epilogue warp
    static constexpr int CLUSTER = (PAIR == 2 || CK) ? 2 : 1;
    static constexpr int BM = 128;               // accumulator rows per CTA (tensor-memory lanes)
    static constexpr int BK = 64;                // halves per 128-byte swizzled row
    static constexpr int BN_LOCAL = BN / PAIR;   // B rows each CTA of a pair loads
    // A wide pair tile (BN = 432 or 512) is two MMAs per 16-wide K step: N = 256 for the
    // tile's first 256 columns and N = BN - 256 for the rest; each CTA loads one 128-row B
    // box per MMA (of the second box's 128 rows, a 432-column tile uses the first 88).
    static constexpr bool WIDE = BN > 256;
    static constexpr int MMA_N = WIDE ? 256 : BN;      // N of the first MMA
    static constexpr int MMA_N1 = WIDE ? BN - 256 : BN;  // N of the second
    static constexpr int N_MMAS = WIDE ? 2 : 1;
    static constexpr int B_BOX_ROWS = MMA_N / PAIR;
    static constexpr int B_BOX_BYTES = B_BOX_ROWS * BK * 2;
    // Accumulators in tensor memory (512 columns): two of BN <= 256 columns, so that the
    // epilogue of one tile overlaps the main loop of the next; one of a wide tile's BN
    // columns, whose two parts (the two MMAs' columns) are released separately.
    static constexpr int ACC_BUFS = (2 * BN <= 512) ? 2 : 1;
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = N_MMAS * B_BOX_BYTES;
    // Whole 64-column chunks of the TMA epilogue, and the columns of a wide tile's partial
    // last chunk (48 for a 432-column tile, written from registers by 16-byte stores).
    static constexpr int FULL_CHUNKS = BN / 64;
    static constexpr int TAIL_COLS = WIDE ? BN % 64 : 0;
    static constexpr uint32_t STAGE_TX = uint32_t(A_BYTES + B_BYTES) * PAIR;
    static constexpr int EPI_WARPS = H2 ? 8 : 4;
    static constexpr int RL_WARPS = RL ? 8 : 0;  // one operand row per loader thread and k-block
    // Warp roles: 0 TMA producer, 1 MMA issuer, then the epilogue warps, then the loader warps.
    // With the row loader the block is four warpgroups whose register shares differ
    // (setmaxnreg): warps 0-3 (producer, MMA, two idle) give registers up, the epilogue
    // warpgroup (4-7) and the two loader warpgroups (8-15) take them.  With two epilogue
    // warpgroups (H2) it is three: warps 0-3 give up, the epilogue warpgroups 4-7 (first
    // part of the accumulator) and 8-11 (second part) take.
    static constexpr bool SETMAXNREG = RL || H2;
    static constexpr int EPI_W0 = SETMAXNREG ? 4 : 2;
    static constexpr int RL_W0 = EPI_W0 + EPI_WARPS;
    static constexpr int THREADS = 32 * RL_W0 + 32 * RL_WARPS;
    // per thread, after setmaxnreg
    static constexpr int REGS_CTRL = H2 ? 104 : 48, REGS_EPI = H2 ? 200 : 176, REGS_RL = 144;
    // epilogue warps arriving on each part's tensor-memory barrier (per CTA)
    static constexpr int TEMPTY_WARPS = H2 ? EPI_WARPS / 2 : EPI_WARPS;
    // Registers per thread: all of the 64K register file over the block's warps, in steps of 8.
    static constexpr int MAX_REGS = ((65536 / THREADS) / 8 * 8) > 255 ? 255 : ((65536 / THREADS) / 8 * 8);
    static constexpr int TMEM_COLS = (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64 : (2 * BN <= 128) ? 128
                                   : (2 * BN <= 256) ? 256 : 512;
    static constexpr int EPI_WARP_BYTES =
        H2 ? 32 * 128  // one staging buffer per warp (eight warps)
        : (epi_base(EPI) == EPI_TMA || EPI == EPI_TMA_C || EPI == EPI_TMA_CG) ? NBUF * 32 * 128
        : (EPI == EPI_PARTIAL) ? 2 * 32 * 128  // TMA staging (or the padded transpose, 32 x 33 x 4)
        : (epi_base(EPI) == EPI_GENERIC) ? 32 * 33 * 4 : 0;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_EPI = OFF_B + STAGES * B_BYTES;
    // cluster K split: the second CTA's partial accumulator, [128 rows][BN] fp32, lands here
    static constexpr int OFF_X = OFF_EPI + ((EPI_WARPS * EPI_WARP_BYTES + 1023) / 1024) * 1024;
    static constexpr int X_BYTES = CK ? 128 * BN * 4 : 0;
    static constexpr int OFF_BAR = OFF_X + X_BYTES;
    static constexpr int NUM_BARS = 2 * STAGES + 4 + (EPI == EPI_TMA_C ? 2 * EPI_WARPS : 0)  // + C-load barriers
                                    + (CK ? 2 : 0);                                           // + partial full / empty
    static constexpr int OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_ABORT = OFF_TMEM_SLOT + 4;
    static constexpr int SMEM_BYTES = OFF_ABORT + 4 + 1024;  // + slack to align the base to 1024

    static_assert(BN % 16 == 0 && BN >= 16 && (BN <= 256 || ((BN == 512 || BN == 432) && PAIR == 2)),
                  "tcgen05 needs N in [16,256], N%16==0; 432 and 512 columns are two MMAs of a CTA pair");
    static_assert(BN <= 256 || EPI == EPI_TMA || EPI == EPI_TMA_C || EPI == EPI_TMA_CG,
                  "512-column tiles have the TMA epilogues only");
    static_assert(BN != 432 || EPI == EPI_TMA, "432-column tiles: D = alpha * acc by TMA stores only");
    static_assert(MMA_N1 % 16 == 0 && MMA_N1 <= 256 && (MMA_N1 / PAIR) % 8 == 0,
                  "second MMA: N%16==0, whole 8-row swizzle atoms of B per CTA");
    static_assert(B_BYTES % 1024 == 0 && A_BYTES % 1024 == 0 && B_BOX_BYTES % 1024 == 0,
                  "tiles must stay 1024-byte aligned");
    static_assert((epi_base(EPI) != EPI_TMA && EPI != EPI_TMA_C && EPI != EPI_TMA_CG && EPI != EPI_VEC) ||
                      BN % 64 == 0 || (BN == 432 && EPI == EPI_TMA),
                  "the TMA and row-word epilogues work in 64-column chunks");
    static_assert(!WIDE || MMA_N % 64 == 0, "a wide tile's first part ends on a 64-column chunk");
    static_assert(TAIL_COLS == 0 || TAIL_COLS == 48, "a partial last chunk is 32 + 16 tensor-memory columns");
    static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB of shared memory per CTA");
    static_assert(PAIR == 1 || PAIR == 2, "CTA pair or single CTA");
    static_assert(!RL || (BM + BN_LOCAL <= 32 * RL_WARPS && BN_LOCAL % 32 == 0 && N_MMAS == 1),
                  "row loader: one row of A or B per loader thread, whole warps per operand");
    static_assert(!RL || EPI == EPI_TMA || EPI == EPI_TMA_C || EPI == EPI_TMA_CG || EPI == EPI_VEC,
                  "row loader: unswapped whole-tile epilogues only");
    static_assert(!CK || (PAIR == 1 && EPI == EPI_SWAP && !RL), "cluster K split: swapped single-CTA tiles");
    static_assert(!RL || (THREADS == 512 && MAX_REGS == 128 &&
                          REGS_CTRL + REGS_EPI + 2 * REGS_RL == 4 * MAX_REGS),
                  "the warpgroups' register shares must add up to the block's launch allocation");
    static_assert(!H2 || (WIDE && EPI == EPI_TMA && PAIR == 2 && !RL && !CK), "two epilogue warpgroups: wide TMA tiles");
    static_assert(!SQ || (EPI == EPI_TMA && !WIDE && !RL && !CK && !H2), "deep store queue: D = alpha*acc by TMA stores");
    // (with 104 registers the producer and MMA code of the 512-column tile compiles without
    // spills, and 200 hold an epilogue warp's 128 packed words of its part plus a load)
    static_assert(!H2 || (THREADS == 384 && MAX_REGS == 168 && REGS_CTRL + 2 * REGS_EPI == 3 * MAX_REGS),
                  "the warpgroups' register shares must add up to the block's launch allocation");
};

// One piece of work for a CTA (pair): k-blocks [kb0, kb1) of one output tile.
struct Seg {
    int32_t b, tm, tn, kb0, kb1, split;
    int32_t rev;      // 1: k-blocks are loaded from kb1 - 1 down to kb0
    int32_t sk_tile;  // index among the stream-K tiles, or -1 when this segment finishes its tile alone
    int32_t sk_j;     // this group's rank among the tile's contributors
    int32_t sk_n;     // number of contributors to the tile
};

// Iterates the segments of CTA group `g` of `G`: its contiguous range of
// stream-K iterations, then its data-parallel units g, g+G, ...  Every role of
// the CTA walks the same sequence.
struct SegIter {
    int64_t g, G;
    int64_t dp_next;
    int32_t dp_wave;  // wave of the next data-parallel unit (dp_next / G)
    int64_t sk_i, sk_end;
    int64_t sk_mid;   // >= 0: run [sk_mid, sk_end) before [sk_i, sk_mid) (see seg_begin)
};

__device__ __forceinline__ void tile_coords(const KParams& p, int64_t t, Seg& s) {
    const int64_t per_batch = static_cast<int64_t>(p.tiles_m) * p.tiles_n;
    s.b = static_cast<int32_t>(t / per_batch);
    const int64_t r = t % per_batch;
    // Grouped rasterisation: group_m tile rows are walked column by column, so
    // the tiles in flight at one time share A rows and B rows in L2.
    const int64_t span = static_cast<int64_t>(p.group_m) * p.tiles_n;
    const int32_t first = static_cast<int32_t>(r / span) * p.group_m;
    const int32_t gm = min(p.group_m, p.tiles_m - first);
    const int64_t rr = r % span;
    s.tm = first + static_cast<int32_t>(rr % gm);
    s.tn = static_cast<int32_t>(rr / gm);
}

__device__ __forceinline__ int64_t sk_start(const KParams& p, int64_t g, int64_t G) { return (g * p.sk_iters) / G; }

// Group that owns stream-K iteration i: the largest g with sk_start(g) <= i.
__device__ __forceinline__ int64_t sk_owner(const KParams& p, int64_t i, int64_t G) {
    return ((i + 1) * G - 1) / p.sk_iters;
}

template <bool SK>
__device__ __forceinline__ SegIter seg_begin(const KParams& p, int64_t g, int64_t G) {
    SegIter it;
    it.g = g;
    it.G = G;
    it.dp_next = g;
    it.dp_wave = 0;
    it.sk_i = (SK && p.sk_iters > 0) ? sk_start(p, g, G) : 0;
    it.sk_end = (SK && p.sk_iters > 0) ? sk_start(p, g + 1, G) : 0;
    // A range that ends a tile and starts the next one is two segments on the two
    // accumulators.  The first segment's epilogue parks its partial sums while the second
    // runs, and the first whole tile after them needs the first accumulator back: when
    // the first piece is the longer one, its parking outlasts the second piece's main
    // loop and the MMA waits (2-4 us on 4096^3).  The shorter piece goes first instead.
    it.sk_mid = -1;
    if (SK && it.sk_i < it.sk_end) {
        const int64_t kb = p.kb_total;
        const int64_t b = (it.sk_i / kb + 1) * kb;  // first tile boundary after sk_i
        if (b < it.sk_end && it.sk_end - b <= kb && it.sk_end - b < b - it.sk_i) it.sk_mid = b;
    }
    return it;
}

template <bool SK>
__device__ __forceinline__ bool seg_next(const KParams& p, SegIter& it, Seg& s) {
    // Stream-K iterations come first, so the tile fixups they lead to overlap the
    // data-parallel work that follows instead of trailing the kernel.
    if (SK && it.sk_i < it.sk_end) {
        const int64_t kb = p.kb_total;
        const int64_t lo = it.sk_mid >= 0 ? it.sk_mid : it.sk_i;  // start of this segment's iterations
        const int64_t tsk = lo / kb;
        const int64_t k0 = lo - tsk * kb;
        const int64_t k1 = min(kb, k0 + (it.sk_end - lo));
        tile_coords(p, p.num_units + tsk, s);
        s.split = 0;
        s.rev = 0;
        s.kb0 = static_cast<int32_t>(k0);
        s.kb1 = static_cast<int32_t>(k1);
        if (k0 == 0 && k1 == kb) {
            s.sk_tile = -1;
            s.sk_j = 0;
            s.sk_n = 1;
        } else {
            const int64_t first = sk_owner(p, tsk * kb, it.G);
            s.sk_tile = static_cast<int32_t>(tsk);
            s.sk_j = static_cast<int32_t>(it.g - first);
            s.sk_n = static_cast<int32_t>(sk_owner(p, (tsk + 1) * kb - 1, it.G) - first + 1);
        }
        if (it.sk_mid >= 0) {  // the later piece ran first; the earlier one follows
            it.sk_end = it.sk_mid;
            it.sk_mid = -1;
        } else {
            it.sk_i += k1 - k0;
        }
        return true;
    }
    if (it.dp_next < p.num_units) {
        const int64_t u = it.dp_next;
        it.dp_next += it.G;
        // Serpentine K order: every other wave walks K backwards, so that it starts on the
        // k-blocks the wave before it loaded last, which are still in L2 where the two
        // waves share operand rows.
        s.rev = p.serp & it.dp_wave;
        it.dp_wave ^= 1;
        if (p.splits == 1) {  // whole tiles: no K-slice arithmetic
            s.split = 0;
            tile_coords(p, u, s);
            s.kb0 = 0;
            s.kb1 = p.kb_total;
        } else {
            s.split = static_cast<int32_t>(u % p.splits);
            tile_coords(p, u / p.splits, s);
            s.kb0 = static_cast<int32_t>((static_cast<int64_t>(s.split) * p.kb_total) / p.splits);
            s.kb1 = static_cast<int32_t>((static_cast<int64_t>(s.split + 1) * p.kb_total) / p.splits);
        }
        s.sk_tile = -1;
        s.sk_j = 0;
        s.sk_n = 1;
        return true;
    }
    return false;
}

// Slow path of a bounded wait.  Returns false (and raises the abort flag) when
// the wait gave up; records the first failure in the device error word.
// Bound on a waiter's suspension inside mbarrier.try_wait (see mbar_try_wait_ns).
constexpr uint32_t kWaitSuspendNs = 32;

static __device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, uint32_t* err, uint64_t timeout_ns,
                                              volatile int* abort_flag, uint32_t who) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait_ns(bar, parity, kWaitSuspendNs)) return true;
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

// The same slow path inlined: kernels that change register shares per warpgroup
// (setmaxnreg) make no calls, since a callee is compiled for one register count.
static __device__ __forceinline__ bool wait_slow_inl(uint32_t bar, uint32_t parity, uint32_t* err,
                                                     uint64_t timeout_ns, volatile int* abort_flag, uint32_t who) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait_ns(bar, parity, kWaitSuspendNs)) return true;
        if ((i & 15u) == 0) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > timeout_ns) {
                atomicCAS(err, 0u, 0x500u | who);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

template <bool INL = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, uint32_t* err, uint64_t timeout_ns,
                                             volatile int* abort_flag, uint32_t who) {
    if (mbar_try_wait_ns(bar, parity, kWaitSuspendNs)) return true;
    if constexpr (INL) return wait_slow_inl(bar, parity, err, timeout_ns, abort_flag, who);
    else return wait_slow(bar, parity, err, timeout_ns, abort_flag, who);
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

// SK: compiled with the stream-K phase (partial slots, arrival counters,
// fixups); without it the kernel is purely data-parallel.
template <int BN, int PAIR, int STAGES, int EPIX, bool SK>
__global__ void __launch_bounds__(TileCfg<BN, PAIR, STAGES, EPIX>::THREADS, 1)
gemm_tn_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                  const KParams p) {
    using Cfg = TileCfg<BN, PAIR, STAGES, EPIX>;
    constexpr int EPI = Cfg::EPI;
    constexpr int EB = epi_base(EPI);       // epilogue mode without the accumulator precision
    constexpr bool ACC16 = epi_acc16(EPI);  // fp16 accumulator in tensor memory
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
    // C tile loads of the TMA epilogue: buffer b of epilogue warp ew.
    auto cload_bar = [&](int ew, int b) { return bar0 + 8u * (2 * STAGES + 4 + 2 * ew + b); };
    // cluster K split: partial buffer full (in CTA 0) / empty (in CTA 1)
    const uint32_t xfull_bar = bar0 + 8u * (Cfg::NUM_BARS - 2), xempty_bar = bar0 + 8u * (Cfg::NUM_BARS - 1);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_TMEM_SLOT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_ABORT);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = (PAIR == 2) ? cluster_cta_rank() : 0u;
    const uint32_t krank = Cfg::CK ? cluster_cta_rank() : 0u;  // K half of a cluster K split
    // A kernel launched as this one's programmatic dependent (the split-K reduction) may
    // be scheduled now; it waits for this grid's completion before it reads anything.
    griddep_launch_dependents();
    const int64_t group = blockIdx.x / Cfg::CLUSTER;
    const int64_t ngroups = gridDim.x / Cfg::CLUSTER;
    // Cluster K split: CTA krank of the cluster takes half krank of every tile's k-blocks.
    auto ck_half = [&](Seg& w) {
        if constexpr (Cfg::CK) {
            const int32_t mid = w.kb0 + (w.kb1 - w.kb0) / 2;
            if (krank == 0) w.kb1 = mid;
            else w.kb0 = mid;
        }
    };

    if (threadIdx.x == 0) {
        // A stage is full once the leader's producer has armed it (and TMA has brought its
        // bytes) and, with the row loader, every loader warp of both CTAs that writes an
        // operand has arrived.
        uint32_t full_count = 1;
        if constexpr (Cfg::RL)
            full_count += static_cast<uint32_t>(((p.rl_on[0] ? Cfg::BM : 0) + (p.rl_on[1] ? Cfg::BN_LOCAL : 0)) / 32 * PAIR);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), full_count);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), Cfg::TEMPTY_WARPS * PAIR);
        }
        if constexpr (EPI == EPI_TMA_C)
            for (int e = 0; e < 2 * Cfg::EPI_WARPS; ++e) mbar_init(cload_bar(e / 2, e % 2), 1);
        if constexpr (Cfg::CK) {
            mbar_init(xfull_bar, Cfg::EPI_WARPS);
            mbar_init(xempty_bar, Cfg::EPI_WARPS);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        if (!(Cfg::RL && p.rl_on[0])) prefetch_tensormap(&tmA);
        if (!(Cfg::RL && p.rl_on[1])) prefetch_tensormap(&tmB);
        if constexpr (EB == EPI_TMA || EPI == EPI_TMA_C || EPI == EPI_TMA_CG || EPI == EPI_PARTIAL)
            prefetch_tensormap(&tmD);
        if constexpr (EPI == EPI_TMA_C) prefetch_tensormap(&tmC);
    }
    if (warp == 1) tmem_alloc<PAIR>(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tc_fence_before();
    if constexpr (Cfg::CLUSTER == 2) cluster_sync(); else __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // Each role's register share is set at the top of its branch (row-loader variants), so
    // that the compiler allocates every role's code within its own share.
    if (warp < Cfg::EPI_W0) {
    if constexpr (Cfg::SETMAXNREG) setmaxnreg_dec<Cfg::REGS_CTRL>();
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            if (p.pdl) griddep_wait();  // the repacked operands are complete and visible
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            bool first = true;
            SegIter it = seg_begin<SK>(p, group, ngroups);
            Seg w;
            while (ok && seg_next<SK>(p, it, w)) {
                ck_half(w);
                const int32_t rowA = w.tm * (Cfg::BM * PAIR) + Cfg::BM * static_cast<int32_t>(rank);
                // B box nb holds the columns of MMA nb (tile columns nb*MMA_N + [0, N of MMA nb)),
                // split between the pair: this CTA's share starts (N of MMA nb) / 2 * rank in.
                const int32_t rowB = w.tn * BN;
                for (int32_t i = 0; i < w.kb1 - w.kb0; ++i) {
                    const int32_t kb = w.rev ? w.kb1 - 1 - i : w.kb0 + i;
                    if (!wait_bounded<Cfg::SETMAXNREG>(empty_bar(stage), phase ^ 1u, p.err, p.timeout_ns, abort_flag, 1)) {
                        ok = false;
                        break;
                    }
                    const bool skip = first && p.debug_skip_first_load && blockIdx.x == 0;
                    first = false;
                    if (!skip) {
                        const uint32_t fb = full_bar(stage);
                        if (rank == 0) mbar_arrive_expect_tx(fb, Cfg::RL ? p.tma_tx : Cfg::STAGE_TX);
                        const uint32_t dA = sA + stage * Cfg::A_BYTES;
                        const uint32_t dB = sB + stage * Cfg::B_BYTES;
                        // K-major operand: one box of 64 K x rows.  MN-major operand: boxes of
                        // 64 rows (MN) x 64 K, 8 KB each, one after the other along MN.
                        const uint32_t fl = (PAIR == 1) ? fb : map_to_cta(fb, 0);
                        auto load = [&](uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z) {
                            if constexpr (PAIR == 1) tma_load_3d(dst, map, fl, x, y, z);
                            else tma_load_3d_pair(dst, map, fl, x, y, z);
                        };
                        if (Cfg::RL && p.rl_on[0]) {
                            // A rows come from the loader warps
                        } else if (!p.a_mn) {
                            load(dA, &tmA, kb * Cfg::BK, rowA, w.b * p.zA);
                        } else {
#pragma unroll
                            for (int i = 0; i < Cfg::BM / 64; ++i)
                                load(dA + 8192u * i, &tmA, rowA + 64 * i, kb * Cfg::BK, w.b * p.zA);
                        }
#pragma unroll
                        for (int nb = 0; nb < Cfg::N_MMAS; ++nb) {
                            const uint32_t dBn = dB + static_cast<uint32_t>(nb * Cfg::B_BOX_BYTES);
                            const int32_t rowBn = rowB + nb * Cfg::MMA_N +
                                                  (nb == 0 ? Cfg::MMA_N : Cfg::MMA_N1) / PAIR * static_cast<int32_t>(rank);
                            if (Cfg::RL && p.rl_on[1]) {
                                // B rows come from the loader warps
                            } else if (!p.b_mn) {
                                load(dBn, &tmB, kb * Cfg::BK, rowBn, w.b * p.zB);
                            } else {
                                if constexpr (Cfg::B_BOX_ROWS % 64 == 0) {
#pragma unroll
                                    for (int i = 0; i < Cfg::B_BOX_ROWS / 64; ++i)
                                        load(dBn + 8192u * i, &tmB, rowBn + 64 * i, kb * Cfg::BK, w.b * p.zB);
                                }
                            }
                        }
                    }
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            // Drain: wait until the MMA has released every slot, so that no
            // tcgen05.commit arrives on this CTA's barriers after it exits.
            for (int i = 0; i < STAGES && ok; ++i) {
                if (!wait_bounded<Cfg::SETMAXNREG>(empty_bar(stage), phase ^ 1u, p.err, p.timeout_ns, abort_flag, 2)) break;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader CTA only)
        if (rank == 0 && lane == 0) {
            const uint32_t IDESC =
                idesc_f16_f32(Cfg::BM * PAIR, Cfg::MMA_N, p.a_mn ? 1u : 0u, p.b_mn ? 1u : 0u, ACC16 ? 0u : 1u);
            const uint32_t IDESC1 =  // the second MMA of a wide tile
                idesc_f16_f32(Cfg::BM * PAIR, Cfg::MMA_N1, p.a_mn ? 1u : 0u, p.b_mn ? 1u : 0u, ACC16 ? 0u : 1u);
            // Per 16-wide K step: +32 bytes inside a K-major 128-byte row, +2048 bytes
            // (16 rows of 128 bytes) in an MN-major box.
            const uint32_t a_step = p.a_mn ? 128u : 2u, b_step = p.b_mn ? 128u : 2u;
            // Descriptors of stage 0; a stage's descriptors differ only in the start-address
            // field (address >> 4, 14 bits: shared memory stays below 256 KB).
            const uint64_t adesc0 = p.a_mn ? smem_desc_mn_sw128(sA) : smem_desc_sw128(sA);
            const uint64_t bdesc0 = p.b_mn ? smem_desc_mn_sw128(sB) : smem_desc_sw128(sB);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            SegIter it = seg_begin<SK>(p, group, ngroups);
            Seg w;
            while (ok && seg_next<SK>(p, it, w)) {
                ck_half(w);
                // One accumulator of 512 columns: wait here for its first half only; the
                // second half is waited for just before its first MMA, so that the tile's
                // first k-block of MMAs runs while the epilogue still drains that half.
                if (!wait_bounded<Cfg::SETMAXNREG>(tempty_bar(Cfg::ACC_BUFS == 1 ? 0 : acc), acc_phase ^ 1u, p.err, p.timeout_ns,
                                  abort_flag, 3))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                bool hi_ready = Cfg::ACC_BUFS != 1;  // second half of the accumulator free
                for (int32_t kb = w.kb0; kb < w.kb1; ++kb) {
                    // The stage was written by TMA (async proxy) and completed through the
                    // mbarrier's transaction count: the wait alone orders the MMA's reads.
                    if (!wait_bounded<Cfg::SETMAXNREG>(full_bar(stage), phase, p.err, p.timeout_ns, abort_flag, 4)) {
                        ok = false;
                        break;
                    }
                    // Loader warps of the other CTA arrive with cluster-scope release.
                    if constexpr (Cfg::RL && PAIR == 2) fence_acq_rel_cluster();
                    const uint64_t adesc = adesc0 + static_cast<uint64_t>(stage * (Cfg::A_BYTES >> 4));
                    const uint64_t bdesc = bdesc0 + static_cast<uint64_t>(stage * (Cfg::B_BYTES >> 4));
#pragma unroll
                    for (int nb = 0; nb < Cfg::N_MMAS; ++nb) {
                        if (nb == 1 && !hi_ready) {
                            if (!wait_bounded<Cfg::SETMAXNREG>(tempty_bar(1), acc_phase ^ 1u, p.err, p.timeout_ns, abort_flag, 3)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            hi_ready = true;
                        }
                        const uint64_t bdesc_n = bdesc + static_cast<uint64_t>(nb * (Cfg::B_BOX_BYTES >> 4));
#pragma unroll
                        for (int k = 0; k < Cfg::BK / 16; ++k) {
                            mma_f16<PAIR>(d_tmem + static_cast<uint32_t>(nb * Cfg::MMA_N), adesc + a_step * k,
                                          bdesc_n + b_step * k, nb == 0 ? IDESC : IDESC1, (kb > w.kb0 || k > 0) ? 1u : 0u);
                        }
                    }
                    if (!ok) break;
                    if constexpr (PAIR == 1) mma_commit(empty_bar(stage));
                    else mma_commit_pair(empty_bar(stage), 0x3);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (ok && !hi_ready)  // (a segment always has k-blocks; keeps the phases in step regardless)
                    ok = wait_bounded<Cfg::SETMAXNREG>(tempty_bar(1), acc_phase ^ 1u, p.err, p.timeout_ns, abort_flag, 3);
                if (!ok) break;
                if constexpr (PAIR == 1) mma_commit(tfull_bar(acc));
                else mma_commit_pair(tfull_bar(acc), 0x3);
                if (++acc == Cfg::ACC_BUFS) { acc = 0; acc_phase ^= 1u; }
            }
        }
    }  // (warps 2-3 of the row-loader variants' first warpgroup are idle)
    } else if (warp >= Cfg::RL_W0) {
        if constexpr (Cfg::RL) setmaxnreg_inc<Cfg::REGS_RL>();
        // ------------------------------------------------------------ row loader (EPI_RL variants)
        // Loader thread lt owns one row of this CTA's part of a stage: A row lt for lt < BM,
        // else B row lt - BM.  Per k-block it loads the aligned 16-byte words covering the
        // row's 64 halves, shifts them into place, zeroes the halves past K, and writes the
        // eight 16-byte chunks of the row where TMA's 128-byte swizzle would put them.
        // Loads run two k-blocks ahead of the stores (register double buffer).
        if constexpr (Cfg::RL) {
            const int lt = static_cast<int>(threadIdx.x) - 32 * Cfg::RL_W0;
            const bool isA = lt < Cfg::BM;
            const int j = isA ? lt : lt - Cfg::BM;  // row within this CTA's block of the operand
            const int op = isA ? 0 : 1;
            if (j < (isA ? Cfg::BM : Cfg::BN_LOCAL) && p.rl_on[op]) {  // warp-uniform
                if (p.pdl) griddep_wait();  // (the other operand is being repacked by the kernel before)
                const uint16_t* const base = static_cast<const uint16_t*>(p.rl_ptr[op]);
                const int64_t ld = p.rl_ld[op], bstride = p.rl_stride[op];
                const int64_t nrows = isA ? p.rows_a : p.rows_b;
                const int32_t kb_total = p.kb_total;
                // Cursor over this CTA group's data-parallel tiles and their k-blocks.
                struct Cur {
                    int64_t u;             // work unit
                    int32_t i;             // k-block index within the tile, in load order
                    int32_t rev;           // serpentine: k-blocks in reverse order
                    const uint16_t* row;   // this thread's row at k = 0, or null past the operand
                };
                auto cur_tile = [&](Cur& c, int32_t wave) {
                    c.i = 0;
                    c.row = nullptr;
                    c.rev = p.serp & wave;
                    if (c.u >= p.num_units) return;
                    Seg t;
                    tile_coords(p, c.u, t);
                    const int64_t r = isA ? static_cast<int64_t>(t.tm) * (Cfg::BM * PAIR) + Cfg::BM * rank + j
                                          : static_cast<int64_t>(t.tn) * BN + Cfg::B_BOX_ROWS * rank + j;
                    if (r < nrows) c.row = base + static_cast<int64_t>(t.b) * bstride + r * ld;
                };
                Cur cl, cs;  // load cursor (two k-blocks ahead) and store cursor
                int32_t wl = 0, ws = 0;  // wave parities of the two cursors
                cl.u = cs.u = group;
                cur_tile(cl, wl);
                cur_tile(cs, ws);
                auto step = [&](Cur& c, int32_t& wave) {
                    if (++c.i >= kb_total) {
                        c.u += ngroups;
                        wave ^= 1;
                        cur_tile(c, wave);
                    }
                };
                // Issues the loads of the cursor's k-block; returns the shift of the row start
                // within its first word and the number of real halves in `valid`.
                auto issue = [&](const Cur& c, uint32_t (&v)[36], int& valid) -> uint32_t {
                    valid = 0;
                    const uint16_t* src = nullptr;
                    if (c.u < p.num_units && c.row != nullptr) {
                        const int32_t kb = c.rev ? kb_total - 1 - c.i : c.i;
                        const int64_t k0 = static_cast<int64_t>(kb) * Cfg::BK;
                        valid = static_cast<int>(p.K - k0 < Cfg::BK ? p.K - k0 : Cfg::BK);
                        src = c.row + k0;
                    }
                    if (isA) return load_cover64(src, valid, v, GTN_ROW_CHECK(p.ext_a, p.err, CHK_RL_A));
                    return load_cover64(src, valid, v, GTN_ROW_CHECK(p.ext_b, p.err, CHK_RL_B));
                };
                const uint32_t sbase_op = isA ? sA : sB;
                const uint32_t stage_bytes = isA ? Cfg::A_BYTES : Cfg::B_BYTES;
                const uint32_t row_off = static_cast<uint32_t>(j) * 128u;
                const uint32_t sw = static_cast<uint32_t>(j) & 7u;
                int stage = 0;
                uint32_t phase = 0;
                bool ok = true;
                // Writes one k-block's row into the ring slot and signals the stage.
                auto put = [&](const uint32_t (&v)[36], uint32_t sh, int valid) {
                    int go = 1;
                    if (lane == 0)
                        go = wait_bounded<Cfg::SETMAXNREG>(empty_bar(stage), phase ^ 1u, p.err, p.timeout_ns, abort_flag, 7) ? 1 : 0;
                    go = __shfl_sync(0xffffffffu, go, 0);
                    if (!go) {
                        ok = false;
                        return;
                    }
                    uint32_t w[32];
                    align_cover64(v, sh, w);
                    if (valid < Cfg::BK) {
#pragma unroll
                        for (int q = 0; q < 32; ++q) {
                            const int e = 2 * q;
                            w[q] = e >= valid ? 0u : (e + 1 >= valid ? (w[q] & 0xffffu) : w[q]);
                        }
                    }
                    const uint32_t dst = sbase_op + static_cast<uint32_t>(stage) * stage_bytes + row_off;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        st_shared_v4(dst + ((static_cast<uint32_t>(c) ^ sw) << 4), w[4 * c], w[4 * c + 1], w[4 * c + 2],
                                     w[4 * c + 3]);
                    fence_proxy_async_smem();  // the tensor core reads the slot through the async proxy
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (PAIR == 1) mbar_arrive(full_bar(stage));
                        else mbar_arrive_cluster(map_to_cta(full_bar(stage), 0));
                    }
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                };
                uint32_t va[36], vb[36];
                int na = 0, nb = 0;
                uint32_t sa = issue(cl, va, na);
                step(cl, wl);
                uint32_t sb = issue(cl, vb, nb);
                step(cl, wl);
                while (ok && cs.u < p.num_units) {
                    put(va, sa, na);
                    if (!ok) break;
                    step(cs, ws);
                    sa = issue(cl, va, na);
                    step(cl, wl);
                    if (cs.u >= p.num_units) break;
                    put(vb, sb, nb);
                    if (!ok) break;
                    step(cs, ws);
                    sb = issue(cl, vb, nb);
                    step(cl, wl);
                }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue warps
        if constexpr (Cfg::SETMAXNREG) setmaxnreg_inc<Cfg::REGS_EPI>();
        const int ew = warp - Cfg::EPI_W0;
        const int quarter = warp & 3;  // tensor-memory lanes 32*quarter .. +31 are this warp's
        uint8_t* ebuf = smem + Cfg::OFF_EPI + ew * Cfg::EPI_WARP_BYTES;
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t chunk_count = 0;
        uint32_t xphase = 0;  // cluster K split: parity of the next partial-buffer wait
        bool x_first = true;  // cluster K split: no partial has gone through the buffers yet
        const bool use_c = (EB == EPI_GENERIC || EB == EPI_SWAP) && p.beta != 0.0f;
        // TMA epilogue with beta != 0: C boxes are fetched by TMA into the staging buffers.
        constexpr bool tma_c = EPI == EPI_TMA_C;
        uint32_t cphase = 0u;  // bit b: parity of the next C load into staging buffer b
        SegIter it = seg_begin<SK>(p, group, ngroups);
        Seg w;
        while (seg_next<SK>(p, it, w)) {
            // First accumulator row / column of this warp, in the tensor-core view.
            const int64_t arow0 = static_cast<int64_t>(w.tm) * (Cfg::BM * PAIR) + Cfg::BM * rank + quarter * 32;
            const int64_t acol0 = static_cast<int64_t>(w.tn) * BN;
            const bool partial = SK && w.sk_tile >= 0;
            // This warp's block of the partial-accumulator slot of contributor j,
            // stored column by column ([col][lane]) so a warp's accesses coalesce.
            auto slot_block = [&](int j) -> float* {
                return p.sk_W + (((static_cast<int64_t>(w.sk_tile) * p.sk_maxc + j) * PAIR + rank) * 4 + quarter) *
                                    static_cast<int64_t>(32 * BN) +
                       lane;
            };
            // Predicated epilogue: C of the first 32-column chunk is fetched before the
            // accumulator is ready, so its memory latency overlaps the main loop.
            __half cnext[32];
            auto load_c_chunk = [&](int c, __half (&dst)[32]) {
                const int64_t col = acol0 + c * 32 + lane;
                const bool col_ok = col < p.N;
                const __half* src = static_cast<const __half*>(p.C) + static_cast<int64_t>(w.b) * p.strideC + col;
#pragma unroll
                for (int r = 0; r < 32; ++r)
                    dst[r] = (col_ok && arow0 + r < p.M &&
                              chk_elem(src + (arow0 + r) * p.ldc, p.ext_c, p.err, CHK_EPI_C_ELEM))
                                 ? src[(arow0 + r) * p.ldc]
                                 : __ushort_as_half(0);
            };
            if constexpr (EB == EPI_GENERIC) {
                if (use_c && !partial) load_c_chunk(0, cnext);
            }
            // TMA epilogue: request the C box (32 rows x 64 columns) of chunk c into staging
            // buffer b (lane 0 only).
            auto issue_c = [&](int c, uint32_t b) {
                const uint32_t cb = cload_bar(ew, static_cast<int>(b));
                mbar_arrive_expect_tx(cb, 4096u);
                tma_load_3d(smem_u32(ebuf) + b * 4096u, &tmC, cb, static_cast<int32_t>(acol0 + c * 64),
                            static_cast<int32_t>(arow0), w.b * p.zC);
            };
            // The first chunk's C is requested before the accumulator is ready; the buffer
            // it lands in was last read by the store issued two chunks ago.
            auto issue_first_c = [&]() {
                if (lane == 0) {
                    bulk_wait_group_read<1>();
                    issue_c(0, chunk_count & 1u);
                }
            };
            if constexpr (EPI == EPI_TMA_C) {
                if (!partial) issue_first_c();
            }
            // Misaligned C: the words covering this thread's row of 64-column chunk c,
            // requested one chunk ahead (the first before the accumulator is ready) and
            // shifted into place when the chunk is written.
            uint32_t ccover[36];
            uint32_t c_sh = 0;
            auto prefetch_cg = [&](int c) {
                const int64_t row = arow0 + lane;
                const int64_t col0 = acol0 + c * 64;
                const __half* src = static_cast<const __half*>(p.C);
                int valid = 0;
                if (row < p.M && col0 < p.N) {
                    valid = static_cast<int>(p.N - col0 < 64 ? p.N - col0 : 64);
                    src += static_cast<int64_t>(w.b) * p.strideC + row * p.ldc + col0;
                }
                c_sh = load_cover64(reinterpret_cast<const uint16_t*>(src), valid, ccover,
                                    GTN_ROW_CHECK(p.ext_c, p.err, CHK_EPI_C_ROW));
            };
            if constexpr (EPI == EPI_TMA_CG || EPI == EPI_VEC) {
                if (!partial && p.beta != 0.0f) prefetch_cg(0);
            }
            int ok = 1;
            if (lane == 0) ok = wait_bounded<Cfg::SETMAXNREG>(tfull_bar(acc), acc_phase, p.err, p.timeout_ns, abort_flag, 5) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * BN);
            // This warp is done reading accumulator part `idx` (a whole accumulator, or a
            // half of the single 512-column one).
            auto arrive_tempty = [&](int idx) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (PAIR == 1) mbar_arrive(tempty_bar(idx));
                    else mbar_arrive_cluster(map_to_cta(tempty_bar(idx), 0));
                }
            };
            bool lo_released = false;
            // 32 accumulator columns of this thread's row as fp32 bits (fp16 accumulators widened).
            auto acc_ld32 = [&](int col, uint32_t (&v)[32]) {
                if constexpr (!ACC16) {
                    tmem_ld_32x32b_x32(t_row + col, v);
                    tmem_ld_wait();
                } else {
                    // an fp16 accumulator holds one element per 32-bit column; two
                    // adjacent columns are packed into each register on the way out
                    uint32_t h[16];
                    tmem_ld_32x32b_x32_pack16(t_row + col, h);
                    tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[q]));
                        v[2 * q] = __float_as_uint(f.x);
                        v[2 * q + 1] = __float_as_uint(f.y);
                    }
                }
            };

            // Sum of all contributors' partials for this thread's row, columns
            // [col, col + NC), added in contributor order (deterministic).  The loads of
            // IN contributors are in flight at a time: four for narrow tiles (all of a
            // skinny GEMM's contributors in one round trip), else two.
            auto sum_parts = [&](int col, auto& v) {
                constexpr int NC = sizeof(v) / sizeof(v[0]);
                constexpr int IN = NC <= 16 ? 4 : 2;
                float acc_f[NC];
#pragma unroll
                for (int q = 0; q < NC; ++q) acc_f[q] = 0.0f;
                for (int j = 0; j < w.sk_n; j += IN) {
                    float a[IN][NC];
#pragma unroll
                    for (int u = 0; u < IN; ++u) {
                        const float* s = slot_block(j + u < w.sk_n ? j + u : j) + col * 32;
#pragma unroll
                        for (int q = 0; q < NC; ++q) a[u][q] = __ldcg(s + q * 32);
                    }
#pragma unroll
                    for (int u = 0; u < IN; ++u) {
                        if (j + u < w.sk_n) {
#pragma unroll
                            for (int q = 0; q < NC; ++q) acc_f[q] += a[u][q];
                        }
                    }
                }
#pragma unroll
                for (int q = 0; q < NC; ++q) v[q] = __float_as_uint(acc_f[q]);
            };

            // Writes the finished tile (this warp's 32 rows) from tensor memory, or
            // (stream-K fixup, PARTS) from the sum of the contributors' partials.
            auto emit_tile = [&](auto parts_tag) {
                constexpr bool PARTS = decltype(parts_tag)::value;
                // Called once chunk c (64 columns) has been read out of tensor memory: the
                // first half of a 512-column accumulator goes back to the MMA early.
                auto fetched = [&](int c) {
                    if constexpr (!PARTS && Cfg::ACC_BUFS == 1) {
                        if (c == Cfg::MMA_N / 64 - 1) {
                            arrive_tempty(0);
                            lo_released = true;
                        }
                    }
                };
                if constexpr (EB == EPI_VEC) {
                    // D (and C) at any 2-byte alignment: this thread's row, 64 columns at a
                    // time, through the aligned 16-byte words that cover it; only the real
                    // elements are written.  Same arithmetic and rounding as the TMA epilogue.
                    const bool with_c = p.beta != 0.0f;
                    if constexpr (PARTS) {
                        if (with_c) prefetch_cg(0);
                    }
                    const int64_t row = arow0 + lane;
                    __half* const drow =
                        static_cast<__half*>(p.D) + static_cast<int64_t>(w.b) * p.strideD + row * p.ldd;
#pragma unroll 1
                    for (int c = 0; c < BN / 64; ++c) {
                        uint32_t cw[32];
                        if (with_c) {
                            align_cover64(ccover, c_sh, cw);
                            if (c + 1 < BN / 64) prefetch_cg(c + 1);
                        }
                        uint32_t v0[32], v1[32];
                        if constexpr (!PARTS) {
                            tmem_ld_32x32b_x32(t_row + c * 64, v0);
                            tmem_ld_32x32b_x32(t_row + c * 64 + 32, v1);
                            tmem_ld_wait();
                        } else {
                            sum_parts(c * 64, v0);
                            sum_parts(c * 64 + 32, v1);
                        }
                        const float al = p.alpha, be = p.beta;
                        uint32_t o[32];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            float x0 = al * __uint_as_float(v0[2 * i]), x1 = al * __uint_as_float(v0[2 * i + 1]);
                            float y0 = al * __uint_as_float(v1[2 * i]), y1 = al * __uint_as_float(v1[2 * i + 1]);
                            if (with_c) {
                                const float2 c0 = __half22float2(*reinterpret_cast<const __half2*>(&cw[i]));
                                const float2 c1 = __half22float2(*reinterpret_cast<const __half2*>(&cw[16 + i]));
                                x0 = fmaf(be, c0.x, x0);
                                x1 = fmaf(be, c0.y, x1);
                                y0 = fmaf(be, c1.x, y0);
                                y1 = fmaf(be, c1.y, y1);
                            }
                            o[i] = pack_half2(x0, x1);
                            o[16 + i] = pack_half2(y0, y1);
                        }
                        const int64_t col0 = acol0 + c * 64;
                        const int valid =
                            (row < p.M && col0 < p.N) ? static_cast<int>(p.N - col0 < 64 ? p.N - col0 : 64) : 0;
                        store_row64(reinterpret_cast<uint16_t*>(drow + col0), valid, o,
                                    GTN_ROW_CHECK(p.ext_d, p.err, CHK_EPI_D_ROW));
                    }
                } else if constexpr (EB == EPI_TMA || EPI == EPI_TMA_C || EPI == EPI_TMA_CG) {
                    auto fetch64 = [&](int c, uint32_t (&v0)[32], uint32_t (&v1)[32]) {
                        if constexpr (!PARTS && ACC16) {
                            acc_ld32(c * 64, v0);
                            acc_ld32(c * 64 + 32, v1);
                        } else if constexpr (!PARTS) {
                            tmem_ld_32x32b_x32(t_row + c * 64, v0);
                            tmem_ld_32x32b_x32(t_row + c * 64 + 32, v1);
                            tmem_ld_wait();
                        } else {
                            sum_parts(c * 64, v0);
                            sum_parts(c * 64 + 32, v1);
                        }
                    };
                    auto store_chunk = [&](int c, uint32_t sb) {
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_3d(&tmD, sb, static_cast<int32_t>(acol0 + c * 64), static_cast<int32_t>(arow0),
                                         w.b * p.zD);
                            bulk_commit_group();
                        }
                        ++chunk_count;
                    };
                    if constexpr (Cfg::H2 && !PARTS) {
                        // Two epilogue warpgroups: warps EPI_W0 .. +3 take the first MMA's
                        // columns [0, MMA_N), the next four the second's [MMA_N, BN).  Each warp
                        // reads all of its part of its 32 rows into registers as fp16 (alpha
                        // applied, rounded once), hands the part back to the MMA, and only then
                        // stores it, chunk by chunk through its staging buffer.  The 48-column
                        // tail of a 432-column tile goes first, straight from registers.
                        constexpr int P0 = Cfg::MMA_N / 64;       // whole chunks of part 0
                        constexpr int P1 = Cfg::FULL_CHUNKS - P0;  // whole chunks of part 1
                        constexpr int PMAX = P0 > P1 ? P0 : P1;
                        const int part = ew / 4;
                        const int c0 = part == 0 ? 0 : P0;
                        const int nch = part == 0 ? P0 : P1;
                        const float al = p.alpha;
                        if constexpr (Cfg::TAIL_COLS == 48) {
                            if (part == 1) {
                                uint32_t v0[32], v1[16];
                                tmem_ld_32x32b_x32(t_row + Cfg::FULL_CHUNKS * 64, v0);
                                tmem_ld_32x32b_x16(t_row + Cfg::FULL_CHUNKS * 64 + 32, v1);
                                tmem_ld_wait();
                                uint32_t o[32];
#pragma unroll
                                for (int j = 0; j < 16; ++j)
                                    o[j] = pack_half2(al * __uint_as_float(v0[2 * j]), al * __uint_as_float(v0[2 * j + 1]));
#pragma unroll
                                for (int j = 0; j < 8; ++j)
                                    o[16 + j] = pack_half2(al * __uint_as_float(v1[2 * j]), al * __uint_as_float(v1[2 * j + 1]));
#pragma unroll
                                for (int j = 24; j < 32; ++j) o[j] = 0u;
                                const int64_t row = arow0 + lane;
                                const int64_t col0 = acol0 + Cfg::FULL_CHUNKS * 64;
                                const int valid = (row < p.M && col0 < p.N)
                                                      ? static_cast<int>(p.N - col0 < Cfg::TAIL_COLS ? p.N - col0
                                                                                                     : Cfg::TAIL_COLS)
                                                      : 0;
                                __half* const drow =
                                    static_cast<__half*>(p.D) + static_cast<int64_t>(w.b) * p.strideD + row * p.ldd;
                                store_row64(reinterpret_cast<uint16_t*>(drow + col0), valid, o,
                                            GTN_ROW_CHECK(p.ext_d, p.err, CHK_EPI_D_ROW));
                            }
                        }
                        uint32_t pk[PMAX][32];
#pragma unroll
                        for (int i = 0; i < PMAX; ++i) {
                            if (i < nch) {
#pragma unroll
                                for (int h = 0; h < 2; ++h) {
                                    uint32_t v[32];
                                    tmem_ld_32x32b_x32(t_row + (c0 + i) * 64 + h * 32, v);
                                    tmem_ld_wait();
#pragma unroll
                                    for (int j = 0; j < 16; ++j)
                                        pk[i][16 * h + j] =
                                            pack_half2(al * __uint_as_float(v[2 * j]), al * __uint_as_float(v[2 * j + 1]));
                                }
                            }
                        }
                        arrive_tempty(part);
#pragma unroll
                        for (int i = 0; i < PMAX; ++i) {
                            if (i < nch) {
                                if (lane == 0) bulk_wait_group_read<0>();  // the staging buffer's last store has read it
                                __syncwarp();
                                const uint32_t sb = smem_u32(ebuf);
                                const uint32_t row_addr = sb + lane * 128u;
#pragma unroll
                                for (int j = 0; j < 8; ++j)
                                    st_shared_v4(row_addr + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4), pk[i][4 * j],
                                                 pk[i][4 * j + 1], pk[i][4 * j + 2], pk[i][4 * j + 3]);
                                store_chunk(c0 + i, sb);
                            }
                        }
                    } else if constexpr (EPI == EPI_TMA_CG) {
                        // D = alpha * acc + beta * C, C read from global memory at its own alignment
                        if constexpr (PARTS) prefetch_cg(0);
#pragma unroll 1
                        for (int c = 0; c < BN / 64; ++c) {
                            uint32_t cw[32];
                            align_cover64(ccover, c_sh, cw);
                            if (c + 1 < BN / 64) prefetch_cg(c + 1);
                            uint32_t v0[32], v1[32];
                            fetch64(c, v0, v1);
                            fetched(c);
                            const uint32_t buf = chunk_count & 1u;
                            if (lane == 0) bulk_wait_group_read<1>();  // this buffer's previous store has read it
                            __syncwarp();
                            const uint32_t sb = smem_u32(ebuf) + buf * 4096u;
                            const uint32_t row_addr = sb + lane * 128u;
                            const float al = p.alpha, be = p.beta;
                            // alpha * acc + beta * C for two columns, rounded once to fp16
                            auto o2 = [&](uint32_t xa, uint32_t xb, uint32_t cword) {
                                const float2 cf = __half22float2(*reinterpret_cast<const __half2*>(&cword));
                                return pack_half2(fmaf(be, cf.x, al * __uint_as_float(xa)),
                                                  fmaf(be, cf.y, al * __uint_as_float(xb)));
                            };
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                st_shared_v4(row_addr + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4),
                                             o2(v0[8 * j + 0], v0[8 * j + 1], cw[4 * j + 0]),
                                             o2(v0[8 * j + 2], v0[8 * j + 3], cw[4 * j + 1]),
                                             o2(v0[8 * j + 4], v0[8 * j + 5], cw[4 * j + 2]),
                                             o2(v0[8 * j + 6], v0[8 * j + 7], cw[4 * j + 3]));
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                st_shared_v4(row_addr + ((static_cast<uint32_t>(j + 4) ^ (lane & 7u)) << 4),
                                             o2(v1[8 * j + 0], v1[8 * j + 1], cw[16 + 4 * j + 0]),
                                             o2(v1[8 * j + 2], v1[8 * j + 3], cw[16 + 4 * j + 1]),
                                             o2(v1[8 * j + 4], v1[8 * j + 5], cw[16 + 4 * j + 2]),
                                             o2(v1[8 * j + 6], v1[8 * j + 7], cw[16 + 4 * j + 3]));
                            store_chunk(c, sb);
                        }
                    } else if constexpr (!tma_c) {
                        // D = alpha * acc
#pragma unroll 1
                        for (int c = 0; c < Cfg::FULL_CHUNKS; ++c) {
                            uint32_t v0[32], v1[32];
                            fetch64(c, v0, v1);
                            fetched(c);
                            const uint32_t buf = chunk_count & (Cfg::NBUF - 1);
                            // this buffer's previous store has read it
                            if (lane == 0) bulk_wait_group_read<Cfg::NBUF - 1>();
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
                            store_chunk(c, sb);
                        }
                        if constexpr (Cfg::TAIL_COLS == 48 && !PARTS && !ACC16) {
                            // The last 48 columns (32 + 16 of tensor memory): this thread's row
                            // segment goes out from registers in 16-byte stores (D is 16-byte
                            // aligned here).
                            uint32_t v0[32], v1[16];
                            tmem_ld_32x32b_x32(t_row + Cfg::FULL_CHUNKS * 64, v0);
                            tmem_ld_32x32b_x16(t_row + Cfg::FULL_CHUNKS * 64 + 32, v1);
                            tmem_ld_wait();
                            const float al = p.alpha;
                            uint32_t o[32];
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                o[i] = pack_half2(al * __uint_as_float(v0[2 * i]), al * __uint_as_float(v0[2 * i + 1]));
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                o[16 + i] = pack_half2(al * __uint_as_float(v1[2 * i]), al * __uint_as_float(v1[2 * i + 1]));
#pragma unroll
                            for (int i = 24; i < 32; ++i) o[i] = 0u;
                            const int64_t row = arow0 + lane;
                            const int64_t col0 = acol0 + Cfg::FULL_CHUNKS * 64;
                            const int valid = (row < p.M && col0 < p.N)
                                                  ? static_cast<int>(p.N - col0 < Cfg::TAIL_COLS ? p.N - col0 : Cfg::TAIL_COLS)
                                                  : 0;
                            __half* const drow =
                                static_cast<__half*>(p.D) + static_cast<int64_t>(w.b) * p.strideD + row * p.ldd;
                            store_row64(reinterpret_cast<uint16_t*>(drow + col0), valid, o,
                                        GTN_ROW_CHECK(p.ext_d, p.err, CHK_EPI_D_ROW));
                        }
                    } else {
                        // D = alpha * acc + beta * C, C boxes loaded by TMA into the staging buffers
                        if constexpr (PARTS) issue_first_c();
#pragma unroll 1
                        for (int c = 0; c < BN / 64; ++c) {
                            uint32_t v0[32], v1[32];
                            fetch64(c, v0, v1);
                            fetched(c);
                            const uint32_t buf = chunk_count & 1u;
                            if (lane == 0) {
                                // the other buffer's store (last chunk) must have read its data
                                // before the next chunk's C lands there
                                bulk_wait_group_read<0>();
                                if (c + 1 < BN / 64) issue_c(c + 1, buf ^ 1u);
                                wait_bounded<Cfg::SETMAXNREG>(cload_bar(ew, static_cast<int>(buf)), (cphase >> buf) & 1u, p.err,
                                             p.timeout_ns, abort_flag, 6);
                            }
                            cphase ^= 1u << buf;
                            __syncwarp();
                            const uint32_t sb = smem_u32(ebuf) + buf * 4096u;
                            const uint32_t row_addr = sb + lane * 128u;
                            const float al = p.alpha, be = p.beta;
                            // alpha * acc + beta * C for 8 columns, rounded once to fp16, in place
                            auto out8 = [&](const uint32_t* v, uint32_t addr) {
                                uint32_t cw[4];
                                ld_shared_v4(addr, cw[0], cw[1], cw[2], cw[3]);
                                float x[8];
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    const float2 cf = __half22float2(*reinterpret_cast<const __half2*>(&cw[q]));
                                    x[2 * q] = fmaf(be, cf.x, al * __uint_as_float(v[2 * q]));
                                    x[2 * q + 1] = fmaf(be, cf.y, al * __uint_as_float(v[2 * q + 1]));
                                }
                                st_shared_v4(addr, pack_half2(x[0], x[1]), pack_half2(x[2], x[3]), pack_half2(x[4], x[5]),
                                             pack_half2(x[6], x[7]));
                            };
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                out8(v0 + 8 * j, row_addr + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4));
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                out8(v1 + 8 * j, row_addr + ((static_cast<uint32_t>(j + 4) ^ (lane & 7u)) << 4));
                            store_chunk(c, sb);
                        }
                    }
                } else if constexpr (EB == EPI_GENERIC || EB == EPI_PARTIAL) {
                    bool stored = false;
                    if constexpr (EB == EPI_PARTIAL) {
                        if (p.w_tma) {
                            // fp32 partials by TMA: 32 columns (128 bytes) of this thread's row
                            // into the swizzled staging buffer, one 32 x 32 box per chunk.
#pragma unroll 1
                            for (int c = 0; c < BN / 32; ++c) {
                                uint32_t v[32];
                                if constexpr (!PARTS) {
                                    acc_ld32(c * 32, v);
                                } else {
                                    sum_parts(c * 32, v);
                                }
                                const uint32_t buf = chunk_count & 1u;
                                if (lane == 0) bulk_wait_group_read<1>();  // this buffer's previous store has read it
                                __syncwarp();
                                const uint32_t sb = smem_u32(ebuf) + buf * 4096u;
                                const uint32_t row_addr = sb + lane * 128u;
#pragma unroll
                                for (int j = 0; j < 8; ++j)
                                    st_shared_v4(row_addr + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4), v[4 * j],
                                                 v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                                fence_proxy_async_smem();
                                __syncwarp();
                                if (lane == 0) {
                                    tma_store_3d(&tmD, sb, static_cast<int32_t>(acol0 + c * 32),
                                                 static_cast<int32_t>(arow0), w.b * p.splits + w.split);
                                    bulk_commit_group();
                                }
                                ++chunk_count;
                            }
                            stored = true;
                        }
                    }
                    if (stored) return;
                    // Transpose each 32x32 block through padded shared memory so that a warp
                    // reads C and writes D along rows (coalesced), whatever the alignment.
                    float* T = reinterpret_cast<float*>(ebuf);
                    __half* Dp = static_cast<__half*>(p.D);
                    if constexpr (EB == EPI_GENERIC) {
                        if (use_c && PARTS) load_c_chunk(0, cnext);
                    }
#pragma unroll 1
                    for (int c = 0; c < BN / 32; ++c) {
                        __half ccur[32];
                        if constexpr (EB == EPI_GENERIC) {
                            if (use_c) {
#pragma unroll
                                for (int r = 0; r < 32; ++r) ccur[r] = cnext[r];
                                // Loads for the next chunk are issued before this chunk's stores
                                // (different columns, so an aliased C == D stays correct).
                                if (c + 1 < BN / 32) load_c_chunk(c + 1, cnext);
                            }
                        }
                        uint32_t v[32];
                        if constexpr (!PARTS) {
                            acc_ld32(c * 32, v);
                        } else {
                            sum_parts(c * 32, v);
                        }
#pragma unroll
                        for (int j = 0; j < 32; ++j) T[lane * 33 + j] = __uint_as_float(v[j]);
                        __syncwarp();
                        const int64_t col = acol0 + c * 32 + lane;
                        if (col < p.N) {
                            if constexpr (EB == EPI_GENERIC) {
                                __half* dst = Dp + static_cast<int64_t>(w.b) * p.strideD + col;
#pragma unroll
                                for (int r = 0; r < 32; ++r) {
                                    const int64_t row = arow0 + r;
                                    if (row < p.M) {
                                        float x = p.alpha * T[r * 33 + lane];
                                        if (use_c) x = fmaf(p.beta, __half2float(ccur[r]), x);
                                        if (chk_elem(dst + row * p.ldd, p.ext_d, p.err, CHK_EPI_D_ELEM))
                                            dst[row * p.ldd] = __float2half_rn(x);
                                    }
                                }
                            } else {
                                float* Wp = p.W + (static_cast<int64_t>(w.b) * p.splits + w.split) * p.M * p.N + col;
#pragma unroll 8
                                for (int r = 0; r < 32; ++r) {
                                    const int64_t row = arow0 + r;
                                    if (row < p.M && chk_elem(Wp + row * p.N, p.ext_w, p.err, CHK_EPI_W))
                                        Wp[row * p.N] = T[r * 33 + lane];
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
                    // Cluster K split: this thread's row of the partial buffer.  CTA 1 stages its
                    // partial in its own buffer and each warp sends its 32 rows to the same place in
                    // CTA 0's with one bulk copy, whose bytes complete CTA 0's barrier: no
                    // cluster-scope fence or remote arrive lies between the two main loops' end
                    // and the sum.
                    const uint32_t xrow = smem_u32(smem + Cfg::OFF_X) + static_cast<uint32_t>((quarter * 32 + lane) * BN * 4);
                    const uint32_t xwarp = smem_u32(smem + Cfg::OFF_X) + static_cast<uint32_t>(quarter * 32 * BN * 4);
                    constexpr uint32_t XW_BYTES = 32u * BN * 4u;  // one warp's rows of the partial
                    // Both CTAs of the cluster walk the same whole-tile units (the cluster K split
                    // is data-parallel): another one follows this tile iff the iterator has one left.
                    [[maybe_unused]] const bool x_more = SK || it.dp_next < p.num_units;
                    if constexpr (Cfg::CK) {
                        int got = 1;
                        if (krank == 0) {
                            // arm this tile's phase with this warp's bytes, then wait for all four warps'
                            if (lane == 0) {
                                mbar_arrive_expect_tx(xfull_bar, XW_BYTES);
                                got = wait_bounded<Cfg::SETMAXNREG>(xfull_bar, xphase, p.err, p.timeout_ns, abort_flag, 8)
                                          ? 1 : 0;
                            }
                        } else if (!x_first) {
                            // CTA 0 has read the previous partial out of its buffer, and this warp's
                            // previous copy has read the staged rows
                            if (lane == 0) {
                                got = wait_bounded<Cfg::SETMAXNREG>(xempty_bar, xphase ^ 1u, p.err, p.timeout_ns, abort_flag, 8)
                                          ? 1 : 0;
                                bulk_wait_group_read<0>();
                            }
                        }
                        got = __shfl_sync(0xffffffffu, got, 0);
                        if (!got) return;
                        // CTA 0's reads of the previous partial (released by its remote arrive)
                        // happen before this tile's copy writes the buffer again
                        if (krank == 1 && !x_first) fence_acq_rel_cluster();
                        x_first = false;
                        xphase ^= 1u;
                    }
#pragma unroll 1
                    for (int c = 0; c < BN / 16; ++c) {
                        uint32_t v[16];
                        if constexpr (!PARTS) {
                            tmem_ld_32x32b_x16(t_row + c * 16, v);
                            tmem_ld_wait();
                        } else {
                            sum_parts(c * 16, v);
                        }
                        if constexpr (Cfg::CK) {
                            const uint32_t xa = xrow + static_cast<uint32_t>(c * 64);
                            if (krank == 1) {
                                // stage the partial for CTA 0 and write nothing
#pragma unroll
                                for (int q = 0; q < 4; ++q)
                                    st_shared_v4(xa + 16u * q, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                                continue;
                            }
                            // CTA 0: add the partial, first half of K before the second
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                uint32_t x0, x1, x2, x3;
                                ld_shared_v4(xa + 16u * q, x0, x1, x2, x3);
                                v[4 * q] = __float_as_uint(__uint_as_float(v[4 * q]) + __uint_as_float(x0));
                                v[4 * q + 1] = __float_as_uint(__uint_as_float(v[4 * q + 1]) + __uint_as_float(x1));
                                v[4 * q + 2] = __float_as_uint(__uint_as_float(v[4 * q + 2]) + __uint_as_float(x2));
                                v[4 * q + 3] = __float_as_uint(__uint_as_float(v[4 * q + 3]) + __uint_as_float(x3));
                            }
                            if (c == BN / 16 - 1 && x_more) {
                                // the whole partial is in registers: CTA 1 may send the next one (the
                                // arrive's release then waits only for these reads, not for the D
                                // stores that follow).  After the cluster's last tile CTA 1 sends
                                // nothing more, and the cluster-scope release would only delay the
                                // stores.
                                __syncwarp();
                                if (lane == 0) mbar_arrive_cluster(map_to_cta(xempty_bar, 1));
                            }
                        }
                        if (n < p.N) {
                            if constexpr (EB == EPI_SWAP) {
                                // all C loads of the chunk first, then the stores
                                __half cv[16];
#pragma unroll
                                for (int j = 0; j < 16; ++j) {
                                    const int64_t m = acol0 + c * 16 + j;
                                    const __half* ca = Cp + static_cast<int64_t>(w.b) * p.strideC + m * p.ldc + n;
                                    cv[j] = (use_c && m < p.M && chk_elem(ca, p.ext_c, p.err, CHK_EPI_C_ELEM))
                                                ? *ca
                                                : __ushort_as_half(0);
                                }
#pragma unroll
                                for (int j = 0; j < 16; ++j) {
                                    const int64_t m = acol0 + c * 16 + j;
                                    __half* da = Dp + static_cast<int64_t>(w.b) * p.strideD + m * p.ldd + n;
                                    if (m < p.M && chk_elem(da, p.ext_d, p.err, CHK_EPI_D_ELEM)) {
                                        float x = p.alpha * __uint_as_float(v[j]);
                                        if (use_c) x = fmaf(p.beta, __half2float(cv[j]), x);
                                        *da = __float2half_rn(x);
                                    }
                                }
                            } else {
#pragma unroll
                                for (int j = 0; j < 16; ++j) {
                                    const int64_t m = acol0 + c * 16 + j;
                                    float* wa = p.W + ((static_cast<int64_t>(w.b) * p.splits + w.split) * p.M + m) * p.N + n;
                                    if (m < p.M && chk_elem(wa, p.ext_w, p.err, CHK_EPI_W)) *wa = __uint_as_float(v[j]);
                                }
                            }
                        }
                    }
                    if constexpr (Cfg::CK) {
                        if (krank == 1) {
                            // the staged rows (generic proxy) are read by the bulk copy (async proxy)
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                bulk_copy_to_cluster(map_to_cta(xwarp, 0), xwarp, XW_BYTES, map_to_cta(xfull_bar, 0));
                                bulk_commit_group();
                            }
                        }
                    }
                }
            };

            auto release_accumulator = [&]() {
                if constexpr (Cfg::ACC_BUFS == 1) {
                    if constexpr (!Cfg::H2) {  // (with two epilogue warpgroups each warp has handed its part back)
                        if (!lo_released) arrive_tempty(0);
                        arrive_tempty(1);
                    }
                    acc_phase ^= 1u;
                } else {
                    arrive_tempty(acc);
                    if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
                }
            };

            if (!partial) {
                emit_tile(std::false_type{});
                release_accumulator();  // this warp is done reading the accumulator
            } else if constexpr (SK) {
                // Stream-K contribution: park this warp's 32 rows of the accumulator in its slot.
                float* mine = slot_block(w.sk_j);
                constexpr int PW = (BN % 32 == 0) ? 32 : 16;  // columns per tensor-memory load
#pragma unroll 1
                for (int c = 0; c < BN / PW; ++c) {
                    uint32_t v[PW];
                    if constexpr (PW == 32) tmem_ld_32x32b_x32(t_row + c * PW, v);
                    else tmem_ld_32x32b_x16(t_row + c * PW, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < PW; ++q) mine[(c * PW + q) * 32] = __uint_as_float(v[q]);
                }
                release_accumulator();
                // Count this warp's 32 rows in; the last contributor for these rows
                // finishes them.  Each warp owns its rows outright, so no warp ever
                // waits for another (an aborted warp cannot strand the others).
                __threadfence();
                __syncwarp();
                uint32_t prev = 0;
                if (lane == 0) {
                    unsigned long long* ctr =
                        p.sk_counters + (static_cast<int64_t>(w.sk_tile) * PAIR + rank) * 4 + quarter;
                    unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(ctr);
                    // at most sk_n contributors race on a word, so the loop is short; the
                    // bound only guards against a word no contributor of this launch wrote
                    for (int attempt = 0; attempt < 4096; ++attempt) {
                        prev = ((old >> 8) == p.sk_epoch) ? static_cast<uint32_t>(old & 0xffu) : 0u;
                        const unsigned long long want = (p.sk_epoch << 8) | (prev + 1u);
                        const unsigned long long seen = atomicCAS(ctr, old, want);
                        if (seen == old) break;
                        old = seen;
                    }
                }
                prev = __shfl_sync(0xffffffffu, prev, 0);
                if (prev == static_cast<uint32_t>(w.sk_n - 1)) {
                    __threadfence();
                    emit_tile(std::true_type{});
                }
            }
        }
        if constexpr (EB == EPI_TMA || EPI == EPI_TMA_C || EPI == EPI_TMA_CG || EPI == EPI_PARTIAL || Cfg::CK) {
            if (lane == 0) bulk_wait_group<0>();  // (cluster K split: CTA 1's copies into CTA 0 have landed)
            __syncwarp();
        }
    }

    // ---------------------------------------------------------------- teardown
    __syncwarp();
    if (*abort_flag) spin_ns(2000000ull);  // let in-flight TMA loads and MMAs land
    tc_fence_before();
    if constexpr (Cfg::CLUSTER == 2) cluster_sync(); else __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc<PAIR>(tmem_base, Cfg::TMEM_COLS);
}

}  // namespace gtn
