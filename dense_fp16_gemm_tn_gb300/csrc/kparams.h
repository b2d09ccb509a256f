// Parameters shared by the host launcher and the tensor-core GEMM kernel.
#pragma once

#include <cstdint>

#include "checked.h"

namespace gtn {

enum EpiMode : int {
    EPI_TMA = 0,           // D = alpha*acc via TMA stores (beta == 0, aligned D)
    EPI_GENERIC = 1,       // D = alpha*acc + beta*C, predicated element stores
    EPI_SWAP = 2,          // same, accumulator holds D^T (swapped operands)
    EPI_PARTIAL = 3,       // fp32 partial sums of one K slice -> workspace
    EPI_PARTIAL_SWAP = 4,  // same, accumulator holds D^T
    EPI_TMA_C = 5,         // D = alpha*acc + beta*C, C loaded and D stored by TMA (aligned C and D)
    EPI_TMA_A16 = 6,       // EPI_TMA with an fp16 accumulator
    EPI_GENERIC_A16 = 7,   // EPI_GENERIC with an fp16 accumulator
    EPI_TMA_CG = 8,        // EPI_TMA_C with C read straight from global memory at any 2-byte alignment
    EPI_VEC = 9,           // D (and C) at any 2-byte alignment through aligned 16-byte words, per row
};

// Variant flag (or-ed into the epilogue mode of a variant): eight more warps read the
// rows of operands TMA cannot address (K-major, any 2-byte alignment) through the aligned
// 16-byte words that cover them and write the swizzled shared-memory image themselves.
constexpr int EPI_RL = 0x100;
// Variant flag: the two CTAs of a cluster take the two halves of K of the same swapped
// tile; the second CTA's fp32 partial sum goes into the first CTA's shared memory
// (distributed shared memory), which adds it and writes D -- split-K in one launch,
// with no scratch in global memory.
constexpr int EPI_CK = 0x200;
// Variant flag (wide pair tiles, D = alpha*acc by TMA stores): two epilogue warpgroups, one
// per part of the accumulator (the two MMAs' columns).  Each warp reads its whole part of
// its 32 rows into registers as fp16 and hands the part back to the MMA before it stores
// anything, so the next tile's MMAs wait only for tensor-memory reads, not for stores.
constexpr int EPI_H2 = 0x400;
// Variant flag (D = alpha*acc by TMA stores): four staging buffers per epilogue warp instead of
// two, for tiles of one k-block, whose time goes to storing D (the attention score Q K^T).
constexpr int EPI_SQ = 0x1000;

#ifdef __CUDACC__
#define GTN_HD __host__ __device__
#else
#define GTN_HD
#endif

// Epilogue mode of a variant without its flags.
GTN_HD constexpr int epi_mode(int epi) { return epi & 0xff; }
// Epilogue mode without the accumulator precision; true when the accumulator is fp16.
GTN_HD constexpr int epi_base(int epi) {
    return epi_mode(epi) == EPI_TMA_A16 ? EPI_TMA : epi_mode(epi) == EPI_GENERIC_A16 ? EPI_GENERIC : epi_mode(epi);
}
GTN_HD constexpr bool epi_acc16(int epi) { return epi_mode(epi) == EPI_TMA_A16 || epi_mode(epi) == EPI_GENERIC_A16; }
GTN_HD constexpr bool epi_rl(int epi) { return (epi & EPI_RL) != 0; }
GTN_HD constexpr bool epi_ck(int epi) { return (epi & EPI_CK) != 0; }
GTN_HD constexpr bool epi_h2(int epi) { return (epi & EPI_H2) != 0; }
GTN_HD constexpr bool epi_sq(int epi) { return (epi & EPI_SQ) != 0; }

struct KParams {
    // Tensor-core view: the MMA's A operand has rows_a rows, its B operand rows_b rows.
    int32_t rows_a, rows_b, K, batch;
    int32_t tiles_m, tiles_n;  // tiles of (128*PAIR) x BN in that view
    int32_t splits;            // K slices per tile
    int32_t kb_total;          // number of 64-wide k-blocks, ceil(K/64)
    int32_t group_m;           // rasterisation group size along the tile rows
    int32_t serp;              // 1: odd waves of data-parallel units walk K backwards (serpentine)
    int32_t zA, zB, zC, zD;    // batch coordinate multipliers (0 = operand not batched)
    int32_t a_mn, b_mn;        // 1: the MMA operand is stored MN-major (rows contiguous), 0: K-major
    int64_t num_units;         // data-parallel units: whole tiles, or (tile, K slice) pairs when splits > 1
    // Problem view, for the epilogue.
    int32_t M, N;
    float alpha, beta;
    void* D;
    int64_t ldd, strideD;
    const void* C;
    int64_t ldc, strideC;
    float* W;  // split-K partials, [batch][splits][M][N] fp32
    // Stream-K: after its data-parallel units, CTA group g (of G) runs k-block
    // iterations [g*I/G, (g+1)*I/G) of the I = sk_tiles * kb_total iterations of the
    // tiles that follow the data-parallel ones.  A tile cut between groups is
    // finished by whichever group contributes last (arrival counter), which sums
    // every group's fp32 partial in group order.
    int64_t sk_iters;          // I; 0 = no stream-K phase
    int32_t sk_maxc;           // partial slots per stream-K tile (>= contributors of any tile)
    float* sk_W;               // [sk_tile][sk_maxc][PAIR][128][BN] fp32 partial accumulators
    // [sk_tile][PAIR][4 epilogue warps] arrival words: (sk_epoch << 8) | count.  A word
    // whose tag is not this launch's epoch counts as zero, so the scratch needs no
    // clearing (a stale or arbitrary word matches a 56-bit epoch with probability 2^-56).
    unsigned long long* sk_counters;
    unsigned long long sk_epoch;  // unique per launch, nonzero, < 2^56
    uint32_t* err;
    uint64_t timeout_ns;
    int32_t debug_skip_first_load;  // test hook: CTA 0 never issues its first load
    // 1: launched as a programmatic dependent of the kernel before it (the operand
    // repack), whose output the producer waits for before its first load; everything
    // up to that point (barriers, tensor memory, tensor maps) overlaps that kernel.
    int32_t pdl;
    // Row loader (EPI_RL variants): MMA operand X (0 = A, 1 = B) is read by the loader warps
    // when rl_on[X] is 1 -- row-major, K contiguous, from rl_ptr[X] with leading dimension
    // rl_ld[X] and batch stride rl_stride[X] (elements, 0 = broadcast) -- else by TMA.
    const void* rl_ptr[2];
    int64_t rl_ld[2];
    int64_t rl_stride[2];
    int32_t rl_on[2];
    uint32_t tma_tx;  // bytes TMA brings per stage (both CTAs of a pair), for EPI_RL variants
    // Byte ranges of the problem's A, B, C, D and of the split-K partial sums W, for the
    // checked build's device-side bounds checks (checked.h); unused otherwise.
    Extent ext_a, ext_b, ext_c, ext_d, ext_w;
    // EPI_PARTIAL: 1 when the tmD slot holds a tensor map of W (fp32, [batch * splits][M][N],
    // boxes of 32 rows x 32 columns, 128-byte swizzle), so partials are stored by TMA.
    int32_t w_tma;
};

}  // namespace gtn
