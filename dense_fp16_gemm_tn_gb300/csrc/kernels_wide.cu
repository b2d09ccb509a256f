// Variants with 256 x 512 CTA-pair tiles (two N=256 MMAs per K step, one 512-column
// accumulator) and TMA-store epilogues.  Per k-block each CTA loads 128 rows of A and
// 256 rows of B for twice the MMA work of a 256 x 256 pair tile, which keeps operand
// delivery well inside the tensor pipe's time.  The 256 x 432 tile (MMAs of N = 256 and
// 176, the same boxes) is for problems whose waves of 512-column tiles come out short.
#include "tc_launch.cuh"

namespace gtn {

#define GTN_WIDE_VARIANTS(X)        \
    X(512, 2, 4, EPI_TMA, 0)        \
    X(512, 2, 4, EPI_TMA, 1)        \
    X(512, 2, 4, EPI_TMA_C, 0)      \
    X(512, 2, 4, EPI_TMA_C, 1)      \
    X(512, 2, 4, EPI_TMA_CG, 0)     \
    X(512, 2, 4, EPI_TMA_CG, 1)     \
    X(432, 2, 4, EPI_TMA, 0)        \
    X(512, 2, 4, EPI_TMA | EPI_H2, 0)

bool launch_family_wide(const TcVariant& v, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                        const CUtensorMap& tmD, const KParams& p, int64_t max_ctas, cudaStream_t stream,
                        int64_t* grid_out, cudaError_t* err) {
#define GTN_CASE(BN, PAIR, ST, EPI, SK)                                                                  \
    if (v.bn == BN && v.pair == PAIR && v.stages == ST && v.epi == EPI && v.sk == SK) {                  \
        *err = TcLauncher<BN, PAIR, ST, EPI, SK>::launch(tmA, tmB, tmC, tmD, p, max_ctas, stream, grid_out); \
        return true;                                                                                     \
    }
    GTN_WIDE_VARIANTS(GTN_CASE)
#undef GTN_CASE
    return false;
}

bool capacity_family_wide(const TcVariant& v, int sms, int64_t* cap) {
#define GTN_CASE(BN, PAIR, ST, EPI, SK)                                                 \
    if (v.bn == BN && v.pair == PAIR && v.stages == ST && v.epi == EPI && v.sk == SK) { \
        *cap = TcLauncher<BN, PAIR, ST, EPI, SK>::capacity(sms);                        \
        return true;                                                                    \
    }
    GTN_WIDE_VARIANTS(GTN_CASE)
#undef GTN_CASE
    return false;
}

}  // namespace gtn
