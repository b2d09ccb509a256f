// Variants with the row loader (EPI_RL): operands whose rows TMA cannot address (a base,
// leading dimension or batch stride that is not a multiple of 16 bytes) are read by eight
// loader warps straight from their own rows, so no repacked copy of A or B is made.
// CTA-pair 256 x 256 tiles and single-CTA 128 x 128 tiles, with every whole-tile epilogue.
#include "tc_launch.cuh"

namespace gtn {

#define GTN_RL_VARIANTS(X)                      \
    X(256, 2, 6, EPI_VEC | EPI_RL, 0)           \
    X(256, 2, 6, EPI_TMA | EPI_RL, 0)           \
    X(256, 2, 6, EPI_TMA_C | EPI_RL, 0)         \
    X(256, 2, 6, EPI_TMA_CG | EPI_RL, 0)        \
    X(128, 1, 6, EPI_VEC | EPI_RL, 0)           \
    X(128, 1, 6, EPI_TMA | EPI_RL, 0)           \
    X(128, 1, 6, EPI_TMA_C | EPI_RL, 0)         \
    X(128, 1, 6, EPI_TMA_CG | EPI_RL, 0)

bool launch_family_rowload(const TcVariant& v, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                           const CUtensorMap& tmD, const KParams& p, int64_t max_ctas, cudaStream_t stream,
                           int64_t* grid_out, cudaError_t* err) {
#define GTN_CASE(BN, PAIR, ST, EPI, SK)                                                                  \
    if (v.bn == BN && v.pair == PAIR && v.stages == ST && v.epi == (EPI) && v.sk == SK) {                \
        *err = TcLauncher<BN, PAIR, ST, EPI, SK>::launch(tmA, tmB, tmC, tmD, p, max_ctas, stream, grid_out); \
        return true;                                                                                     \
    }
    GTN_RL_VARIANTS(GTN_CASE)
#undef GTN_CASE
    return false;
}

bool capacity_family_rowload(const TcVariant& v, int sms, int64_t* cap) {
#define GTN_CASE(BN, PAIR, ST, EPI, SK)                                                \
    if (v.bn == BN && v.pair == PAIR && v.stages == ST && v.epi == (EPI) && v.sk == SK) { \
        *cap = TcLauncher<BN, PAIR, ST, EPI, SK>::capacity(sms);                       \
        return true;                                                                   \
    }
    GTN_RL_VARIANTS(GTN_CASE)
#undef GTN_CASE
    return false;
}

}  // namespace gtn
