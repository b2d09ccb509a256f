// Variants whose epilogue writes D with TMA stores (aligned D; with EPI_TMA_C, C is read by TMA too,
// with EPI_TMA_CG straight from global memory at any alignment).
#include "tc_launch.cuh"

namespace gtn {

bool launch_family_tma(const TcVariant& v, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                          const CUtensorMap& tmD, const KParams& p, int64_t max_ctas, cudaStream_t stream, int64_t* grid_out,
                          cudaError_t* err) {
#define GTN_CASE(BN, PAIR, ST, EPI, SK)                                                                    \
    if (v.bn == BN && v.pair == PAIR && v.stages == ST && v.epi == EPI && v.sk == SK) {                             \
        *err = TcLauncher<BN, PAIR, ST, EPI, SK>::launch(tmA, tmB, tmC, tmD, p, max_ctas, stream, grid_out);   \
        return true;                                                                                  \
    }
    GTN_CASE(256, 1, 4, EPI_TMA, 0)
    GTN_CASE(256, 1, 3, EPI_TMA | EPI_SQ, 0)
    GTN_CASE(256, 1, 4, EPI_TMA_C, 0)
    GTN_CASE(256, 1, 4, EPI_TMA_CG, 0)
    GTN_CASE(256, 1, 4, EPI_TMA, 1)
    GTN_CASE(256, 1, 4, EPI_TMA_A16, 0)
    GTN_CASE(256, 1, 4, EPI_TMA_C, 1)
    GTN_CASE(256, 1, 4, EPI_TMA_CG, 1)
    GTN_CASE(256, 2, 6, EPI_TMA, 0)
    GTN_CASE(256, 2, 6, EPI_TMA_C, 0)
    GTN_CASE(256, 2, 6, EPI_TMA_CG, 0)
    GTN_CASE(256, 2, 6, EPI_TMA, 1)
    GTN_CASE(256, 2, 6, EPI_TMA_A16, 0)
    GTN_CASE(256, 2, 6, EPI_TMA_C, 1)
    GTN_CASE(256, 2, 6, EPI_TMA_CG, 1)
    GTN_CASE(128, 1, 6, EPI_TMA, 0)
    GTN_CASE(128, 1, 6, EPI_TMA_C, 0)
    GTN_CASE(128, 1, 6, EPI_TMA_CG, 0)
    GTN_CASE(128, 1, 6, EPI_TMA, 1)
    GTN_CASE(128, 1, 6, EPI_TMA_A16, 0)
    GTN_CASE(128, 1, 6, EPI_TMA_C, 1)
    GTN_CASE(128, 1, 6, EPI_TMA_CG, 1)
    GTN_CASE(128, 2, 8, EPI_TMA, 0)
    GTN_CASE(128, 2, 8, EPI_TMA_C, 0)
    GTN_CASE(128, 2, 8, EPI_TMA_CG, 0)
    GTN_CASE(128, 2, 8, EPI_TMA, 1)
    GTN_CASE(128, 2, 8, EPI_TMA_C, 1)
    GTN_CASE(128, 2, 8, EPI_TMA_CG, 1)
#undef GTN_CASE
    return false;
}

bool capacity_family_tma(const TcVariant& v, int sms, int64_t* cap) {
#define GTN_CASE(BN, PAIR, ST, EPI, SK)                                          \
    if (v.bn == BN && v.pair == PAIR && v.stages == ST && v.epi == EPI && v.sk == SK) {   \
        *cap = TcLauncher<BN, PAIR, ST, EPI, SK>::capacity(sms);                \
        return true;                                                        \
    }
    GTN_CASE(256, 1, 4, EPI_TMA, 0)
    GTN_CASE(256, 1, 3, EPI_TMA | EPI_SQ, 0)
    GTN_CASE(256, 1, 4, EPI_TMA_C, 0)
    GTN_CASE(256, 1, 4, EPI_TMA_CG, 0)
    GTN_CASE(256, 1, 4, EPI_TMA, 1)
    GTN_CASE(256, 1, 4, EPI_TMA_A16, 0)
    GTN_CASE(256, 1, 4, EPI_TMA_C, 1)
    GTN_CASE(256, 1, 4, EPI_TMA_CG, 1)
    GTN_CASE(256, 2, 6, EPI_TMA, 0)
    GTN_CASE(256, 2, 6, EPI_TMA_C, 0)
    GTN_CASE(256, 2, 6, EPI_TMA_CG, 0)
    GTN_CASE(256, 2, 6, EPI_TMA, 1)
    GTN_CASE(256, 2, 6, EPI_TMA_A16, 0)
    GTN_CASE(256, 2, 6, EPI_TMA_C, 1)
    GTN_CASE(256, 2, 6, EPI_TMA_CG, 1)
    GTN_CASE(128, 1, 6, EPI_TMA, 0)
    GTN_CASE(128, 1, 6, EPI_TMA_C, 0)
    GTN_CASE(128, 1, 6, EPI_TMA_CG, 0)
    GTN_CASE(128, 1, 6, EPI_TMA, 1)
    GTN_CASE(128, 1, 6, EPI_TMA_A16, 0)
    GTN_CASE(128, 1, 6, EPI_TMA_C, 1)
    GTN_CASE(128, 1, 6, EPI_TMA_CG, 1)
    GTN_CASE(128, 2, 8, EPI_TMA, 0)
    GTN_CASE(128, 2, 8, EPI_TMA_C, 0)
    GTN_CASE(128, 2, 8, EPI_TMA_CG, 0)
    GTN_CASE(128, 2, 8, EPI_TMA, 1)
    GTN_CASE(128, 2, 8, EPI_TMA_C, 1)
    GTN_CASE(128, 2, 8, EPI_TMA_CG, 1)
#undef GTN_CASE
    return false;
}

}  // namespace gtn
