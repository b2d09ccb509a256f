// Variants with predicated epilogues (alpha/beta, any alignment), split-K partial sums, and the
// row-word epilogue for C and D at any alignment.
#include "tc_launch.cuh"

namespace gtn {

bool launch_family_generic(const TcVariant& v, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                          const CUtensorMap& tmD, const KParams& p, int64_t max_ctas, cudaStream_t stream, int64_t* grid_out,
                          cudaError_t* err) {
#define GTN_CASE(BN, PAIR, ST, EPI, SK)                                                                    \
    if (v.bn == BN && v.pair == PAIR && v.stages == ST && v.epi == EPI && v.sk == SK) {                             \
        *err = TcLauncher<BN, PAIR, ST, EPI, SK>::launch(tmA, tmB, tmC, tmD, p, max_ctas, stream, grid_out);   \
        return true;                                                                                  \
    }
    GTN_CASE(256, 1, 4, EPI_GENERIC, 0)
    GTN_CASE(256, 1, 4, EPI_GENERIC, 1)
    GTN_CASE(256, 1, 4, EPI_GENERIC_A16, 0)
    GTN_CASE(256, 2, 6, EPI_GENERIC, 0)
    GTN_CASE(256, 2, 6, EPI_GENERIC, 1)
    GTN_CASE(256, 2, 6, EPI_GENERIC_A16, 0)
    GTN_CASE(128, 1, 6, EPI_GENERIC, 0)
    GTN_CASE(128, 1, 6, EPI_GENERIC, 1)
    GTN_CASE(128, 1, 6, EPI_GENERIC_A16, 0)
    GTN_CASE(128, 1, 6, EPI_PARTIAL, 0)
    GTN_CASE(256, 1, 4, EPI_VEC, 0)
    GTN_CASE(256, 1, 4, EPI_VEC, 1)
    GTN_CASE(256, 2, 6, EPI_VEC, 0)
    GTN_CASE(256, 2, 6, EPI_VEC, 1)
    GTN_CASE(128, 1, 6, EPI_VEC, 0)
    GTN_CASE(128, 1, 6, EPI_VEC, 1)
    GTN_CASE(128, 2, 8, EPI_VEC, 0)
    GTN_CASE(128, 2, 8, EPI_VEC, 1)
#undef GTN_CASE
    return false;
}

bool capacity_family_generic(const TcVariant& v, int sms, int64_t* cap) {
#define GTN_CASE(BN, PAIR, ST, EPI, SK)                                          \
    if (v.bn == BN && v.pair == PAIR && v.stages == ST && v.epi == EPI && v.sk == SK) {   \
        *cap = TcLauncher<BN, PAIR, ST, EPI, SK>::capacity(sms);                \
        return true;                                                        \
    }
    GTN_CASE(256, 1, 4, EPI_GENERIC, 0)
    GTN_CASE(256, 1, 4, EPI_GENERIC, 1)
    GTN_CASE(256, 1, 4, EPI_GENERIC_A16, 0)
    GTN_CASE(256, 2, 6, EPI_GENERIC, 0)
    GTN_CASE(256, 2, 6, EPI_GENERIC, 1)
    GTN_CASE(256, 2, 6, EPI_GENERIC_A16, 0)
    GTN_CASE(128, 1, 6, EPI_GENERIC, 0)
    GTN_CASE(128, 1, 6, EPI_GENERIC, 1)
    GTN_CASE(128, 1, 6, EPI_GENERIC_A16, 0)
    GTN_CASE(128, 1, 6, EPI_PARTIAL, 0)
    GTN_CASE(256, 1, 4, EPI_VEC, 0)
    GTN_CASE(256, 1, 4, EPI_VEC, 1)
    GTN_CASE(256, 2, 6, EPI_VEC, 0)
    GTN_CASE(256, 2, 6, EPI_VEC, 1)
    GTN_CASE(128, 1, 6, EPI_VEC, 0)
    GTN_CASE(128, 1, 6, EPI_VEC, 1)
    GTN_CASE(128, 2, 8, EPI_VEC, 0)
    GTN_CASE(128, 2, 8, EPI_VEC, 1)
#undef GTN_CASE
    return false;
}

}  // namespace gtn
