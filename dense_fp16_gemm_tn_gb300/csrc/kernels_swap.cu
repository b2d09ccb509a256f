// Variants for small M: operands swapped so the tensor core computes D^T = B . A^T.  The
// EPI_CK ones split each tile's K between the two CTAs of a cluster.
#include "tc_launch.cuh"

namespace gtn {

bool launch_family_swap(const TcVariant& v, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                          const CUtensorMap& tmD, const KParams& p, int64_t max_ctas, cudaStream_t stream, int64_t* grid_out,
                          cudaError_t* err) {
#define GTN_CASE(BN, PAIR, ST, EPI, SK)                                                                    \
    if (v.bn == BN && v.pair == PAIR && v.stages == ST && v.epi == (EPI) && v.sk == SK) {                             \
        *err = TcLauncher<BN, PAIR, ST, EPI, SK>::launch(tmA, tmB, tmC, tmD, p, max_ctas, stream, grid_out);   \
        return true;                                                                                  \
    }
    GTN_CASE(16, 1, 12, EPI_SWAP, 0)
    GTN_CASE(16, 1, 12, EPI_SWAP, 1)
    GTN_CASE(32, 1, 11, EPI_SWAP, 0)
    GTN_CASE(32, 1, 11, EPI_SWAP, 1)
    GTN_CASE(64, 1, 9, EPI_SWAP, 0)
    GTN_CASE(64, 1, 9, EPI_SWAP, 1)
    GTN_CASE(16, 1, 12, EPI_PARTIAL_SWAP, 0)
    GTN_CASE(32, 1, 11, EPI_PARTIAL_SWAP, 0)
    GTN_CASE(64, 1, 9, EPI_PARTIAL_SWAP, 0)
    GTN_CASE(16, 1, 12, EPI_SWAP | EPI_CK, 0)
    GTN_CASE(32, 1, 10, EPI_SWAP | EPI_CK, 0)
    GTN_CASE(64, 1, 8, EPI_SWAP | EPI_CK, 0)
#undef GTN_CASE
    return false;
}

bool capacity_family_swap(const TcVariant& v, int sms, int64_t* cap) {
#define GTN_CASE(BN, PAIR, ST, EPI, SK)                                          \
    if (v.bn == BN && v.pair == PAIR && v.stages == ST && v.epi == (EPI) && v.sk == SK) {   \
        *cap = TcLauncher<BN, PAIR, ST, EPI, SK>::capacity(sms);                \
        return true;                                                        \
    }
    GTN_CASE(16, 1, 12, EPI_SWAP, 0)
    GTN_CASE(16, 1, 12, EPI_SWAP, 1)
    GTN_CASE(32, 1, 11, EPI_SWAP, 0)
    GTN_CASE(32, 1, 11, EPI_SWAP, 1)
    GTN_CASE(64, 1, 9, EPI_SWAP, 0)
    GTN_CASE(64, 1, 9, EPI_SWAP, 1)
    GTN_CASE(16, 1, 12, EPI_PARTIAL_SWAP, 0)
    GTN_CASE(32, 1, 11, EPI_PARTIAL_SWAP, 0)
    GTN_CASE(64, 1, 9, EPI_PARTIAL_SWAP, 0)
    GTN_CASE(16, 1, 12, EPI_SWAP | EPI_CK, 0)
    GTN_CASE(32, 1, 10, EPI_SWAP | EPI_CK, 0)
    GTN_CASE(64, 1, 8, EPI_SWAP | EPI_CK, 0)
#undef GTN_CASE
    return false;
}

}  // namespace gtn
