// Table of the compiled tensor-core kernel variants and dispatch to the
// translation unit that holds each one.
#include "internal.h"

namespace gtn {

bool launch_family_tma(const TcVariant&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const KParams&,
                       int64_t, cudaStream_t, int64_t*, cudaError_t*);
bool launch_family_generic(const TcVariant&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                           const KParams&, int64_t, cudaStream_t, int64_t*, cudaError_t*);
bool launch_family_swap(const TcVariant&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const KParams&,
                        int64_t, cudaStream_t, int64_t*, cudaError_t*);
bool launch_family_wide(const TcVariant&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                        const KParams&, int64_t, cudaStream_t, int64_t*, cudaError_t*);
bool launch_family_rowload(const TcVariant&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                           const CUtensorMap&, const KParams&, int64_t, cudaStream_t, int64_t*, cudaError_t*);
bool capacity_family_tma(const TcVariant&, int, int64_t*);
bool capacity_family_rowload(const TcVariant&, int, int64_t*);
bool capacity_family_wide(const TcVariant&, int, int64_t*);
bool capacity_family_generic(const TcVariant&, int, int64_t*);
bool capacity_family_swap(const TcVariant&, int, int64_t*);

static const TcVariant kVariants[] = {
    {256, 1, 4, EPI_TMA, 0, 0},
    {256, 1, 3, EPI_TMA | EPI_SQ, 0, 0},
    {256, 1, 4, EPI_TMA_C, 0, 0},
    {256, 1, 4, EPI_TMA_CG, 0, 0},
    {256, 1, 4, EPI_TMA, 1, 0},
    {256, 1, 4, EPI_TMA_A16, 0, 0},
    {256, 1, 4, EPI_TMA_C, 1, 0},
    {256, 1, 4, EPI_TMA_CG, 1, 0},
    {256, 2, 6, EPI_TMA, 0, 0},
    {256, 2, 6, EPI_TMA_C, 0, 0},
    {256, 2, 6, EPI_TMA_CG, 0, 0},
    {256, 2, 6, EPI_TMA, 1, 0},
    {256, 2, 6, EPI_TMA_A16, 0, 0},
    {256, 2, 6, EPI_TMA_C, 1, 0},
    {256, 2, 6, EPI_TMA_CG, 1, 0},
    {128, 1, 6, EPI_TMA, 0, 0},
    {128, 1, 6, EPI_TMA_C, 0, 0},
    {128, 1, 6, EPI_TMA_CG, 0, 0},
    {128, 1, 6, EPI_TMA, 1, 0},
    {128, 1, 6, EPI_TMA_A16, 0, 0},
    {128, 1, 6, EPI_TMA_C, 1, 0},
    {128, 1, 6, EPI_TMA_CG, 1, 0},
    {128, 2, 8, EPI_TMA, 0, 0},
    {128, 2, 8, EPI_TMA_C, 0, 0},
    {128, 2, 8, EPI_TMA_CG, 0, 0},
    {128, 2, 8, EPI_TMA, 1, 0},
    {128, 2, 8, EPI_TMA_C, 1, 0},
    {128, 2, 8, EPI_TMA_CG, 1, 0},
    {256, 1, 4, EPI_GENERIC, 0, 0},
    {256, 1, 4, EPI_GENERIC, 1, 0},
    {256, 1, 4, EPI_GENERIC_A16, 0, 0},
    {256, 2, 6, EPI_GENERIC, 0, 0},
    {256, 2, 6, EPI_GENERIC, 1, 0},
    {256, 2, 6, EPI_GENERIC_A16, 0, 0},
    {128, 1, 6, EPI_GENERIC, 0, 0},
    {128, 1, 6, EPI_GENERIC, 1, 0},
    {128, 1, 6, EPI_GENERIC_A16, 0, 0},
    {128, 1, 6, EPI_PARTIAL, 0, 0},
    {256, 1, 4, EPI_VEC, 0, 0},
    {256, 1, 4, EPI_VEC, 1, 0},
    {256, 2, 6, EPI_VEC, 0, 0},
    {256, 2, 6, EPI_VEC, 1, 0},
    {128, 1, 6, EPI_VEC, 0, 0},
    {128, 1, 6, EPI_VEC, 1, 0},
    {128, 2, 8, EPI_VEC, 0, 0},
    {128, 2, 8, EPI_VEC, 1, 0},
    {16, 1, 12, EPI_SWAP, 0, 0},
    {16, 1, 12, EPI_SWAP, 1, 0},
    {32, 1, 11, EPI_SWAP, 0, 0},
    {32, 1, 11, EPI_SWAP, 1, 0},
    {64, 1, 9, EPI_SWAP, 0, 0},
    {64, 1, 9, EPI_SWAP, 1, 0},
    {512, 2, 4, EPI_TMA, 0, 0},
    {432, 2, 4, EPI_TMA, 0, 0},
    {512, 2, 4, EPI_TMA | EPI_H2, 0, 0},
    {512, 2, 4, EPI_TMA, 1, 0},
    {512, 2, 4, EPI_TMA_C, 0, 0},
    {512, 2, 4, EPI_TMA_C, 1, 0},
    {512, 2, 4, EPI_TMA_CG, 0, 0},
    {512, 2, 4, EPI_TMA_CG, 1, 0},
    {16, 1, 12, EPI_PARTIAL_SWAP, 0, 0},
    {32, 1, 11, EPI_PARTIAL_SWAP, 0, 0},
    {64, 1, 9, EPI_PARTIAL_SWAP, 0, 0},
    {256, 2, 6, EPI_VEC | EPI_RL, 0, 0},
    {256, 2, 6, EPI_TMA | EPI_RL, 0, 0},
    {256, 2, 6, EPI_TMA_C | EPI_RL, 0, 0},
    {256, 2, 6, EPI_TMA_CG | EPI_RL, 0, 0},
    {128, 1, 6, EPI_VEC | EPI_RL, 0, 0},
    {128, 1, 6, EPI_TMA | EPI_RL, 0, 0},
    {128, 1, 6, EPI_TMA_C | EPI_RL, 0, 0},
    {128, 1, 6, EPI_TMA_CG | EPI_RL, 0, 0},
    {16, 1, 12, EPI_SWAP | EPI_CK, 0, 0},
    {32, 1, 10, EPI_SWAP | EPI_CK, 0, 0},
    {64, 1, 8, EPI_SWAP | EPI_CK, 0, 0},
};

static_assert(sizeof(kVariants) / sizeof(kVariants[0]) <= kMaxVariants, "variant table too large");

bool find_tc_variant(int bn, int pair, int epi, int sk, TcVariant* out) {
    const int n = static_cast<int>(sizeof(kVariants) / sizeof(kVariants[0]));
    for (int i = 0; i < n; ++i) {
        const TcVariant& v = kVariants[i];
        if (v.bn == bn && v.pair == pair && v.epi == epi && v.sk == sk) {
            if (out) {
                *out = v;
                out->index = i;
            }
            return true;
        }
    }
    return false;
}

cudaError_t launch_tc_variant(const TcVariant& v, const CUtensorMap& tmA, const CUtensorMap& tmB,
                              const CUtensorMap& tmC, const CUtensorMap& tmD, const KParams& p, int64_t max_ctas,
                              cudaStream_t stream, int64_t* grid_out) {
    cudaError_t e = cudaErrorInvalidValue;
    if (launch_family_tma(v, tmA, tmB, tmC, tmD, p, max_ctas, stream, grid_out, &e)) return e;
    if (launch_family_wide(v, tmA, tmB, tmC, tmD, p, max_ctas, stream, grid_out, &e)) return e;
    if (launch_family_generic(v, tmA, tmB, tmC, tmD, p, max_ctas, stream, grid_out, &e)) return e;
    if (launch_family_swap(v, tmA, tmB, tmC, tmD, p, max_ctas, stream, grid_out, &e)) return e;
    if (launch_family_rowload(v, tmA, tmB, tmC, tmD, p, max_ctas, stream, grid_out, &e)) return e;
    return cudaErrorInvalidValue;
}

int64_t tc_variant_capacity(const TcVariant& v, int sms) {
    int64_t cap = 0;
    if (capacity_family_tma(v, sms, &cap) || capacity_family_wide(v, sms, &cap) || capacity_family_generic(v, sms, &cap) ||
        capacity_family_swap(v, sms, &cap) || capacity_family_rowload(v, sms, &cap))
        return cap;
    return 0;
}

}  // namespace gtn
