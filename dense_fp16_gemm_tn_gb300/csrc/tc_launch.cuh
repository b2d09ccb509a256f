// Launch helper for one instantiation of the tensor-core GEMM kernel.
#pragma once

#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "tc_gemm.cuh"

namespace gtn {

template <int BN, int PAIR, int STAGES, int EPI, bool SK>
struct TcLauncher {
    using Cfg = TileCfg<BN, PAIR, STAGES, EPI>;

    // Opt in to the large dynamic shared memory once per device.
    static cudaError_t prepare() {
        static std::mutex mu;
        static bool done[64] = {};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        std::lock_guard<std::mutex> lock(mu);
        if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
        e = cudaFuncSetAttribute(gemm_tn_tc_kernel<BN, PAIR, STAGES, EPI, SK>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        if constexpr (Cfg::SETMAXNREG) {
            // The warpgroups' register shares (setmaxnreg) add up to exactly MAX_REGS per
            // thread; a kernel built with any other count could leave an increase waiting
            // for registers that never come free, so it is refused.
            cudaFuncAttributes fa;
            e = cudaFuncGetAttributes(&fa, gemm_tn_tc_kernel<BN, PAIR, STAGES, EPI, SK>);
            if (e != cudaSuccess) return e;
            if (fa.numRegs != Cfg::MAX_REGS || fa.maxThreadsPerBlock < Cfg::THREADS) return cudaErrorInvalidConfiguration;
        }
        if (dev >= 0 && dev < 64) done[dev] = true;
        return cudaSuccess;
    }

    static int64_t capacity(int sms) {
        if (prepare() != cudaSuccess) return 0;
        if constexpr (Cfg::CLUSTER == 1) {
            return sms;  // one CTA per SM (shared memory and tensor memory both forbid two)
        } else {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1), 1, 1);
            cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
            cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, gemm_tn_tc_kernel<BN, PAIR, STAGES, EPI, SK>, &cfg) !=
                    cudaSuccess ||
                clusters <= 0) {
                cudaGetLastError();
                return sms & ~1;
            }
            return 2 * static_cast<int64_t>(clusters);
        }
    }

    static cudaError_t launch(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                              const CUtensorMap& tmD, const KParams& p, int64_t max_ctas, cudaStream_t stream,
                              int64_t* grid_out) {
        cudaError_t e = prepare();
        if (e != cudaSuccess) return e;
        // Data-parallel only: no more CTAs than units.  With a stream-K phase every
        // group takes part, so the caller's grid is used as it is.
        constexpr int CL = Cfg::CLUSTER;
        const int64_t units_ctas = p.num_units * CL;
        int64_t grid = (p.sk_iters > 0 || max_ctas < units_ctas) ? max_ctas : units_ctas;
        grid = (grid / CL) * CL;
        if (grid < CL) grid = CL;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[2];
        unsigned na = 0;
        cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
        cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
        cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
        cfg.stream = stream;
        if constexpr (CL == 2) {
            attr[na].id = cudaLaunchAttributeClusterDimension;
            attr[na].val.clusterDim.x = 2;
            attr[na].val.clusterDim.y = 1;
            attr[na].val.clusterDim.z = 1;
            ++na;
        }
        if (p.pdl) {
            attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[na].val.programmaticStreamSerializationAllowed = 1;
            ++na;
        }
        if (na > 0) {
            cfg.attrs = attr;
            cfg.numAttrs = na;
        }
        if (grid_out) *grid_out = grid;
        return cudaLaunchKernelEx(&cfg, gemm_tn_tc_kernel<BN, PAIR, STAGES, EPI, SK>, tmA, tmB, tmC, tmD, p);
    }
};

}  // namespace gtn
