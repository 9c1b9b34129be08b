// Host-side wrappers around one gemm_kernel instantiation.
#pragma once
#include "gemm_kernel.cuh"
#include "gemm_launch.h"

namespace pts {

template <int KIND, int CG>
struct Inst {
    static cudaError_t set_smem(int smem)
    {
        return cudaFuncSetAttribute(gemm_kernel<KIND, CG>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    }

    // Launch attributes: a (2,1,1) cluster for CTA pairs, and programmatic
    // stream serialization so that this grid may start while the previous
    // grid in the stream finishes (the kernel waits for it before touching
    // global memory).
    static void fill_config(cudaLaunchConfig_t &cfg, cudaLaunchAttribute *attr, int grid_ctas, int smem,
                            cudaStream_t stream, bool overlap = true)
    {
        cfg = cudaLaunchConfig_t{};
        cfg.gridDim = dim3(static_cast<unsigned>(grid_ctas), 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = static_cast<size_t>(smem);
        cfg.stream = stream;
        cfg.attrs = attr;
        int n = 0;
        if (overlap) {
            attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[n].val.programmaticStreamSerializationAllowed = 1;
            ++n;
        }
        if (CG == 2) {
            attr[n].id = cudaLaunchAttributeClusterDimension;
            attr[n].val.clusterDim.x = 2;
            attr[n].val.clusterDim.y = 1;
            attr[n].val.clusterDim.z = 1;
            ++n;
        }
        cfg.numAttrs = static_cast<unsigned>(n);
    }

    static cudaError_t max_active_clusters(int smem, int *out)
    {
        cudaLaunchConfig_t cfg;
        cudaLaunchAttribute attr[2];
        fill_config(cfg, attr, 2 * CG, smem, nullptr);
        if (CG == 1) {
            int per_sm = 0, dev = 0, sms = 0;
            cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemm_kernel<KIND, CG>,
                                                                          kThreads, static_cast<size_t>(smem));
            if (e != cudaSuccess) return e;
            if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
            if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
            *out = per_sm * sms;
            return cudaSuccess;
        }
        return cudaOccupancyMaxActiveClusters(out, gemm_kernel<KIND, CG>, &cfg);
    }

    static cudaError_t launch(const CUtensorMap &a, const CUtensorMap *const b[3], const CUtensorMap &c,
                              const GemmParams &p, int grid_ctas, int smem, cudaStream_t stream, bool overlap)
    {
        cudaLaunchConfig_t cfg;
        cudaLaunchAttribute attr[2];
        fill_config(cfg, attr, grid_ctas, smem, stream, overlap);
        return cudaLaunchKernelEx(&cfg, gemm_kernel<KIND, CG>, a, *b[0], *b[1], *b[2], c, p);
    }

    static KernelOps ops() { return KernelOps{&set_smem, &max_active_clusters, &launch}; }
};

}  // namespace pts
