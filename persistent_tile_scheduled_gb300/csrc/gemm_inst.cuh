// Host-side wrappers around one gemm_kernel instantiation.
#pragma once
#include "gemm_kernel.cuh"
#include "gemm_launch.h"

namespace pts {

template <int KIND, int CG, int BN = kTileN, bool FULL = true>
struct Inst {
    // Raise the dynamic shared-memory limit, and ask for the largest shared-
    // memory share of the SM's unified L1/shared storage: without that
    // preference the driver may size the share for one CTA of the narrow tile
    // and leave no room for the second.
    static cudaError_t set_smem(int smem)
    {
        cudaError_t e =
            cudaFuncSetAttribute(gemm_kernel<KIND, CG, BN, FULL>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        return cudaFuncSetAttribute(gemm_kernel<KIND, CG, BN, FULL>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                    static_cast<int>(cudaSharedmemCarveoutMaxShared));
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

    // Resident clusters.  For single CTAs the count is worked out from the
    // SM's resources -- shared memory (with the per-block reservation),
    // registers (whole warps' allocations), threads and TMEM columns -- rather
    // than taken from cudaOccupancyMaxActiveBlocksPerMultiprocessor: on GB300
    // that call reports one block per SM for any kernel that uses tcgen05
    // (even a 4-register kernel that only allocates TMEM), while the hardware
    // runs two of the narrow-tile CTAs on one SM at once (measured: per-tile
    // records of a one-CTA-per-tile launch show two CTAs overlapping in time
    // on every SM, and CLC's first wave is 2 x SMs CTAs).  CTA pairs keep the
    // runtime's cluster count.
    static cudaError_t max_active_clusters(int smem, int *out)
    {
        cudaLaunchConfig_t cfg;
        cudaLaunchAttribute attr[2];
        fill_config(cfg, attr, 2 * CG, smem, nullptr);
        if (CG == 1) {
            int dev = 0, sms = 0, smem_sm = 0, reserved = 0, regs_sm = 0, threads_sm = 0;
            cudaError_t e = cudaGetDevice(&dev);
            if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
            if (e == cudaSuccess) e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
            if (e == cudaSuccess) e = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev);
            if (e == cudaSuccess) e = cudaDeviceGetAttribute(&threads_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev);
            cudaFuncAttributes fa;
            if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, gemm_kernel<KIND, CG, BN, FULL>);
            if (e != cudaSuccess) return e;
            const int by_smem = smem_sm / (smem + static_cast<int>(fa.sharedSizeBytes) + reserved);
            const int regs_warp = (fa.numRegs * 32 + 255) / 256 * 256;   // allocated per warp in units of 256
            const int by_regs = regs_sm / (regs_warp * (kThreads / 32));
            const int by_threads = threads_sm / kThreads;
            const int by_tmem = kTmemCols / (2 * BN);                    // two accumulators of BN columns
            int per_sm = by_smem < by_regs ? by_smem : by_regs;
            per_sm = per_sm < by_threads ? per_sm : by_threads;
            per_sm = per_sm < by_tmem ? per_sm : by_tmem;
            *out = per_sm * sms;
            return cudaSuccess;
        }
        return cudaOccupancyMaxActiveClusters(out, gemm_kernel<KIND, CG, BN, FULL>, &cfg);
    }

    static cudaError_t launch(const CUtensorMap &a, const CUtensorMap *const b[3], const CUtensorMap &c,
                              const GemmParams &p, int grid_ctas, int smem, cudaStream_t stream, bool overlap)
    {
        cudaLaunchConfig_t cfg;
        cudaLaunchAttribute attr[2];
        fill_config(cfg, attr, grid_ctas, smem, stream, overlap);
        return cudaLaunchKernelEx(&cfg, gemm_kernel<KIND, CG, BN, FULL>, a, *b[0], *b[1], *b[2], c, p);
    }

    static KernelOps ops() { return KernelOps{&set_smem, &max_active_clusters, &launch}; }
};

}  // namespace pts
