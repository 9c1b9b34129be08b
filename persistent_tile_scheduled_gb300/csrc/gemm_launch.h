// Launch entry points of the kernel instantiations (one translation unit per
// cta_group, compiled in parallel).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_params.h"

namespace pts {

struct KernelOps {
    // Raise the kernel's dynamic shared-memory limit to `smem` bytes.
    cudaError_t (*set_smem)(int smem);
    // Resident clusters the device can hold at once for this kernel.
    cudaError_t (*max_active_clusters)(int smem, int *out);
    // b[0..2]: B maps with boxes of 256/CG, 128/CG and 64/CG rows
    cudaError_t (*launch)(const CUtensorMap &a, const CUtensorMap *const b[3], const CUtensorMap &c,
                          const GemmParams &p, int grid_ctas, int smem, cudaStream_t stream, bool overlap);
};

// kind: 0 fp16, 1 bf16, 2 e4m3.  full: the kernel with every feature (grouped
// launches, debug records, the direct-store epilogue, L2 prefetch, test
// hooks); else the common launch's kernel, with those compiled out.
KernelOps kernel_ops_cg1(int kind, bool full);
KernelOps kernel_ops_cg2(int kind, bool full);
// the narrow tile: 128 x 128 per CTA, single CTAs, two per SM
KernelOps kernel_ops_narrow(int kind, bool full);
// the narrow tile as CTA pairs: 256 x 128 per pair, one CTA per SM
KernelOps kernel_ops_narrow_cg2(int kind, bool full);
cudaError_t launch_zero_fill(void *c, long long bytes, cudaStream_t stream);

}  // namespace pts
