// 1-SM instantiations: a 128 x 256 output tile per CTA (tcgen05 cta_group::1).
#include "gemm_inst.cuh"

namespace pts {

// C = 0 for K == 0 (the empty sum): 16-byte stores over M x N 2-byte outputs.
__global__ void zero_fill_kernel(uint4 *c, long long n16)
{
    for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < n16;
         t += static_cast<long long>(gridDim.x) * blockDim.x)
        c[t] = make_uint4(0, 0, 0, 0);
}

KernelOps kernel_ops_cg1(int kind, bool full)
{
    switch (kind) {
    case 0: return full ? Inst<0, 1, kTileN, true>::ops() : Inst<0, 1, kTileN, false>::ops();
    case 1: return full ? Inst<1, 1, kTileN, true>::ops() : Inst<1, 1, kTileN, false>::ops();
    default: return full ? Inst<2, 1, kTileN, true>::ops() : Inst<2, 1, kTileN, false>::ops();
    }
}

cudaError_t launch_zero_fill(void *c, long long bytes, cudaStream_t stream)
{
    const long long n16 = bytes / 16;
    if (n16 == 0) return cudaSuccess;
    long long blocks = (n16 + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    zero_fill_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(static_cast<uint4 *>(c), n16);
    return cudaGetLastError();
}

}  // namespace pts
