// Tensor-pipe peak probe (a measurement aid, not a GEMM).
//
// Every SM (single CTAs) or SM pair (cta_group::2) issues back-to-back
// tcgen05.mma of one k-step of the GEMM kernel's tile shape (128 x 256, or
// 256 x 256 per pair) on operands already in shared memory: no loads, no
// stores, no epilogue, so only the tensor pipe limits it.  It measures the
// dense FLOP per SM clock that every "% of peak" figure of the GEMM assumes.
// Declared in pts_gemm.h (gemm_tensor_peak_probe).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <vector>

#include "../../include/pts_gemm.h"
#include "gemm_kernel.cuh"

namespace pts {
namespace {

struct ProbeOut {
    unsigned long long cycles, t0, t1;   // SM cycles; global-timer start and end (ns)
};

constexpr int kProbeThreads = 128;
constexpr int kProbeCols = 256;              // one 256-column fp32 accumulator
constexpr int kProbeSmem = 200 * 1024;       // more than half an SM's shared memory: one CTA per SM

__device__ __forceinline__ long long clock_cycles()
{
    long long c;
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(c));
    return c;
}

// Finite operand values of the input type (magnitude in [1, 2), random sign),
// so that the tensor pipe switches as it does on real data.
template <int KIND>
__device__ __forceinline__ uint32_t operand_word(uint32_t i, uint32_t salt)
{
    uint32_t h = (i * 2654435761u) ^ (salt * 40503u);
    h ^= h >> 15;
    h *= 2246822519u;
    h ^= h >> 13;
    if constexpr (KIND == 2) {   // four e4m3: exponent field 7 (value 1.mmm), sign random
        uint32_t v = 0;
        for (int b = 0; b < 4; ++b) v |= ((0x38u | ((h >> (4 * b)) & 7u) | (((h >> (16 + b)) & 1u) << 7)) << (8 * b));
        return v;
    } else if constexpr (KIND == 1) {   // two bf16 in [1, 2)
        const uint32_t lo = 0x3F80u | (h & 0x7Fu) | (((h >> 7) & 1u) << 15);
        const uint32_t hi = 0x3F80u | ((h >> 8) & 0x7Fu) | (((h >> 15) & 1u) << 15);
        return lo | (hi << 16);
    } else {                            // two fp16 in [1, 2)
        const uint32_t lo = 0x3C00u | (h & 0x3FFu) | (((h >> 10) & 1u) << 15);
        const uint32_t hi = 0x3C00u | ((h >> 11) & 0x3FFu) | (((h >> 21) & 1u) << 15);
        return lo | (hi << 16);
    }
}

template <int KIND, int CG>
__global__ void __launch_bounds__(kProbeThreads, 1)
    peak_probe_kernel(long long mmas, ProbeOut *out, int32_t *status, unsigned long long timeout_ns)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sA = base;                                  // 128 rows x 128 bytes
    const uint32_t sB = sA + kRowsPerCta * kKBlockBytes;       // 256/CG rows x 128 bytes
    const uint32_t bar = sB + (kTileN / CG) * kKBlockBytes;
    const uint32_t tmem_slot = bar + 8;
    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = lane_id();
    const uint32_t rank = (CG == 2) ? cluster_ctarank() : 0u;

    const uint32_t words = static_cast<uint32_t>((kRowsPerCta + kTileN / CG) * kKBlockBytes / 4);
    for (uint32_t i = threadIdx.x; i < words; i += blockDim.x)
        asm volatile("st.shared.u32 [%0], %1;" ::"r"(sA + 4 * i), "r"(operand_word<KIND>(i, blockIdx.x)) : "memory");
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc<CG>(tmem_slot, kProbeCols);
        tmem_relinquish<CG>();
    }
    fence_proxy_async_smem();   // the operands' generic stores before the MMAs read them
    tc_fence_before();
    __syncthreads();
    if constexpr (CG == 2) cluster_sync();
    tc_fence_after();
    uint32_t tmem;
    asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(tmem) : "r"(tmem_slot) : "memory");

    if (warp == 0) {
        const uint32_t one = lane == 0 ? 1u : 0u;
        const bool issuer = CG == 1 || rank == 0;
        long long c0 = clock_cycles();
        const uint64_t t0 = globaltimer_ns();
        if (issuer) {
            const uint32_t idesc = make_idesc<KIND, CG>(kTileN);
            const uint64_t ad = smem_desc_sw128(sA), bd = smem_desc_sw128(sB);
            for (long long m = 0; m < mmas; ++m) {
                const uint64_t k = static_cast<uint64_t>(2 * (m & 3));   // 32 bytes of K per instruction
                umma<KIND, CG>(one, tmem, ad + k, bd + k, idesc, m > 0 ? 1u : 0u);
            }
            umma_commit<CG>(one, bar, 0x3);
        }
        // both CTAs of a pair see the (multicast) completion before they go on
        bool done = false;
        while (!done) {
            done = mbar_try_wait(bar, 0);
            if (!done && globaltimer_ns() - t0 > timeout_ns) break;
        }
        done = __all_sync(0xffffffffu, done);
        const long long c1 = clock_cycles();
        const uint64_t t1 = globaltimer_ns();
        if (lane == 0) {
            if (!done) atomicExch(status, 1);
            if (issuer) {
                out[blockIdx.x / CG].cycles = static_cast<unsigned long long>(c1 - c0);
                out[blockIdx.x / CG].t0 = t0;
                out[blockIdx.x / CG].t1 = t1;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (CG == 2) cluster_sync();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc<CG>(tmem, kProbeCols);
    }
}

template <int KIND, int CG>
cudaError_t launch_probe(int units, long long mmas, ProbeOut *out, int32_t *status, unsigned long long timeout_ns)
{
    cudaError_t e = cudaFuncSetAttribute(peak_probe_kernel<KIND, CG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kProbeSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(static_cast<unsigned>(units * CG), 1, 1);
    cfg.blockDim = dim3(kProbeThreads, 1, 1);
    cfg.dynamicSmemBytes = kProbeSmem;
    cfg.stream = nullptr;
    if (CG == 2) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, peak_probe_kernel<KIND, CG>, mmas, out, status, timeout_ns);
}

}  // namespace
}  // namespace pts

extern "C" gemm_status_t gemm_tensor_peak_probe(int device, gemm_dtype_t dtype, int cta_group, int64_t mmas,
                                                double *flop_per_clk_per_sm, double *tflops, double *sm_ghz)
{
    using namespace pts;
    if (dtype < GEMM_F16 || dtype > GEMM_E4M3 || (cta_group != 1 && cta_group != 2) || mmas < 1
        || mmas > (int64_t(1) << 20) || flop_per_clk_per_sm == nullptr || tflops == nullptr || sm_ghz == nullptr)
        return GEMM_ERR_INVALID_ARG;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) {
        (void)cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (cudaSetDevice(device) != cudaSuccess) return GEMM_ERR_CUDA;
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (major != 10 || minor != 3) return GEMM_ERR_UNSUPPORTED;
    const int units = sms / cta_group;   // one CTA per SM (its shared memory allows no second)
    ProbeOut *d_out = nullptr;
    int32_t *d_status = nullptr;
    if (cudaMalloc(&d_out, sizeof(ProbeOut) * units) != cudaSuccess || cudaMalloc(&d_status, sizeof(int32_t)) != cudaSuccess
        || cudaMemset(d_out, 0, sizeof(ProbeOut) * units) != cudaSuccess
        || cudaMemset(d_status, 0, sizeof(int32_t)) != cudaSuccess) {
        cudaFree(d_out);
        cudaFree(d_status);
        (void)cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    const unsigned long long timeout_ns = 2000000000ull;
    cudaError_t e;
    const int kind = static_cast<int>(dtype);
    if (cta_group == 1)
        e = kind == 0 ? launch_probe<0, 1>(units, mmas, d_out, d_status, timeout_ns)
            : kind == 1 ? launch_probe<1, 1>(units, mmas, d_out, d_status, timeout_ns)
                        : launch_probe<2, 1>(units, mmas, d_out, d_status, timeout_ns);
    else
        e = kind == 0 ? launch_probe<0, 2>(units, mmas, d_out, d_status, timeout_ns)
            : kind == 1 ? launch_probe<1, 2>(units, mmas, d_out, d_status, timeout_ns)
                        : launch_probe<2, 2>(units, mmas, d_out, d_status, timeout_ns);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    std::vector<ProbeOut> h(static_cast<size_t>(units));
    int32_t st = 0;
    if (e == cudaSuccess) e = cudaMemcpy(h.data(), d_out, sizeof(ProbeOut) * units, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(&st, d_status, sizeof(st), cudaMemcpyDeviceToHost);
    cudaFree(d_out);
    cudaFree(d_status);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (st != 0) return GEMM_ERR_TIMEOUT;
    // per SM: the MMA work of one instruction is 2 * (128 * CG) * 256 * K flop
    // on CG SMs (K = 16 for fp16/bf16, 32 for e4m3)
    const double k_per_instr = dtype == GEMM_E4M3 ? 32.0 : 16.0;
    const double flop_per_sm = 2.0 * kRowsPerCta * kTileN * k_per_instr * static_cast<double>(mmas);
    std::vector<double> per_clk, ghz;
    unsigned long long first = ~0ull, last = 0;
    for (const ProbeOut &o : h) {
        if (o.cycles == 0 || o.t1 <= o.t0) return GEMM_ERR_CUDA;
        per_clk.push_back(flop_per_sm / static_cast<double>(o.cycles));
        ghz.push_back(static_cast<double>(o.cycles) / static_cast<double>(o.t1 - o.t0));
        first = std::min(first, o.t0);
        last = std::max(last, o.t1);
    }
    std::sort(per_clk.begin(), per_clk.end());
    std::sort(ghz.begin(), ghz.end());
    *flop_per_clk_per_sm = per_clk[per_clk.size() / 2];
    *sm_ghz = ghz[ghz.size() / 2];
    // all SMs' work over the span from the first start to the last end
    *tflops = flop_per_sm * units * cta_group / (static_cast<double>(last - first) * 1e-9) / 1e12;
    return GEMM_OK;
}
