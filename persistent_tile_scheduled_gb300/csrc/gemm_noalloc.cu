// gemm_run_noalloc: the GEMM without a handle and without allocating memory.
//
// Some callers cannot allocate device memory when they need a GEMM: runtimes
// that reserve all device memory up front and refuse later allocations, and
// latency-critical loops that cannot accept the implicit synchronisation
// cudaMalloc / cudaFree may perform.  gemm_create allocates a status block, so
// those callers cannot use the handle API.  This entry point keeps the kernel's
// scratch -- the device status block and one record per work item (the
// coverage counters) -- in a file-scope __device__ array instead.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/pts_gemm.h"
#include "gemm_launch.h"
#include "gemm_plan.h"

namespace {

constexpr size_t kStatusBytes = 256;   // 4 status words, padded to the array's alignment
constexpr size_t kScratchBytes =
    kStatusBytes + static_cast<size_t>(GEMM_NOALLOC_MAX_WORK_ITEMS) * sizeof(pts::TileRecord);

}  // namespace

// Scratch of every call: [0, 256) status block, then one record per work item.
// Every GPU that loads this library holds it (kScratchBytes = 832.25 KiB)
// until the process exits.  Calls share it; calls that overlap on the GPU race.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

namespace {

constexpr int kMaxDevices = 64;

struct DeviceSetup {
    bool ready = false;                // set only once the whole set-up has succeeded
    unsigned char *scratch = nullptr;  // device address of g_noalloc_scratch on this device
    int max_smem = 0;
    int stages[2] = {0, 0};
    int smem[2] = {0, 0};
    int clusters[3][2] = {};
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
};

std::mutex g_setup_mutex;
DeviceSetup g_setup[kMaxDevices];

// Once per device, with that device current: scratch address, kernel
// attributes, resident-cluster counts and the tensor-map encoder.  A set-up
// that fails is not remembered: the error goes to this call's caller and the
// next call on the device tries again from the start.
gemm_status_t setup_device(int dev, const DeviceSetup **out)
{
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    DeviceSetup &s = g_setup[dev];
    *out = &s;
    if (s.ready) return GEMM_OK;
    DeviceSetup n;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess
        || cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess
        || cudaDeviceGetAttribute(&n.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return GEMM_ERR_UNSUPPORTED;
    void *addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) {
        (void)cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    n.scratch = static_cast<unsigned char *>(addr);
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess
        || q != cudaDriverEntryPointSuccess || fn == nullptr) {
        (void)cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    n.encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    for (int cg = 1; cg <= 2; ++cg) {
        int st = pts::kMaxStages;
        while (st > 2 && pts::smem_bytes(cg, st) > n.max_smem) --st;
        n.stages[cg - 1] = st;
        n.smem[cg - 1] = pts::smem_bytes(cg, st);
        for (int kind = 0; kind < 3; ++kind) {
            pts::KernelOps ops = cg == 2 ? pts::kernel_ops_cg2(kind, true) : pts::kernel_ops_cg1(kind, true);
            if (ops.set_smem(n.max_smem) != cudaSuccess
                || ops.max_active_clusters(n.smem[cg - 1], &n.clusters[kind][cg - 1]) != cudaSuccess
                || n.clusters[kind][cg - 1] < 1) {
                (void)cudaGetLastError();
                return GEMM_ERR_CUDA;
            }
        }
    }
    n.ready = true;
    s = n;
    return GEMM_OK;
}

bool encode_2d(const DeviceSetup *s, CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols,
               int dtype, uint32_t box_rows, uint32_t box_cols)
{
    CUtensorMapDataType t = dtype == GEMM_F16    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                            : dtype == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const uint64_t es = dtype == GEMM_E4M3 ? 1 : 2;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * es};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return s->encode(map, t, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

gemm_status_t fail(cudaError_t e)
{
    (void)cudaGetLastError();
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

}  // namespace

extern "C" gemm_status_t gemm_run_noalloc(int64_t M, int64_t N, int64_t K, const void *A, const void *B, void *C,
                                          gemm_dtype_t dtype, gemm_sched_t sched, float scale_a, float scale_b,
                                          int cta_group, void *stream, int *device_status)
{
    if (device_status) *device_status = 0;
    if (dtype < GEMM_F16 || dtype > GEMM_E4M3 || sched < GEMM_SCHED_NONPERSISTENT || sched > GEMM_SCHED_CLC)
        return GEMM_ERR_INVALID_ARG;
    if (cta_group != 1 && cta_group != 2) return GEMM_ERR_INVALID_ARG;
    const int64_t lim = (int64_t(1) << 31) - 1;
    const int64_t es = dtype == GEMM_E4M3 ? 1 : 2;
    if (M < 0 || N < 0 || K < 0 || M > lim || N > lim || K > lim) return GEMM_ERR_INVALID_ARG;
    if ((K * es) % 16 != 0 || (N * 2) % 16 != 0) return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return GEMM_OK;
    if (!C || reinterpret_cast<uintptr_t>(C) % 16) return GEMM_ERR_INVALID_ARG;
    if (K == 0) return fail(pts::launch_zero_fill(C, M * N * 2, static_cast<cudaStream_t>(stream)));
    if (!A || !B || reinterpret_cast<uintptr_t>(A) % 16 || reinterpret_cast<uintptr_t>(B) % 16)
        return GEMM_ERR_INVALID_ARG;
    float out_scale = 1.0f;
    if (dtype == GEMM_E4M3) {
        if (!(scale_a > 0.0f) || !(scale_b > 0.0f) || !std::isfinite(scale_a) || !std::isfinite(scale_b))
            return GEMM_ERR_INVALID_ARG;
        out_scale = 1.0f / (scale_a * scale_b);
        if (!std::isfinite(out_scale)) return GEMM_ERR_INVALID_ARG;
    }
    const int64_t tile_m = int64_t(pts::kRowsPerCta) * cta_group;
    const int64_t tiles_m = (M + tile_m - 1) / tile_m;
    const int64_t tiles_n = (N + pts::kTileN - 1) / pts::kTileN;
    const int64_t tiles = tiles_m * tiles_n;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return fail(cudaErrorInvalidDevice);
    const DeviceSetup *s = nullptr;
    const gemm_status_t setup = setup_device(dev, &s);
    if (setup != GEMM_OK) return setup;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int ci = cta_group - 1;
    const int64_t resident = s->clusters[dtype][ci];
    const int split = pts::choose_split(tiles, resident);   // column slices below one wave
    // column halves of a partial last wave (persistent schedulers; never the
    // stream-K share, whose fixup workspace a static array could not hold)
    const uint32_t kelems = dtype == GEMM_E4M3 ? 128u : 64u;
    const int64_t num_kb = (K + kelems - 1) / kelems;
    int64_t tail = 0;
    if (split == 1) (void)pts::choose_last_wave(tiles, resident, num_kb, true, -1, int(sched), tail);
    const int64_t work = tiles * split + tail;
    if (work > GEMM_NOALLOC_MAX_WORK_ITEMS) return GEMM_ERR_INVALID_ARG;   // one scratch record per item

    // status words and the records of this problem's work items must start at zero
    const size_t used = kStatusBytes + static_cast<size_t>(work) * sizeof(pts::TileRecord);
    if (cudaMemsetAsync(s->scratch, 0, used, st) != cudaSuccess) return fail(cudaErrorInvalidValue);

    CUtensorMap ma, mb, mb_slice, mc;
    const uint32_t brows = uint32_t(pts::kTileN / cta_group);
    if (!encode_2d(s, &ma, A, uint64_t(M), uint64_t(K), dtype, pts::kRowsPerCta, kelems)
        || !encode_2d(s, &mb, B, uint64_t(N), uint64_t(K), dtype, brows, kelems)
        || !encode_2d(s, &mb_slice, B, uint64_t(N), uint64_t(K), dtype, brows / uint32_t(tail > 0 ? 2 : split),
                      kelems)
        || !encode_2d(s, &mc, C, uint64_t(M), uint64_t(N), dtype == GEMM_F16 ? GEMM_F16 : GEMM_BF16,
                      pts::kEpiRowsPerWarp, pts::kEpiChunkCols))
        return GEMM_ERR_CUDA;
    const CUtensorMap *mbs[3] = {&mb, (split == 2 || tail > 0) ? &mb_slice : &mb, split == 4 ? &mb_slice : &mb};

    pts::GemmParams p{};
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.num_kb = static_cast<int32_t>(num_kb);
    p.tiles_m = static_cast<int32_t>(tiles_m);
    p.tiles_n = static_cast<int32_t>(tiles_n);
    p.num_tiles = static_cast<int32_t>(tiles);
    p.split = split;
    p.sk_tiles = 0;   // no stream-K share: its fixup workspace would not fit a modest static array
    p.sk_units = 0;
    p.ws_partial = nullptr;
    p.ws_sync = nullptr;
    p.num_units = static_cast<int32_t>(work);
    p.num_work = static_cast<int32_t>(work);
    p.group_m = 8;
    p.sched = static_cast<int32_t>(sched);
    p.stages = s->stages[ci];
    p.prefetch_kb = pts::kDefaultPrefetchKb;
    p.epi_direct = 0;
    p.clc_lead = pts::kDefaultClcLead;
    p.tail_tiles = static_cast<int32_t>(tail);
    p.c_ptr = C;
    p.out_scale = out_scale;
    p.debug_flags = pts::DBG_RECORDS;
    p.fault_arg = 0;
    p.timeout_ns = 1000000000ull;
    p.status = reinterpret_cast<int32_t *>(s->scratch);
    p.records = reinterpret_cast<pts::TileRecord *>(s->scratch + kStatusBytes);

    int64_t clusters = work;
    if (sched == GEMM_SCHED_STATIC && clusters > resident) clusters = resident;
    pts::KernelOps ops = cta_group == 2 ? pts::kernel_ops_cg2(dtype, true)   // full: it writes coverage records
                                        : pts::kernel_ops_cg1(dtype, true);
    cudaError_t e = ops.launch(ma, mbs, mc, p, static_cast<int>(clusters * cta_group), s->smem[ci], st, true);
    if (e != cudaSuccess) return fail(e);
    if ((e = cudaGetLastError()) != cudaSuccess) return fail(e);
    if (device_status == nullptr) return GEMM_OK;

    // synchronous check: status block, then every tile's visit count (read in
    // fixed-size chunks into stack memory; nothing is allocated)
    if (cudaStreamSynchronize(st) != cudaSuccess) return fail(cudaErrorUnknown);
    int32_t words[4];
    if (cudaMemcpy(words, s->scratch, sizeof(words), cudaMemcpyDeviceToHost) != cudaSuccess)
        return fail(cudaErrorUnknown);
    if (words[0] != 0) {
        *device_status = (words[0] << 24) | ((words[1] & 0xff) << 16) | (words[2] & 0xffff);
        return words[0] == pts::DEV_ERR_TIMEOUT ? GEMM_ERR_TIMEOUT : GEMM_ERR_CUDA;
    }
    pts::TileRecord chunk[128];
    for (int64_t t0 = 0; t0 < work; t0 += 128) {
        const int64_t n = work - t0 < 128 ? work - t0 : 128;
        if (cudaMemcpy(chunk, s->scratch + kStatusBytes + size_t(t0) * sizeof(pts::TileRecord),
                       size_t(n) * sizeof(pts::TileRecord), cudaMemcpyDeviceToHost) != cudaSuccess)
            return fail(cudaErrorUnknown);
        for (int64_t i = 0; i < n; ++i)
            if (chunk[i].visits != static_cast<uint32_t>(cta_group)) return GEMM_ERR_COVERAGE;
    }
    return GEMM_OK;
}
