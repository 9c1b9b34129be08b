// C ABI of the persistent tile-scheduled GEMM: argument checks, launch shape,
// TMA tensor maps and the device status block.  Declared in pts_gemm.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/pts_gemm.h"
#include "gemm_launch.h"
#include "gemm_plan.h"

namespace {

constexpr int kBatchSlots = 6;   // gemm_run_host_batch staging depth
constexpr int kGroupSlots = 2;   // gemm_run_grouped problem tables in flight
constexpr int kMapCache = 1024;   // direct-mapped; a K sweep's A, B, C maps rarely collide
constexpr unsigned long long kDefaultTimeoutNs = 1000000000ull;   // 1 s per wait

struct MapEntry {
    const void *ptr = nullptr;
    uint64_t rows = 0, cols = 0;
    int dtype = -1;
    uint32_t box_rows = 0, box_cols = 0;
    CUtensorMap map;
};

int elem_bytes(gemm_dtype_t d) { return d == GEMM_E4M3 ? 1 : 2; }

}  // namespace

struct gemm_ctx {
    int device = 0;
    int sm_count = 0;
    int max_smem_optin = 0;
    gemm_opts_t opts{};
    int32_t *d_status = nullptr;              // 4 ints
    pts::TileRecord *d_records = nullptr;
    int64_t records_cap = 0;                  // in work items
    int64_t last_work = 0;
    int last_cta_group = 1;
    int64_t last_sk_tiles = 0, last_sk_units = 0, last_num_kb = 0;   // which record slots are pieces
    void *d_host_bufs = nullptr;              // gemm_run_host staging (A | B | C)
    size_t host_bufs_cap = 0;
    float *d_ws_partial = nullptr;            // stream-K fixup workspace
    size_t ws_partial_cap = 0;                // bytes
    uint32_t *d_ws_sync = nullptr;            // stream-K claim counters / ready flags (zero between launches)
    size_t ws_sync_cap = 0;                   // bytes
    // gemm_run_host_batch: staging slots (A | B | C each), copy streams and events
    void *d_slot[kBatchSlots] = {};
    size_t slot_cap = 0;
    cudaStream_t s_h2d = nullptr, s_d2h[2] = {nullptr, nullptr};   // copy-out alternates between two
                                                                    // streams: one reaches ~146 GB/s of
                                                                    // the ~190 two reach (GB300)
    cudaEvent_t ev_entry = nullptr, ev_in[kBatchSlots] = {}, ev_comp[kBatchSlots] = {}, ev_free[kBatchSlots] = {};
    // gemm_run_grouped: problem tables (GroupDesc[count] then int32 group_start[count + 1]),
    // each as uploaded (pinned host copy) and on the device, and the event after the
    // last launch that read it
    void *tab_host[kGroupSlots] = {};
    void *tab_dev[kGroupSlots] = {};
    size_t tab_cap[kGroupSlots] = {};
    size_t tab_bytes[kGroupSlots] = {};   // bytes of the table the slot holds (0 = none)
    cudaEvent_t ev_tab[kGroupSlots] = {};
    int tab_cur = 0;
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    // per dtype, kernel variant (0: wide tile, single CTAs; 1: wide, pairs; 2: narrow tile,
    // single CTAs; 3: narrow tile, pairs) and build (0: the common launch's kernel, 1: full)
    bool smem_set[3][4][2] = {};
    int occ_smem[3][4][2] = {};               // smem the cached occupancy was computed for
    int occ_clusters[3][4][2] = {};
    MapEntry maps[kMapCache];
};

namespace {

gemm_status_t cuda_fail(cudaError_t e)
{
    (void)cudaGetLastError();   // clear a non-sticky error so the next call starts clean
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

// Encode (or find) a 2-D row-major tensor map over rows x cols elements.
const CUtensorMap *get_map(gemm_ctx *h, const void *ptr, uint64_t rows, uint64_t cols, int dtype,
                           uint32_t box_rows, uint32_t box_cols)
{
    // direct-mapped cache keyed by every field of the map
    uint64_t key = reinterpret_cast<uintptr_t>(ptr) ^ (rows * 0x9E3779B97F4A7C15ull) ^ (cols * 0xC2B2AE3D27D4EB4Full)
                   ^ (uint64_t(dtype) << 7) ^ (uint64_t(box_rows) << 17) ^ (uint64_t(box_cols) << 29);
    key ^= key >> 31;
    key *= 0x94D049BB133111EBull;
    key ^= key >> 29;
    MapEntry &m = h->maps[key % kMapCache];
    if (m.ptr == ptr && m.rows == rows && m.cols == cols && m.dtype == dtype && m.box_rows == box_rows
        && m.box_cols == box_cols)
        return &m.map;
    m.ptr = nullptr;
    CUtensorMapDataType t = dtype == GEMM_F16    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                            : dtype == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const int es = dtype == GEMM_E4M3 ? 1 : 2;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * static_cast<cuuint64_t>(es)};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = h->encode(&m.map, t, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return nullptr;
    m.ptr = ptr;
    m.rows = rows;
    m.cols = cols;
    m.dtype = dtype;
    m.box_rows = box_rows;
    m.box_cols = box_cols;
    return &m.map;
}

// Kernel variant: 0 wide tile, single CTAs; 1 wide tile, CTA pairs; 2 narrow
// tile, single CTAs; 3 narrow tile, CTA pairs.
int variant_of(int cg, int bn) { return (bn == pts::kTileNNarrow ? 2 : 0) + cg - 1; }

pts::KernelOps ops_for(int kind, int cg, int bn, bool full)
{
    if (bn == pts::kTileNNarrow)
        return cg == 2 ? pts::kernel_ops_narrow_cg2(kind, full) : pts::kernel_ops_narrow(kind, full);
    return cg == 2 ? pts::kernel_ops_cg2(kind, full) : pts::kernel_ops_cg1(kind, full);
}

struct Plan {
    int cg, bn = pts::kTileN, stages, smem;
    bool full = true;        // the kernel with every feature, or the common launch's (see kernel_full)
    int64_t tiles_m, tiles_n, tiles;
    int split;               // column slices per tile (1, 2 or 4)
    int64_t sk_tiles;        // stream-K region: its tiles and units (0 = none)
    int64_t sk_units;
    int64_t tail = 0;        // last tiles run as two column halves each (0 = none)
    int64_t num_kb;          // k-blocks per whole tile
    int64_t units;           // work ids the schedulers hand out
    int64_t work;            // work items (record slots)
    int64_t grid_ctas;
    int max_active_clusters;
    int ctas_per_sm;
};


gemm_status_t check_sizes(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype, gemm_sched_t sched)
{
    if (dtype < GEMM_F16 || dtype > GEMM_E4M3) return GEMM_ERR_INVALID_ARG;
    if (sched < GEMM_SCHED_NONPERSISTENT || sched > GEMM_SCHED_CLC) return GEMM_ERR_INVALID_ARG;
    const int64_t lim = (int64_t(1) << 31) - 1;
    if (M < 0 || N < 0 || K < 0 || M > lim || N > lim || K > lim) return GEMM_ERR_INVALID_ARG;
    if ((K * elem_bytes(dtype)) % 16 != 0) return GEMM_ERR_INVALID_ARG;
    if ((N * 2) % 16 != 0) return GEMM_ERR_INVALID_ARG;
    return GEMM_OK;
}

// Ring depth, shared memory and resident clusters of the kernel for pl.cg
// and pl.bn.
gemm_status_t kernel_shape(gemm_ctx *h, gemm_dtype_t dtype, Plan &pl)
{
    int stages = h->opts.stages;
    if (stages == 0 && pl.bn == pts::kTileNNarrow && pl.cg == 1) {
        stages = pts::kNarrowStages;   // the ring that lets two CTAs share an SM
    } else if (stages == 0) {          // the deepest ring that fits
        stages = pts::kMaxStages;
        while (stages > 2 && pts::smem_bytes(pl.cg, stages, pl.bn) > h->max_smem_optin) --stages;
    }
    pl.stages = stages;
    pl.smem = pts::smem_bytes(pl.cg, stages, pl.bn);
    if (pl.smem > h->max_smem_optin) return GEMM_ERR_INVALID_ARG;
    const int kind = static_cast<int>(dtype);
    const int ci = variant_of(pl.cg, pl.bn);
    const int fi = pl.full ? 1 : 0;
    pts::KernelOps ops = ops_for(kind, pl.cg, pl.bn, pl.full);
    if (!h->smem_set[kind][ci][fi]) {
        if (ops.set_smem(h->max_smem_optin) != cudaSuccess) return cuda_fail(cudaErrorInvalidValue);
        h->smem_set[kind][ci][fi] = true;
    }
    if (h->occ_smem[kind][ci][fi] != pl.smem) {
        int n = 0;
        if (ops.max_active_clusters(pl.smem, &n) != cudaSuccess) return cuda_fail(cudaErrorInvalidValue);
        h->occ_smem[kind][ci][fi] = pl.smem;
        h->occ_clusters[kind][ci][fi] = n;
    }
    pl.max_active_clusters = h->occ_clusters[kind][ci][fi];
    if (pl.max_active_clusters < 1) return GEMM_ERR_CUDA;
    pl.ctas_per_sm = static_cast<int>((int64_t(pl.max_active_clusters) * pl.cg + h->sm_count - 1) / h->sm_count);
    return GEMM_OK;
}

// Whether a launch needs the kernel built with every feature: debug records
// or test hooks, the direct-store epilogue or an L2 prefetch distance (a
// grouped launch always does).  Otherwise it runs the common launch's kernel,
// which has those paths compiled out and starts faster.
bool kernel_full(const gemm_ctx *h)
{
    const int prefetch = h->opts.prefetch < 0 ? 0 : (h->opts.prefetch == 0 ? pts::kDefaultPrefetchKb : h->opts.prefetch);
    return h->opts.debug_flags != 0 || h->opts.epilogue == 2 || prefetch > 0;
}

int64_t resident_clusters(const gemm_ctx *h, const Plan &pl)
{
    int64_t resident = pl.max_active_clusters;
    if (h->opts.max_clusters > 0 && h->opts.max_clusters < resident) resident = h->opts.max_clusters;
    return resident;
}

gemm_status_t make_plan(gemm_ctx *h, int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype, gemm_sched_t sched,
                        Plan &pl)
{
    const int64_t kelems = dtype == GEMM_E4M3 ? 128 : 64;
    pl.num_kb = (K + kelems - 1) / kelems;
    // tile width: the narrow tile (single CTAs, two per SM) for short tiles
    // when the caller leaves the shape to the library and forces nothing it
    // lacks (the stream-K share, column quarters); its pair form only when
    // asked for (tile_n 128 with cta_group 2)
    const bool forced_wide_only = h->opts.split_k == 1 || h->opts.split == 4;
    pl.bn = h->opts.tile_n != 0 ? h->opts.tile_n
                                : (forced_wide_only ? pts::kTileN
                                                    : pts::choose_tile_n(pl.num_kb, h->opts.cta_group, int(sched)));
    pl.cg = pl.bn == pts::kTileNNarrow ? (h->opts.cta_group == 2 ? 2 : 1)
                                        : (h->opts.cta_group != 0 ? h->opts.cta_group
                                                                  : pts::choose_cta_group(pl.num_kb, int(sched)));
    const int64_t tile_m = int64_t(pts::kRowsPerCta) * pl.cg;
    pl.tiles_m = (M + tile_m - 1) / tile_m;
    pl.tiles_n = (N + pl.bn - 1) / pl.bn;
    pl.tiles = pl.tiles_m * pl.tiles_n;
    if (pl.tiles > (int64_t(1) << 30)) return GEMM_ERR_INVALID_ARG;
    pl.full = kernel_full(h);
    gemm_status_t st = kernel_shape(h, dtype, pl);
    if (st != GEMM_OK) return st;
    int64_t resident = resident_clusters(h, pl);
    // column slices for a problem smaller than one wave (or forced, for
    // testing); the narrow tile is cut in halves at most (64-column slices)
    pl.split = h->opts.split > 0 ? h->opts.split : pts::choose_split(pl.tiles, resident);
    if (pl.bn == pts::kTileNNarrow && pl.split > 2) pl.split = 2;
    pl.sk_tiles = 0;
    pl.sk_units = 0;
    pl.tail = 0;
    // the partial last wave: column halves of its tiles or the stream-K share
    if (pl.bn == pts::kTileN && pl.split == 1
        && (pl.sk_tiles = pts::choose_last_wave(pl.tiles, resident, pl.num_kb, h->opts.split == 0,
                                                h->opts.split_k, int(sched), pl.tail)) > 0)
        pl.sk_units = resident;
    pl.units = pl.sk_units > 0 ? pl.sk_units + pl.tiles - pl.sk_tiles : pl.tiles * pl.split + pl.tail;
    pl.work = pl.sk_units > 0 ? pts::kSkMaxPieces * pl.sk_units + pl.tiles - pl.sk_tiles : pl.units;
    if (pl.work > (int64_t(1) << 31) - 1) return GEMM_ERR_INVALID_ARG;
    int64_t clusters = pl.units;
    if (sched == GEMM_SCHED_STATIC) clusters = pl.units < resident ? pl.units : resident;
    pl.grid_ctas = clusters * pl.cg;
    return GEMM_OK;
}

// With GEMM_DEBUG_RECORDS: zeroed records for `work` work items on `stream`
// (grown as needed), handed to the kernel in p.records; else p.records = null.
gemm_status_t prepare_records(gemm_ctx *h, int64_t work, cudaStream_t stream, pts::GemmParams &p)
{
    p.records = nullptr;
    if (!(h->opts.debug_flags & GEMM_DEBUG_RECORDS)) return GEMM_OK;
    if (h->records_cap < work) {
        cudaFree(h->d_records);
        h->d_records = nullptr;
        h->records_cap = 0;
        if (cudaMalloc(&h->d_records, size_t(work) * sizeof(pts::TileRecord)) != cudaSuccess)
            return cuda_fail(cudaErrorMemoryAllocation);
        h->records_cap = work;
    }
    if (cudaMemsetAsync(h->d_records, 0, size_t(work) * sizeof(pts::TileRecord), stream) != cudaSuccess)
        return cuda_fail(cudaErrorInvalidValue);
    p.records = h->d_records;
    return GEMM_OK;
}

gemm_status_t launch(gemm_ctx *h, int64_t M, int64_t N, int64_t K, const void *A, const void *B, void *C,
                     gemm_dtype_t dtype, gemm_sched_t sched, float scale_a, float scale_b,
                     cudaStream_t stream)
{
    if (M == 0 || N == 0) return GEMM_OK;
    if (C == nullptr || reinterpret_cast<uintptr_t>(C) % 16 != 0) return GEMM_ERR_INVALID_ARG;
    if (K == 0) return cuda_fail(pts::launch_zero_fill(C, M * N * 2, stream));
    if (A == nullptr || B == nullptr) return GEMM_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(A) % 16 != 0 || reinterpret_cast<uintptr_t>(B) % 16 != 0)
        return GEMM_ERR_INVALID_ARG;
    float out_scale = 1.0f;
    if (dtype == GEMM_E4M3) {
        if (!(scale_a > 0.0f) || !(scale_b > 0.0f) || !std::isfinite(scale_a) || !std::isfinite(scale_b))
            return GEMM_ERR_INVALID_ARG;
        out_scale = 1.0f / (scale_a * scale_b);
        if (!std::isfinite(out_scale)) return GEMM_ERR_INVALID_ARG;
    }
    if (cudaSetDevice(h->device) != cudaSuccess) return cuda_fail(cudaErrorInvalidDevice);

    Plan pl;
    gemm_status_t st = make_plan(h, M, N, K, dtype, sched, pl);
    if (st != GEMM_OK) return st;
    if (pl.sk_units > 0) {   // fixup workspace: a partial slot and 4 sync words per (region tile, CTA, warp)
        const size_t tiles = size_t(pl.sk_tiles);
        const size_t need_p = tiles * size_t(pts::kSkMaxParts - 1) * pl.cg * pts::kPartialFloats * sizeof(float);
        const size_t need_s = tiles * pl.cg * pts::kEpiWarps * 4 * sizeof(uint32_t);
        if (h->ws_partial_cap < need_p) {
            cudaFree(h->d_ws_partial);
            h->d_ws_partial = nullptr;
            h->ws_partial_cap = 0;
            if (cudaMalloc(&h->d_ws_partial, need_p) != cudaSuccess) return cuda_fail(cudaErrorMemoryAllocation);
            h->ws_partial_cap = need_p;
        }
        if (h->ws_sync_cap < need_s) {
            cudaFree(h->d_ws_sync);
            h->d_ws_sync = nullptr;
            h->ws_sync_cap = 0;
            if (cudaMalloc(&h->d_ws_sync, need_s) != cudaSuccess) return cuda_fail(cudaErrorMemoryAllocation);
            if (cudaMemset(h->d_ws_sync, 0, need_s) != cudaSuccess) return cuda_fail(cudaErrorMemoryAllocation);
            h->ws_sync_cap = need_s;
        }
    }
    // Each map is copied out of the cache at once: a later lookup in this same
    // call may reuse the cache slot an earlier map came from.
    const uint32_t kelems = dtype == GEMM_E4M3 ? 128u : 64u;
    const uint32_t brows = uint32_t(pl.bn / pl.cg);
    const int cdt = dtype == GEMM_F16 ? GEMM_F16 : GEMM_BF16;
    const bool slices = pl.split > 1 || pl.tail > 0;
    const int slice_div = pl.tail > 0 ? 2 : pl.split;
    CUtensorMap ma, mb0, mb_slice, mc;
    const CUtensorMap *m;
    if (!(m = get_map(h, A, uint64_t(M), uint64_t(K), dtype, pts::kRowsPerCta, kelems))) return GEMM_ERR_CUDA;
    ma = *m;
    if (!(m = get_map(h, B, uint64_t(N), uint64_t(K), dtype, brows, kelems))) return GEMM_ERR_CUDA;
    mb0 = *m;
    mb_slice = mb0;
    if (slices) {
        if (!(m = get_map(h, B, uint64_t(N), uint64_t(K), dtype, brows / uint32_t(slice_div), kelems)))
            return GEMM_ERR_CUDA;
        mb_slice = *m;
    }
    if (!(m = get_map(h, C, uint64_t(M), uint64_t(N), cdt, pts::kEpiRowsPerWarp, pts::kEpiChunkCols)))
        return GEMM_ERR_CUDA;
    mc = *m;
    const CUtensorMap *mb[3] = {&mb0, (slices && slice_div == 2) ? &mb_slice : &mb0,
                                (slices && slice_div == 4) ? &mb_slice : &mb0};

    pts::GemmParams p{};
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.num_kb = static_cast<int32_t>(pl.num_kb);
    p.tiles_m = static_cast<int32_t>(pl.tiles_m);
    p.tiles_n = static_cast<int32_t>(pl.tiles_n);
    p.num_tiles = static_cast<int32_t>(pl.tiles);
    p.split = pl.split;
    p.sk_tiles = static_cast<int32_t>(pl.sk_tiles);
    p.sk_units = static_cast<int32_t>(pl.sk_units);
    p.ws_partial = pl.sk_units > 0 ? h->d_ws_partial : nullptr;
    p.ws_sync = pl.sk_units > 0 ? h->d_ws_sync : nullptr;
    p.num_units = static_cast<int32_t>(pl.units);
    p.num_work = static_cast<int32_t>(pl.work);
    p.group_m = h->opts.group_size_m;
    p.sched = static_cast<int32_t>(sched);
    p.stages = pl.stages;
    p.prefetch_kb = h->opts.prefetch < 0 ? 0 : (h->opts.prefetch == 0 ? pts::kDefaultPrefetchKb : h->opts.prefetch);
    p.epi_direct = h->opts.epilogue == 2 ? 1 : 0;
    p.clc_lead = h->opts.clc_depth;
    p.tail_tiles = static_cast<int32_t>(pl.tail);
    p.c_ptr = C;
    p.out_scale = out_scale;
    p.debug_flags = h->opts.debug_flags;
    p.fault_arg = h->opts.fault_arg;
    p.timeout_ns = h->opts.timeout_ns;
    p.status = h->d_status;
    if ((st = prepare_records(h, pl.work, stream, p)) != GEMM_OK) return st;
    h->last_work = pl.work;
    h->last_cta_group = pl.cg;
    h->last_sk_tiles = pl.sk_tiles;
    h->last_sk_units = pl.sk_units;
    h->last_num_kb = pl.num_kb;

    cudaError_t e = ops_for(static_cast<int>(dtype), pl.cg, pl.bn, pl.full)
                        .launch(ma, mb, mc, p, static_cast<int>(pl.grid_ctas), pl.smem, stream,
                                h->opts.overlap_launch >= 0);
    if (e != cudaSuccess) return cuda_fail(e);
    return cuda_fail(cudaGetLastError());
}

// ---- grouped launch ---------------------------------------------------------

gemm_status_t check_group_problem(const gemm_group_problem_t &q, gemm_dtype_t dtype, gemm_sched_t sched)
{
    gemm_status_t st = check_sizes(q.M, q.N, q.K, dtype, sched);
    if (st != GEMM_OK) return st;
    if (q.M == 0 || q.N == 0) return GEMM_OK;
    if (q.C == nullptr || reinterpret_cast<uintptr_t>(q.C) % 16 != 0) return GEMM_ERR_INVALID_ARG;
    if (q.K == 0) return GEMM_OK;
    if (q.A == nullptr || q.B == nullptr || reinterpret_cast<uintptr_t>(q.A) % 16 != 0
        || reinterpret_cast<uintptr_t>(q.B) % 16 != 0)
        return GEMM_ERR_INVALID_ARG;
    if (dtype == GEMM_E4M3) {
        if (!(q.scale_a > 0.0f) || !(q.scale_b > 0.0f) || !std::isfinite(q.scale_a) || !std::isfinite(q.scale_b)
            || !std::isfinite(1.0f / (q.scale_a * q.scale_b)))
            return GEMM_ERR_INVALID_ARG;
    }
    return GEMM_OK;
}

// Launch shape of a grouped launch, and (encode) its problem table: one
// GroupDesc per problem in work-id order, then the tile prefix sums
// group_start[0..count].
struct GroupedPlan {
    Plan pl;
    std::vector<int64_t> order;   // order[j] = the caller's index of the j-th problem of the work-id list
    std::vector<pts::GroupDesc> desc;
    std::vector<int32_t> start;
};

gemm_status_t plan_grouped(gemm_ctx *h, const gemm_group_problem_t *q, int64_t count, gemm_dtype_t dtype,
                           gemm_sched_t sched, bool encode, GroupedPlan &gp)
{
    if (count < 0 || count > GEMM_GROUPED_MAX_PROBLEMS || (count > 0 && q == nullptr)) return GEMM_ERR_INVALID_ARG;
    if (dtype < GEMM_F16 || dtype > GEMM_E4M3) return GEMM_ERR_INVALID_ARG;
    const int64_t kelems = dtype == GEMM_E4M3 ? 128 : 64;
    // CTA group: the single-problem rule applied to the mean k-blocks per
    // tile, weighted by output size
    double w_sum = 0.0, kb_sum = 0.0;
    for (int64_t g = 0; g < count; ++g) {
        gemm_status_t st = check_group_problem(q[g], dtype, sched);
        if (st != GEMM_OK) return st;
        const double w = double(q[g].M) * double(q[g].N);
        w_sum += w;
        kb_sum += w * double((q[g].K + kelems - 1) / kelems);
    }
    Plan &pl = gp.pl;
    pl.cg = h->opts.cta_group != 0 ? h->opts.cta_group
                                   : pts::choose_cta_group(w_sum > 0.0 ? int64_t(kb_sum / w_sum) : 0);
    const int64_t tile_m = int64_t(pts::kRowsPerCta) * pl.cg;
    // work-id order of the problems: most k-blocks first (longest processing
    // time first: the tiles handed out last, which decide how evenly the
    // clusters finish, are the short ones), or as given
    gp.order.resize(size_t(count));
    for (int64_t g = 0; g < count; ++g) gp.order[size_t(g)] = g;
    if (h->opts.group_order != 2)
        std::stable_sort(gp.order.begin(), gp.order.end(), [&](int64_t a, int64_t b) {
            return (q[a].K + kelems - 1) / kelems > (q[b].K + kelems - 1) / kelems;
        });
    gp.start.assign(size_t(count) + 1, 0);
    int64_t tiles = 0;
    for (int64_t j = 0; j < count; ++j) {
        const gemm_group_problem_t &x = q[gp.order[size_t(j)]];
        if (x.M > 0 && x.N > 0)
            tiles += ((x.M + tile_m - 1) / tile_m) * ((x.N + pts::kTileN - 1) / pts::kTileN);
        if (tiles > (int64_t(1) << 30)) return GEMM_ERR_INVALID_ARG;
        gp.start[size_t(j) + 1] = static_cast<int32_t>(tiles);
    }
    pl.tiles_m = pl.tiles_n = 0;
    pl.tiles = tiles;
    pl.num_kb = 0;
    pl.split = 1;
    pl.sk_tiles = pl.sk_units = 0;
    pl.units = pl.work = tiles;
    pl.full = true;   // the grouped decoder is one of the features
    gemm_status_t st = kernel_shape(h, dtype, pl);
    if (st != GEMM_OK) return st;
    const int64_t resident = resident_clusters(h, pl);
    pl.grid_ctas = (sched == GEMM_SCHED_STATIC && tiles > resident ? resident : tiles) * pl.cg;
    if (!encode) return GEMM_OK;

    // Each map is copied out of the cache at once (a later lookup may reuse its slot).
    gp.desc.resize(size_t(count));
    const uint32_t brows = uint32_t(pts::kTileN / pl.cg);
    const int cdt = dtype == GEMM_F16 ? GEMM_F16 : GEMM_BF16;
    for (int64_t j = 0; j < count; ++j) {
        pts::GroupDesc &d = gp.desc[size_t(j)];
        std::memset(&d, 0, sizeof(d));   // padding too: tables are compared byte for byte
        const gemm_group_problem_t &x = q[gp.order[size_t(j)]];
        d.index = static_cast<int32_t>(gp.order[size_t(j)]);
        if (x.M == 0 || x.N == 0) continue;
        d.M = static_cast<int32_t>(x.M);
        d.N = static_cast<int32_t>(x.N);
        d.num_kb = static_cast<int32_t>((x.K + kelems - 1) / kelems);
        d.tiles_m = static_cast<int32_t>((x.M + tile_m - 1) / tile_m);
        d.tiles_n = static_cast<int32_t>((x.N + pts::kTileN - 1) / pts::kTileN);
        d.out_scale = (dtype == GEMM_E4M3 && x.K > 0) ? 1.0f / (x.scale_a * x.scale_b) : 1.0f;
        const CUtensorMap *m;
        if (!(m = get_map(h, x.C, uint64_t(x.M), uint64_t(x.N), cdt, pts::kEpiRowsPerWarp, pts::kEpiChunkCols)))
            return GEMM_ERR_CUDA;
        d.tmC = *m;
        if (x.K == 0) continue;
        if (!(m = get_map(h, x.A, uint64_t(x.M), uint64_t(x.K), dtype, pts::kRowsPerCta, uint32_t(kelems))))
            return GEMM_ERR_CUDA;
        d.tmA = *m;
        if (!(m = get_map(h, x.B, uint64_t(x.N), uint64_t(x.K), dtype, brows, uint32_t(kelems))))
            return GEMM_ERR_CUDA;
        d.tmB = *m;
    }
    return GEMM_OK;
}

// Put the problem table on the device.  The same table as the last one
// uploaded is used again as it is; a new one goes to the other slot, once
// the launch that last read that slot has finished (the host waits for it),
// copied from pinned memory on `stream`.
gemm_status_t upload_table(gemm_ctx *h, const GroupedPlan &gp, cudaStream_t stream, int &slot, bool &uploaded)
{
    const size_t desc_bytes = gp.desc.size() * sizeof(pts::GroupDesc);
    const size_t bytes = desc_bytes + gp.start.size() * sizeof(int32_t);
    const int cur = h->tab_cur;
    if (h->tab_bytes[cur] == bytes && std::memcmp(h->tab_host[cur], gp.desc.data(), desc_bytes) == 0
        && std::memcmp(static_cast<char *>(h->tab_host[cur]) + desc_bytes, gp.start.data(), bytes - desc_bytes) == 0) {
        slot = cur;
        uploaded = false;
        return GEMM_OK;
    }
    if (h->ev_tab[0] == nullptr)
        for (int b = 0; b < kGroupSlots; ++b)
            if (cudaEventCreateWithFlags(&h->ev_tab[b], cudaEventDisableTiming) != cudaSuccess)
                return cuda_fail(cudaErrorUnknown);
    const int s = (cur + 1) % kGroupSlots;
    if (cudaEventSynchronize(h->ev_tab[s]) != cudaSuccess) return cuda_fail(cudaErrorUnknown);
    h->tab_bytes[s] = 0;
    if (h->tab_cap[s] < bytes) {
        cudaFreeHost(h->tab_host[s]);
        cudaFree(h->tab_dev[s]);
        h->tab_host[s] = h->tab_dev[s] = nullptr;
        h->tab_cap[s] = 0;
        const size_t cap = std::max(bytes, size_t(64) << 10);
        if (cudaMallocHost(&h->tab_host[s], cap) != cudaSuccess || cudaMalloc(&h->tab_dev[s], cap) != cudaSuccess)
            return cuda_fail(cudaErrorMemoryAllocation);
        h->tab_cap[s] = cap;
    }
    std::memcpy(h->tab_host[s], gp.desc.data(), desc_bytes);
    std::memcpy(static_cast<char *>(h->tab_host[s]) + desc_bytes, gp.start.data(), bytes - desc_bytes);
    if (cudaMemcpyAsync(h->tab_dev[s], h->tab_host[s], bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess)
        return cuda_fail(cudaErrorUnknown);
    h->tab_bytes[s] = bytes;
    h->tab_cur = s;
    slot = s;
    uploaded = true;
    return GEMM_OK;
}

gemm_status_t launch_grouped(gemm_ctx *h, const gemm_group_problem_t *q, int64_t count, gemm_dtype_t dtype,
                             gemm_sched_t sched, cudaStream_t stream)
{
    if (cudaSetDevice(h->device) != cudaSuccess) return cuda_fail(cudaErrorInvalidDevice);
    // the problem table outlives no launch that a graph could replay later
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return cuda_fail(cudaErrorUnknown);
    if (cap != cudaStreamCaptureStatusNone) return GEMM_ERR_INVALID_ARG;
    GroupedPlan gp;
    gemm_status_t st = plan_grouped(h, q, count, dtype, sched, true, gp);
    if (st != GEMM_OK) return st;
    const Plan &pl = gp.pl;
    if (pl.tiles == 0) return GEMM_OK;
    int slot = 0;
    bool uploaded = false;
    if ((st = upload_table(h, gp, stream, slot, uploaded)) != GEMM_OK) return st;

    pts::GemmParams p{};
    p.num_tiles = static_cast<int32_t>(pl.tiles);
    p.split = 1;
    p.num_units = static_cast<int32_t>(pl.units);
    p.num_work = static_cast<int32_t>(pl.work);
    p.group_m = h->opts.group_size_m;
    p.sched = static_cast<int32_t>(sched);
    p.stages = pl.stages;
    p.prefetch_kb = h->opts.prefetch < 0 ? 0 : (h->opts.prefetch == 0 ? pts::kDefaultPrefetchKb : h->opts.prefetch);
    p.clc_lead = h->opts.clc_depth;
    p.out_scale = 1.0f;
    p.debug_flags = h->opts.debug_flags;
    p.fault_arg = h->opts.fault_arg;
    p.timeout_ns = h->opts.timeout_ns;
    p.status = h->d_status;
    p.num_groups = static_cast<int32_t>(count);
    p.groups = static_cast<const pts::GroupDesc *>(h->tab_dev[slot]);
    p.group_start = reinterpret_cast<const int32_t *>(static_cast<const char *>(h->tab_dev[slot])
                                                      + gp.desc.size() * sizeof(pts::GroupDesc));
    if ((st = prepare_records(h, pl.work, stream, p)) != GEMM_OK) return st;
    h->last_work = pl.work;
    h->last_cta_group = pl.cg;
    h->last_sk_tiles = h->last_sk_units = h->last_num_kb = 0;

    // the kernel's own maps are unused in a grouped launch
    CUtensorMap none;
    std::memset(&none, 0, sizeof(none));
    const CUtensorMap *mb[3] = {&none, &none, &none};
    // A launch right after an upload does not overlap the previous grid: the
    // copy sits between them in the stream.
    cudaError_t e = ops_for(static_cast<int>(dtype), pl.cg, pl.bn, pl.full)
                        .launch(none, mb, none, p, static_cast<int>(pl.grid_ctas), pl.smem, stream,
                                h->opts.overlap_launch >= 0 && !uploaded);
    if (e != cudaSuccess) return cuda_fail(e);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
    // (the first launch always uploads, which creates the events)
    if (cudaEventRecord(h->ev_tab[slot], stream) != cudaSuccess) return cuda_fail(cudaErrorUnknown);
    return GEMM_OK;
}

gemm_status_t read_status(gemm_ctx *h, cudaStream_t stream, int *device_status)
{
    if (cudaSetDevice(h->device) != cudaSuccess) return cuda_fail(cudaErrorInvalidDevice);
    if (cudaStreamSynchronize(stream) != cudaSuccess) return cuda_fail(cudaErrorUnknown);
    int32_t s[4] = {0, 0, 0, 0};
    if (cudaMemcpy(s, h->d_status, sizeof(s), cudaMemcpyDeviceToHost) != cudaSuccess)
        return cuda_fail(cudaErrorUnknown);
    if (s[0] != 0 && cudaMemset(h->d_status, 0, sizeof(s)) != cudaSuccess) return cuda_fail(cudaErrorUnknown);
    // A launch that stopped on an error may have left stream-K claim counters
    // or ready flags set (a completed launch leaves them at zero): clear them
    // so that the next launch starts clean.
    if (s[0] != 0 && h->d_ws_sync != nullptr && cudaMemset(h->d_ws_sync, 0, h->ws_sync_cap) != cudaSuccess)
        return cuda_fail(cudaErrorUnknown);
    if (device_status) *device_status = s[0] == 0 ? 0 : (s[0] << 24) | ((s[1] & 0xff) << 16) | (s[2] & 0xffff);
    return s[0] == pts::DEV_ERR_TIMEOUT ? GEMM_ERR_TIMEOUT : GEMM_OK;
}

}  // namespace

extern "C" {

const char *gemm_status_string(gemm_status_t s)
{
    switch (s) {
    case GEMM_OK: return "ok";
    case GEMM_ERR_INVALID_ARG: return "invalid argument";
    case GEMM_ERR_UNSUPPORTED: return "unsupported device (needs compute capability 10.3)";
    case GEMM_ERR_CUDA: return "CUDA error";
    case GEMM_ERR_TIMEOUT: return "device wait timed out";
    case GEMM_ERR_COVERAGE: return "a tile was not computed exactly once";
    default: return "unknown status";
    }
}

gemm_status_t gemm_create(gemm_handle_t *out, int device, const gemm_opts_t *opts)
{
    if (out == nullptr) return GEMM_ERR_INVALID_ARG;
    *out = nullptr;
    gemm_opts_t o{};
    if (opts) o = *opts;
    if (o.group_size_m == 0) o.group_size_m = 8;
    if (o.timeout_ns == 0) o.timeout_ns = kDefaultTimeoutNs;
    if (o.cta_group < 0 || o.cta_group > 2) return GEMM_ERR_INVALID_ARG;
    if (o.group_size_m < 1 || o.stages < 0 || o.stages == 1 || o.stages > pts::kMaxStages || o.max_clusters < 0)
        return GEMM_ERR_INVALID_ARG;
    if (o.prefetch < -1 || o.prefetch > 64 || o.overlap_launch < -1 || o.overlap_launch > 0 || o.epilogue < 0 || o.epilogue > 2)
        return GEMM_ERR_INVALID_ARG;
    if (o.group_order < 0 || o.group_order > 2) return GEMM_ERR_INVALID_ARG;
    if (o.split < 0 || o.split > 4 || o.split == 3 || o.split_k < -1 || o.split_k > 1
        || (o.split > 1 && o.split_k == 1))
        return GEMM_ERR_INVALID_ARG;
    if (o.tile_n != 0 && o.tile_n != pts::kTileN && o.tile_n != pts::kTileNNarrow) return GEMM_ERR_INVALID_ARG;
    if (o.clc_depth < 0 || o.clc_depth > 2) return GEMM_ERR_INVALID_ARG;
    if (o.clc_depth == 0) o.clc_depth = pts::kDefaultClcLead;
    if (o.tile_n == pts::kTileNNarrow && (o.split == 4 || o.split_k == 1)) return GEMM_ERR_INVALID_ARG;
    if (o.debug_flags & ~(GEMM_DEBUG_RECORDS | GEMM_DEBUG_CLC_STOP_AT | GEMM_DEBUG_FAULT_SKIP_TMA))
        return GEMM_ERR_INVALID_ARG;

    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return cuda_fail(cudaErrorNoDevice);
    if (cudaSetDevice(device) != cudaSuccess) return cuda_fail(cudaErrorInvalidDevice);
    int major = 0, minor = 0, sms = 0, smem = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
    if (major != 10 || minor != 3) return GEMM_ERR_UNSUPPORTED;

    gemm_ctx *h = new (std::nothrow) gemm_ctx();
    if (!h) return GEMM_ERR_CUDA;
    h->device = device;
    h->sm_count = sms;
    h->max_smem_optin = smem;
    h->opts = o;
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess
        || q != cudaDriverEntryPointSuccess || fn == nullptr) {
        delete h;
        return cuda_fail(cudaErrorUnknown);
    }
    h->encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    if (cudaMalloc(&h->d_status, 4 * sizeof(int32_t)) != cudaSuccess
        || cudaMemset(h->d_status, 0, 4 * sizeof(int32_t)) != cudaSuccess) {
        cudaFree(h->d_status);
        delete h;
        return cuda_fail(cudaErrorMemoryAllocation);
    }
    *out = h;
    return GEMM_OK;
}

gemm_status_t gemm_run(gemm_handle_t h, int64_t M, int64_t N, int64_t K, const void *A, const void *B, void *C,
                       gemm_dtype_t dtype, gemm_sched_t sched, float scale_a, float scale_b, void *stream)
{
    if (h == nullptr) return GEMM_ERR_INVALID_ARG;
    gemm_status_t st = check_sizes(M, N, K, dtype, sched);
    if (st != GEMM_OK) return st;
    return launch(h, M, N, K, A, B, C, dtype, sched, scale_a, scale_b, static_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_run_host(gemm_handle_t h, int64_t M, int64_t N, int64_t K, const void *A_host,
                            const void *B_host, void *C_host, gemm_dtype_t dtype, gemm_sched_t sched,
                            float scale_a, float scale_b, void *stream)
{
    if (h == nullptr) return GEMM_ERR_INVALID_ARG;
    gemm_status_t st = check_sizes(M, N, K, dtype, sched);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) return GEMM_OK;
    if (C_host == nullptr || (K > 0 && (A_host == nullptr || B_host == nullptr))) return GEMM_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaSetDevice(h->device) != cudaSuccess) return cuda_fail(cudaErrorInvalidDevice);
    auto round_up = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t a_bytes = size_t(M) * size_t(K) * elem_bytes(dtype);
    const size_t b_bytes = size_t(N) * size_t(K) * elem_bytes(dtype);
    const size_t c_bytes = size_t(M) * size_t(N) * 2;
    const size_t need = round_up(a_bytes) + round_up(b_bytes) + round_up(c_bytes);
    if (h->host_bufs_cap < need) {
        if (cudaStreamSynchronize(s) != cudaSuccess) return cuda_fail(cudaErrorUnknown);
        cudaFree(h->d_host_bufs);
        h->d_host_bufs = nullptr;
        h->host_bufs_cap = 0;
        if (cudaMalloc(&h->d_host_bufs, need) != cudaSuccess) return cuda_fail(cudaErrorMemoryAllocation);
        h->host_bufs_cap = need;
    }
    char *dA = static_cast<char *>(h->d_host_bufs);
    char *dB = dA + round_up(a_bytes);
    char *dC = dB + round_up(b_bytes);
    if (a_bytes && cudaMemcpyAsync(dA, A_host, a_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return cuda_fail(cudaErrorUnknown);
    if (b_bytes && cudaMemcpyAsync(dB, B_host, b_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return cuda_fail(cudaErrorUnknown);
    st = launch(h, M, N, K, dA, dB, dC, dtype, sched, scale_a, scale_b, s);
    if (st != GEMM_OK) return st;
    if (cudaMemcpyAsync(C_host, dC, c_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return cuda_fail(cudaErrorUnknown);
    return read_status(h, s, nullptr);
}

gemm_status_t gemm_run_host_batch(gemm_handle_t h, const gemm_host_problem_t *probs, int64_t n,
                                  gemm_sched_t sched, void *stream)
{
    if (h == nullptr || n < 0 || (n > 0 && probs == nullptr)) return GEMM_ERR_INVALID_ARG;
    auto round_up = [](size_t x) { return (x + 255) & ~size_t(255); };
    size_t need = 0;
    for (int64_t i = 0; i < n; ++i) {
        const gemm_host_problem_t &q = probs[i];
        gemm_status_t st = check_sizes(q.M, q.N, q.K, q.dtype, sched);
        if (st != GEMM_OK) return st;
        if (q.M == 0 || q.N == 0) continue;
        if (q.C == nullptr || (q.K > 0 && (q.A == nullptr || q.B == nullptr))) return GEMM_ERR_INVALID_ARG;
        const size_t es = size_t(elem_bytes(q.dtype));
        const size_t slot = round_up(size_t(q.M) * size_t(q.K) * es) + round_up(size_t(q.N) * size_t(q.K) * es)
                            + round_up(size_t(q.M) * size_t(q.N) * 2);
        if (slot > need) need = slot;
    }
    if (n == 0 || need == 0) return GEMM_OK;
    if (cudaSetDevice(h->device) != cudaSuccess) return cuda_fail(cudaErrorInvalidDevice);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (h->s_h2d == nullptr) {   // copy streams and events, created once
        if (cudaStreamCreateWithFlags(&h->s_h2d, cudaStreamNonBlocking) != cudaSuccess
            || cudaStreamCreateWithFlags(&h->s_d2h[0], cudaStreamNonBlocking) != cudaSuccess
            || cudaStreamCreateWithFlags(&h->s_d2h[1], cudaStreamNonBlocking) != cudaSuccess
            || cudaEventCreateWithFlags(&h->ev_entry, cudaEventDisableTiming) != cudaSuccess)
            return cuda_fail(cudaErrorUnknown);
        for (int b = 0; b < kBatchSlots; ++b)
            if (cudaEventCreateWithFlags(&h->ev_in[b], cudaEventDisableTiming) != cudaSuccess
                || cudaEventCreateWithFlags(&h->ev_comp[b], cudaEventDisableTiming) != cudaSuccess
                || cudaEventCreateWithFlags(&h->ev_free[b], cudaEventDisableTiming) != cudaSuccess)
                return cuda_fail(cudaErrorUnknown);
    }
    if (h->slot_cap < need) {
        if (cudaDeviceSynchronize() != cudaSuccess) return cuda_fail(cudaErrorUnknown);
        for (int b = 0; b < kBatchSlots; ++b) {
            cudaFree(h->d_slot[b]);
            h->d_slot[b] = nullptr;
        }
        h->slot_cap = 0;
        for (int b = 0; b < kBatchSlots; ++b)
            if (cudaMalloc(&h->d_slot[b], need) != cudaSuccess) return cuda_fail(cudaErrorMemoryAllocation);
        h->slot_cap = need;
    }
    // Processing order.  The problems are independent, so the order is free:
    // alternate between the most output-heavy and the most input-heavy
    // remaining problem, so that copy-in and copy-out (separate directions of
    // the host link) are busy at the same time instead of one after the other.
    std::vector<int64_t> order;
    order.reserve(size_t(n));
    {
        std::vector<std::pair<double, int64_t>> net;
        for (int64_t i = 0; i < n; ++i) {
            const gemm_host_problem_t &q = probs[i];
            if (q.M == 0 || q.N == 0) continue;
            const double es = elem_bytes(q.dtype);
            net.emplace_back(double(q.M + q.N) * double(q.K) * es - double(q.M) * double(q.N) * 2.0, i);
        }
        std::stable_sort(net.begin(), net.end(),
                         [](const std::pair<double, int64_t> &x, const std::pair<double, int64_t> &y) {
                             return x.first < y.first;
                         });
        for (size_t lo = 0, hi = net.size(); lo < hi;) {
            order.push_back(net[lo++].second);
            if (lo < hi) order.push_back(net[--hi].second);
        }
    }
    // everything already queued on the caller's stream comes first
    if (cudaEventRecord(h->ev_entry, cs) != cudaSuccess || cudaStreamWaitEvent(h->s_h2d, h->ev_entry, 0) != cudaSuccess)
        return cuda_fail(cudaErrorUnknown);
    gemm_status_t first_error = GEMM_OK;
    for (size_t j = 0; j < order.size(); ++j) {
        const gemm_host_problem_t &q = probs[order[j]];
        const int b = int(j % kBatchSlots);
        const size_t es = size_t(elem_bytes(q.dtype));
        const size_t a_bytes = size_t(q.M) * size_t(q.K) * es, b_bytes = size_t(q.N) * size_t(q.K) * es;
        const size_t c_bytes = size_t(q.M) * size_t(q.N) * 2;
        char *dA = static_cast<char *>(h->d_slot[b]);
        char *dB = dA + round_up(a_bytes);
        char *dC = dB + round_up(b_bytes);
        // slot b is free once the copy-out of the GEMM that used it kBatchSlots steps ago is done
        if (j >= size_t(kBatchSlots) && cudaStreamWaitEvent(h->s_h2d, h->ev_free[b], 0) != cudaSuccess)
            return cuda_fail(cudaErrorUnknown);
        if ((a_bytes && cudaMemcpyAsync(dA, q.A, a_bytes, cudaMemcpyHostToDevice, h->s_h2d) != cudaSuccess)
            || (b_bytes && cudaMemcpyAsync(dB, q.B, b_bytes, cudaMemcpyHostToDevice, h->s_h2d) != cudaSuccess)
            || cudaEventRecord(h->ev_in[b], h->s_h2d) != cudaSuccess || cudaStreamWaitEvent(cs, h->ev_in[b], 0) != cudaSuccess)
            return cuda_fail(cudaErrorUnknown);
        gemm_status_t st = launch(h, q.M, q.N, q.K, dA, dB, dC, q.dtype, sched, q.scale_a, q.scale_b, cs);
        if (st != GEMM_OK && first_error == GEMM_OK) first_error = st;
        cudaStream_t out = h->s_d2h[j & 1];
        if (cudaEventRecord(h->ev_comp[b], cs) != cudaSuccess || cudaStreamWaitEvent(out, h->ev_comp[b], 0) != cudaSuccess
            || cudaMemcpyAsync(q.C, dC, c_bytes, cudaMemcpyDeviceToHost, out) != cudaSuccess
            || cudaEventRecord(h->ev_free[b], out) != cudaSuccess)
            return cuda_fail(cudaErrorUnknown);
    }
    // the caller's stream continues after the last copy-out
    for (int b = 0; b < kBatchSlots; ++b)
        if (cudaStreamWaitEvent(cs, h->ev_free[b], 0) != cudaSuccess) return cuda_fail(cudaErrorUnknown);
    gemm_status_t st = read_status(h, cs, nullptr);
    return first_error != GEMM_OK ? first_error : st;
}

gemm_status_t gemm_query(gemm_handle_t h, int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                         gemm_sched_t sched, gemm_launch_info_t *info)
{
    if (h == nullptr || info == nullptr) return GEMM_ERR_INVALID_ARG;
    gemm_status_t st = check_sizes(M, N, K, dtype, sched);
    if (st != GEMM_OK) return st;
    if (cudaSetDevice(h->device) != cudaSuccess) return cuda_fail(cudaErrorInvalidDevice);
    Plan pl;
    st = make_plan(h, M, N, K, dtype, sched, pl);
    if (st != GEMM_OK) return st;
    std::memset(info, 0, sizeof(*info));
    info->tile_m = pts::kRowsPerCta * pl.cg;
    info->tile_n = pl.bn;
    info->tile_k = dtype == GEMM_E4M3 ? 128 : 64;
    info->cta_group = pl.cg;
    info->stages = pl.stages;
    info->ctas_per_sm = pl.ctas_per_sm;
    info->tiles_m = pl.tiles_m;
    info->tiles_n = pl.tiles_n;
    info->tiles = pl.tiles;
    info->split = pl.split;
    info->split_k = pl.sk_units > 0 ? 1 : 0;
    info->sk_tiles = pl.sk_tiles;
    info->sk_units = pl.sk_units;
    info->tail_tiles = pl.tail;
    info->work_items = pl.work;
    info->units = pl.units;
    info->grid_ctas = (M == 0 || N == 0 || K == 0) ? 0 : pl.grid_ctas;
    info->max_active_clusters = pl.max_active_clusters;
    info->smem_bytes = pl.smem;
    info->threads = pts::kThreads;
    return GEMM_OK;
}

gemm_status_t gemm_run_grouped(gemm_handle_t h, const gemm_group_problem_t *problems, int64_t count,
                               gemm_dtype_t dtype, gemm_sched_t sched, void *stream)
{
    if (h == nullptr) return GEMM_ERR_INVALID_ARG;
    return launch_grouped(h, problems, count, dtype, sched, static_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_query_grouped(gemm_handle_t h, const gemm_group_problem_t *problems, int64_t count,
                                 gemm_dtype_t dtype, gemm_sched_t sched, gemm_launch_info_t *info)
{
    if (h == nullptr || info == nullptr) return GEMM_ERR_INVALID_ARG;
    if (cudaSetDevice(h->device) != cudaSuccess) return cuda_fail(cudaErrorInvalidDevice);
    GroupedPlan gp;
    gemm_status_t st = plan_grouped(h, problems, count, dtype, sched, false, gp);
    if (st != GEMM_OK) return st;
    const Plan &pl = gp.pl;
    std::memset(info, 0, sizeof(*info));
    info->tile_m = pts::kRowsPerCta * pl.cg;
    info->tile_n = pts::kTileN;
    info->tile_k = dtype == GEMM_E4M3 ? 128 : 64;
    info->cta_group = pl.cg;
    info->stages = pl.stages;
    info->tiles = pl.tiles;
    info->grid_ctas = pl.tiles == 0 ? 0 : pl.grid_ctas;
    info->max_active_clusters = pl.max_active_clusters;
    info->ctas_per_sm = pl.ctas_per_sm;
    info->smem_bytes = pl.smem;
    info->threads = pts::kThreads;
    info->split = 1;
    info->work_items = pl.work;
    info->units = pl.units;
    return GEMM_OK;
}

gemm_status_t gemm_check(gemm_handle_t h, void *stream, int *device_status)
{
    if (h == nullptr) return GEMM_ERR_INVALID_ARG;
    return read_status(h, static_cast<cudaStream_t>(stream), device_status);
}

gemm_status_t gemm_read_debug(gemm_handle_t h, void *stream, gemm_tile_record_t *records, int64_t n_work,
                              int *device_status)
{
    if (h == nullptr || n_work < 0 || (n_work > 0 && records == nullptr)) return GEMM_ERR_INVALID_ARG;
    if (!(h->opts.debug_flags & GEMM_DEBUG_RECORDS) || n_work > h->records_cap || n_work != h->last_work)
        return GEMM_ERR_INVALID_ARG;
    static_assert(sizeof(gemm_tile_record_t) == sizeof(pts::TileRecord), "record layout");
    gemm_status_t st = read_status(h, static_cast<cudaStream_t>(stream), device_status);
    if (n_work > 0 && cudaMemcpy(records, h->d_records, size_t(n_work) * sizeof(gemm_tile_record_t),
                                 cudaMemcpyDeviceToHost) != cudaSuccess)
        return cuda_fail(cudaErrorUnknown);
    if (st != GEMM_OK) return st;
    // every work item stored by each CTA of its cluster once; the unused
    // record slots of stream-K units with fewer than 3 pieces never
    const int64_t U = h->last_sk_units, L = h->last_sk_tiles * h->last_num_kb;
    for (int64_t t = 0; t < n_work; ++t) {
        bool used = true;
        if (U > 0 && t < pts::kSkMaxPieces * U)
            used = t % pts::kSkMaxPieces < pts::sk_pieces(t / pts::kSkMaxPieces, L, U, h->last_num_kb);
        if (records[t].visits != (used ? static_cast<uint32_t>(h->last_cta_group) : 0u)) return GEMM_ERR_COVERAGE;
    }
    return GEMM_OK;
}

gemm_status_t gemm_destroy(gemm_handle_t h)
{
    if (h == nullptr) return GEMM_OK;
    cudaSetDevice(h->device);
    cudaFree(h->d_status);
    cudaFree(h->d_records);
    cudaFree(h->d_host_bufs);
    cudaFree(h->d_ws_partial);
    cudaFree(h->d_ws_sync);
    for (int b = 0; b < kBatchSlots; ++b) {
        cudaFree(h->d_slot[b]);
        if (h->ev_in[b]) cudaEventDestroy(h->ev_in[b]);
        if (h->ev_comp[b]) cudaEventDestroy(h->ev_comp[b]);
        if (h->ev_free[b]) cudaEventDestroy(h->ev_free[b]);
    }
    if (h->ev_entry) cudaEventDestroy(h->ev_entry);
    for (int b = 0; b < kGroupSlots; ++b) {
        cudaFreeHost(h->tab_host[b]);
        cudaFree(h->tab_dev[b]);
        if (h->ev_tab[b]) cudaEventDestroy(h->ev_tab[b]);
    }
    if (h->s_h2d) cudaStreamDestroy(h->s_h2d);
    for (cudaStream_t s : h->s_d2h)
        if (s) cudaStreamDestroy(s);
    delete h;
    return GEMM_OK;
}

}  // extern "C"
