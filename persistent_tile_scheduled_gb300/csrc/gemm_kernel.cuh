// Persistent, tile-scheduled GEMM kernel for sm_103a.
//
//   C[M x N] = A[M x K] . B[N x K]^T      (fp32 accumulation in TMEM)
//
// One CTA (CG = 1) or one CTA pair (CG = 2, tcgen05 cta_group::2) computes a
// (128*CG) x BN output tile at a time (BN = 256, or 128 for the narrow tile).
// Warp roles:
//   warp 0     producer: TMA loads of A and B k-blocks into an S-stage
//              shared-memory ring guarded by full/empty mbarriers (one k-block
//              per stage for a single CTA, two for a pair)
//   warp 1     MMA issuer (the leader CTA's warp, lane 0 issuing): tcgen05.mma
//              into one of two 256-column TMEM accumulators, so the epilogue
//              of item i overlaps the mainloop of item i+1
//   warps 2-5  epilogue: tcgen05.ld -> (scale) -> fp16/bf16 -> swizzled
//              shared-memory staging -> TMA store; for a tile cut in two by
//              the stream-K share, the fp32 partial fixup
//   warp 6     scheduler (the leader CTA's): static arithmetic or Cluster
//              Launch Control; it takes units, splits each into its work
//              items, decodes them and publishes them into a small broadcast
//              ring read by every other role
// The producer, MMA and scheduler warps run their loops with all 32 lanes in
// step and issue through predicated instructions from lane 0.
//
// Scheduling follows "Persistent Kernels with Cluster Launch Control": a
// static scheduler derives later units in software (u, u+G, u+2G, ...); a CLC
// scheduler asks the hardware to cancel a not-yet-launched cluster of the same
// grid and takes that cluster's id as its next unit, never asking again after
// one failed request.  The non-persistent mode runs exactly one unit per
// cluster ("question about persistent kernel concept": a thread block per tile).
// A unit is a whole tile, a column slice of one (below one wave, or a half of
// a tile of a partial last wave), or a stream-K unit's pieces (see
// work_tile()).
//
// Every mbarrier wait is bounded: on time-out the kernel records an error in
// the device status block, tells every role (and the peer CTA) to stop, drains
// its own copies in flight, frees TMEM and returns.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gemm_params.h"
#include "ptx.cuh"

namespace pts {

enum : int32_t {
    WHERE_EMPTY = 1,        // producer waiting for a free stage
    WHERE_FULL = 2,         // MMA waiting for a loaded stage
    WHERE_ACC_EMPTY = 3,    // MMA waiting for a drained accumulator
    WHERE_ACC_FULL = 4,     // epilogue waiting for a finished accumulator
    WHERE_RING_EMPTY = 5,   // scheduler waiting for a free broadcast slot
    WHERE_RING_FULL = 6,    // a role waiting for the next work item id
    WHERE_CLC = 7,          // scheduler waiting for a CLC response
    WHERE_BAD_TILE = 8,     // a CLC response named a cluster outside the grid
    WHERE_FIXUP = 9,        // the second piece of a cut tile waiting for the first's partial
    WHERE_STARTED = 10,     // CLC scheduler waiting for the producer to start an item it published
};

__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v)
{
    asm volatile("st.volatile.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.volatile.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// tcgen05 shared-memory matrix descriptor for a K-major operand laid out by
// TMA with the 128-byte swizzle: rows of 128 bytes, groups of 8 rows 1024
// bytes apart (stride byte offset), leading byte offset unused (set to 16 B),
// descriptor version 1, swizzle mode 2 (128 B).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr)
{
    return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (1ull << 16) | (64ull << 32) | (1ull << 46)
           | (2ull << 61);
}

// tcgen05 instruction descriptor: fp32 D (bits 4-5 = 1), A/B formats at bits
// 7-9 / 10-12 (kind::f16: fp16 0, bf16 1; kind::f8f6f4: e4m3 0), both
// operands K-major (bits 15/16 = 0), N >> 3 at bits 17-22, M >> 4 at 24-28.
template <int KIND, int CG>
__host__ __device__ constexpr uint32_t make_idesc(uint32_t n)
{
    constexpr uint32_t fmt = (KIND == 1) ? 1u : 0u;
    constexpr uint32_t m = 128u * CG;
    return (1u << 4) | (fmt << 7) | (fmt << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

// Work id -> (tile-row, tile-col) in GROUP_SIZE_M-grouped order: ids walk down
// a group of at most group_m tile-rows one column at a time.
__device__ __forceinline__ void tile_of(int w, int tiles_m, int tiles_n, int group_m, int &tm, int &tn)
{
    const int per_group = group_m * tiles_n;
    const int g = w / per_group;
    const int first = g * group_m;
    const int rows = min(tiles_m - first, group_m);
    const int r = w - g * per_group;
    tm = first + r % rows;
    tn = r / rows;
}

// A work item: tile (tm, tn) of problem g (0 unless the launch is grouped),
// idx = tm * tiles_n + tn, its column slice [n_off, n_off + n_len), its
// k-block range [kb_begin, kb_end), and for a stream-K piece of a tile that
// is cut in two, the tile's index in the stream-K region (ks; else -1).
struct WorkTile {
    int tm, tn, n_off, n_len, kb_begin, kb_end, ks, g, idx;
};

// Problem of work id w in a grouped launch: the g with group_start[g] <= w <
// group_start[g + 1] (problems without tiles have equal bounds and are never
// the answer).  Called by a whole converged warp: each round the 32 lanes
// test 32 evenly spaced bounds at once and keep the interval between the
// last bound at or below w and the next one, so 1024 problems take two
// rounds of one load per lane.
__device__ __forceinline__ int group_of(int w, const GemmParams &p)
{
    int lo = 0, hi = p.num_groups;   // group_start[lo] <= w < group_start[hi]
    while (hi - lo > 1) {
        const int step = (hi - lo + 31) / 32;
        const int idx = lo + static_cast<int>(lane_id()) * step;
        const bool below = idx < hi && __ldg(p.group_start + idx) <= w;
        const uint32_t b = __ballot_sync(0xffffffffu, below);   // lane 0 always set
        lo += (31 - __clz(b)) * step;
        hi = min(hi, lo + step);
    }
    return lo;
}

// Work item (record slot) s.
//  - With a stream-K region (sk_units = U > 0): s < 3U is piece s % 3 of
//    unit s / 3, the part of the unit's k-block range inside its (s % 3)-th
//    tile (only slots of pieces that exist are handed out); s >= 3U is the
//    whole tile sk_tiles + s - 3U.
//  - With column slices (split 2 or 4): slice s % split of tile s / split.
//  - With tail halves (tail_tiles = R > 0): s < T - R is the whole tile s;
//    s = T - R + j is the column half j % 2 of tile T - R + j / 2.
//  - Otherwise the whole tile s.
// Tiles are numbered in grouped order (tile_of).  (A grouped launch's items
// are decoded by the scheduler warp, which caches its problem table.)
template <int BN>
__device__ __forceinline__ WorkTile work_tile(int s, const GemmParams &p)
{
    WorkTile t;
    int tile = s;
    t.n_off = 0;
    t.n_len = BN;
    t.kb_begin = 0;
    t.kb_end = p.num_kb;
    t.ks = -1;
    t.g = 0;
    if (p.sk_units > 0) {
        const int U = p.sk_units;
        if (s < kSkMaxPieces * U) {
            const int64_t L = static_cast<int64_t>(p.sk_tiles) * p.num_kb;
            const int c = s / kSkMaxPieces;
            const int j = s - c * kSkMaxPieces;
            const int64_t a = sk_unit_begin(c, L, U), b = sk_unit_begin(c + 1, L, U);
            tile = static_cast<int>(a / p.num_kb) + j;
            const int64_t t0 = static_cast<int64_t>(tile) * p.num_kb;
            t.kb_begin = static_cast<int>((a > t0 ? a : t0) - t0);
            t.kb_end = static_cast<int>((b < t0 + p.num_kb ? b : t0 + p.num_kb) - t0);
            // cut in two when its first and last k-blocks belong to different units
            if (sk_unit_of(t0, L, U) != sk_unit_of(t0 + p.num_kb - 1, L, U)) t.ks = tile;
        } else {
            tile = p.sk_tiles + (s - kSkMaxPieces * U);
        }
    } else if (p.split > 1) {
        tile = s / p.split;
        const int h = s - tile * p.split;
        t.n_len = BN / p.split;
        t.n_off = h * t.n_len;
    } else if (p.tail_tiles > 0 && s >= p.num_tiles - p.tail_tiles) {
        const int j = s - (p.num_tiles - p.tail_tiles);
        tile = p.num_tiles - p.tail_tiles + j / 2;
        t.n_len = BN / 2;
        t.n_off = (j & 1) * t.n_len;
    }
    tile_of(tile, p.tiles_m, p.tiles_n, p.group_m, t.tm, t.tn);
    t.idx = t.tm * p.tiles_n + t.tn;
    return t;
}

// Pieces of unit u (the work ids the schedulers hand out): 1 to 3 for a
// stream-K unit (one per tile its k-block range touches), else 1.
__device__ __forceinline__ int unit_items(int u, const GemmParams &p)
{
    if (p.sk_units > 0 && u < p.sk_units)
        return sk_pieces(u, static_cast<int64_t>(p.sk_tiles) * p.num_kb, p.sk_units, p.num_kb);
    return 1;
}

// Work item that unit u (of `pieces` pieces) runs j-th.  A stream-K unit
// runs its pieces last tile first: every unit then starts at k-block 0 of a
// tile, as whole tiles do, so clusters that share A rows or B columns read
// the same k-blocks at the start and find them in L2.  (Its first piece also
// finishes early and its last late, so the early piece of a cut tile writes
// the partial and the late one, followed by whole tiles, adds it.)
__device__ __forceinline__ int unit_item(int u, int j, int pieces, const GemmParams &p)
{
    if (p.sk_units > 0)
        return u < p.sk_units ? u * kSkMaxPieces + (pieces - 1 - j) : kSkMaxPieces * p.sk_units + (u - p.sk_units);
    return u;
}

// Stream-K fixup, per (cut tile, CTA of the pair, epilogue warp): the warp's
// 32 rows of the tile are reduced independently of the other warps, so no
// warp ever waits for another warp of its CTA.  Sync words: [0] claim counter
// (pieces claimed so far), [1 .. kSkMaxParts - 1] ready flags of the partial
// slots (1 = filled).  A cut tile has kSkMaxParts pieces and kSkMaxParts - 1
// partial slots.  Every launch finds the words at zero and leaves them at
// zero: the last piece to claim, once it has seen every flag raised, is the
// only one of the launch still to touch them and resets them.  Nothing the
// host passes in tags them, so a launch captured in a CUDA graph and replayed
// behaves exactly like a fresh one.  (A launch that stops on a device error
// may leave them set; reading that error through the handle clears them.)
// Partial slot layout: float4 index (chunk * 16 + g) * 32 + lane, so every
// warp-wide access is 512 contiguous bytes.
constexpr int kPartialFloat4PerWarp = kEpiRowsPerWarp * kTileN / 4;

struct WaitCtl {
    uint32_t abort_addr;       // this CTA's abort flag (shared::cta)
    uint32_t peer_abort;       // the peer's abort flag (shared::cluster), 0 if none
    uint64_t timeout_ns;
    int32_t *status;

    // Record a failure and tell this CTA (and its peer) to stop.  Called by
    // every lane of a converged warp, it acts once: in lane 0.
    __device__ void fail(int32_t where) const
    {
        if (lane_id() != 0) return;
        if (atomicCAS(status, 0, DEV_ERR_TIMEOUT) == 0) {
            status[1] = where;
            status[2] = static_cast<int32_t>(blockIdx.x);
        }
        atomicAdd(status + 3, 1);
        st_shared_u32(abort_addr, 1u);
        if (peer_abort) st_cluster_u32(peer_abort, 1u);
    }

    // Wait for phase `parity` of `bar`.  False when this CTA was told to stop
    // or the wait ran past the time limit (which is then recorded).
    __device__ bool wait(uint32_t bar, uint32_t parity, int32_t where) const
    {
        if (mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t n = 1;; ++n) {
            if (mbar_try_wait(bar, parity)) return true;
            if ((n & 15u) == 0) {
                if (ld_shared_u32(abort_addr)) return false;
                if (globaltimer_ns() - t0 > timeout_ns) {
                    fail(where);
                    return false;
                }
            }
        }
    }

    // The same for a whole converged warp: every lane waits (each wait is
    // bounded, so every lane reaches the vote) and all get one answer, so
    // the warp never splits on a wait's outcome.
    __device__ bool wait_all(uint32_t bar, uint32_t parity, int32_t where) const
    {
        const bool mine = wait(bar, parity, where);
        const bool all = __all_sync(0xffffffffu, mine);
        if (!all && mine && lane_id() == 0 && !ld_shared_u32(abort_addr)) fail(where);
        return all;
    }

    // Wait until the shared word at `addr` holds at least `target` (a count
    // another warp of this CTA raises), bounded like wait(); every lane of a
    // converged warp polls and all get one answer.
    __device__ bool wait_count_all(uint32_t addr, int target, int32_t where) const
    {
        bool mine = static_cast<int>(ld_shared_u32(addr)) >= target;
        if (!mine) {
            const uint64_t t0 = globaltimer_ns();
            for (uint32_t n = 1;; ++n) {
                if (static_cast<int>(ld_shared_u32(addr)) >= target) {
                    mine = true;
                    break;
                }
                if ((n & 15u) == 0) {
                    if (ld_shared_u32(abort_addr)) break;
                    if (globaltimer_ns() - t0 > timeout_ns) {
                        fail(where);
                        break;
                    }
                }
            }
        }
        const bool all = __all_sync(0xffffffffu, mine);
        if (!all && mine && lane_id() == 0 && !ld_shared_u32(abort_addr)) fail(where);
        return all;
    }

    // Bounded wait used only while shutting down after an error: ignores the
    // abort flag, gives up silently after `limit_ns`.
    __device__ bool drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) const
    {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar, parity))
            if (globaltimer_ns() - t0 > limit_ns) return false;
        return true;
    }
};

template <int KIND>
__device__ __forceinline__ uint32_t pack2(uint32_t lo_bits, uint32_t hi_bits, float scale)
{
    float lo = __uint_as_float(lo_bits), hi = __uint_as_float(hi_bits);
    if constexpr (KIND == 2) {
        lo *= scale;
        hi *= scale;
    }
    if constexpr (KIND == 0) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    } else {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
}

template <int KIND, int CG, int BN = kTileN, bool FULL = true>
__global__ void __launch_bounds__(kThreads, ctas_per_sm(CG, BN))
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmB4,
                const __grid_constant__ CUtensorMap tmC, const GemmParams p)
{
    // BN: tile columns, 256 (the wide tile, one CTA per SM) or 128 (the
    // narrow tile: single CTAs two per SM, or CTA pairs one per SM; no
    // stream-K share and no column quarters, so its epilogue holds fewer
    // registers).
    // tmB / tmB2 / tmB4: B boxes of BN/CG, BN/CG/2 and BN/CG/4 rows, for whole
    // tiles and for the column slices (halves, quarters) of a problem smaller
    // than one wave or of the tiles of a partial last wave (halves)
    // FULL = false: the common launch -- one problem, no debug records, the
    // TMA-store epilogue, no L2 prefetch, no test hooks -- with the code of
    // those features compiled out.  Less code to fetch at the start of a
    // launch: measured on GB300, fp16 4096^2 x 128 took 10.9 instead of 11.9 us
    // per chained launch and 14.3 instead of 16.3 us alone.
    static_assert(BN == kTileN || BN == kTileNNarrow, "tile shape");
    constexpr bool kStreamK = BN == kTileN;   // the stream-K fixup is built for the wide tile only
    constexpr uint32_t kAccCols = 2 * BN;     // TMEM columns: two accumulators
    constexpr int KBS = kb_per_stage(CG);   // k-blocks per ring stage
    constexpr int SA = stage_bytes_a(CG);
    constexpr int SB = stage_bytes_b(CG, BN);
    constexpr int KELEMS = (KIND == 2) ? kKBlockBytes : kKBlockBytes / 2;   // K elements per k-block

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const int S = p.stages;
    const uint32_t sA = base;
    const uint32_t sB = sA + S * SA;
    const uint32_t sEpi = sB + S * SB;
    const uint32_t bar0 = sEpi + epi_bytes();
    const uint32_t full0 = bar0;                             // + 8*s
    const uint32_t empty0 = bar0 + 8 * kMaxStages;           // + 8*s
    const uint32_t acc_full0 = bar0 + 16 * kMaxStages;       // + 8*b
    const uint32_t acc_empty0 = acc_full0 + 16;              // + 8*b
    const uint32_t ring_full0 = acc_empty0 + 16;             // + 8*r
    const uint32_t ring_empty0 = ring_full0 + 8 * kRing;     // + 8*r
    const uint32_t clc_bar = ring_empty0 + 8 * kRing;
    const uint32_t started_bar = clc_bar + 8;                // producer (leader) starts an item
    const uint32_t clc_resp = (started_bar + 8 + 15) & ~15u;
    const uint32_t ring0 = clc_resp + 16;                    // + 4*kRingWords*r: a decoded work item
    const uint32_t tmem_slot = ring0 + 4 * kRingWords * kRing;
    const uint32_t abort_flag = tmem_slot + 4;
    const uint32_t started_cnt = tmem_slot + 8;              // items the (leader's) producer has started

    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = lane_id();
    const uint32_t rank = (CG == 2) ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    const int cluster_id = static_cast<int>(blockIdx.x) / CG;
    const int num_clusters = static_cast<int>(gridDim.x) / CG;

    WaitCtl ctl;
    ctl.abort_addr = abort_flag;
    ctl.peer_abort = (CG == 2) ? mapa(abort_flag, rank ^ 1u) : 0u;
    ctl.timeout_ns = p.timeout_ns;
    ctl.status = p.status;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full0 + 8 * b, 1);
            mbar_init(acc_empty0 + 8 * b, kEpiWarps * CG);
        }
        for (int r = 0; r < kRing; ++r) {
            mbar_init(ring_full0 + 8 * r, 1);
            // readers: the producer, MMA and epilogue warps of the leader, the
            // producer and epilogue warps of the peer
            mbar_init(ring_empty0 + 8 * r, CG == 1 ? 2 + kEpiWarps : 3 + 2 * kEpiWarps);
        }
        mbar_init(clc_bar, 1);
        mbar_init(started_bar, 1);
        st_shared_u32(started_cnt, 0u);
        st_shared_u32(abort_flag, 0u);
        fence_mbar_init();
    }
    const bool grouped = FULL && p.num_groups > 0;
    if (warp == 0 && lane == 0 && !grouped) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        if (p.split == 2 || p.tail_tiles > 0) prefetch_tmap(&tmB2);
        if (p.split == 4) prefetch_tmap(&tmB4);
        prefetch_tmap(&tmC);
    }
    if (warp == 1) {
        tmem_alloc<CG>(tmem_slot, kAccCols);
        tmem_relinquish<CG>();
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (CG == 2) cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = ld_shared_u32(tmem_slot);
    const uint32_t one = lane == 0 ? 1u : 0u;

    // Rows of this CTA's A and B boxes for work item t, its A map, and the B
    // map of the item's column width (a grouped launch: its problem's maps).
    auto boxes = [&](const WorkTile &t, int &ya, int &yb, const CUtensorMap *&ma) -> const CUtensorMap * {
        ya = t.tm * (kRowsPerCta * CG) + static_cast<int>(rank) * kRowsPerCta;
        yb = t.tn * BN + t.n_off + static_cast<int>(rank) * (t.n_len / CG);
        if (grouped) {
            ma = &p.groups[t.g].tmA;
            return &p.groups[t.g].tmB;
        }
        ma = &tmA;
        return t.n_len == BN ? &tmB : (t.n_len == BN / 2 ? &tmB2 : &tmB4);
    };

    // Back-to-back launches: the set-up above may overlap the end of the
    // previous grid in the stream; no load or store of A, B or C happens
    // before it has completed (A and B may be its outputs, C its inputs).
    // Before waiting, the producer asks L2 for the first k-blocks of its
    // cluster's first unit: an L2 prefetch brings lines into the coherent L2
    // and changes nothing any load returns, so the first stages then fill
    // from L2 instead of HBM.
    // (Not in a grouped launch, whose problem table is read only after the wait.)
    pdl_launch_dependents();
    if (warp == 0 && cluster_id < p.num_units && !grouped) {
        const WorkTile t0 = work_tile<BN>(unit_item(cluster_id, 0, unit_items(cluster_id, p), p), p);
        int ya, yb;
        const CUtensorMap *ma;
        const CUtensorMap *mb = boxes(t0, ya, yb, ma);
        const int kb_end = t0.kb_end < t0.kb_begin + S ? t0.kb_end : t0.kb_begin + S;
        for (int kb = t0.kb_begin; kb < kb_end; ++kb) {
            tma_prefetch_2d(one, ma, kb * KELEMS, ya);
            tma_prefetch_2d(one, mb, kb * KELEMS, yb);
        }
    }
    // The scheduler warp of a single-problem launch waits only after it has
    // published its first item (its decode reads no global memory), so the
    // producers find that item in the ring when their own wait returns.
    if (grouped || warp != kSchedWarp) pdl_wait();

    // ---- work-item broadcast ring -----------------------------------------
    // Slot r holds work item i (i % kRing == r), decoded: its id w (the
    // record slot; -1 = no more) and its WorkTile.  publish is called by the
    // whole scheduler warp, ring_read by whole converged warps (producer, MMA)
    // or by lane 0 of an epilogue warp; the slot writes and the arrivals
    // happen in lane 0.
    auto publish = [&](int i, int w, const WorkTile &t) -> bool {
        const int slot = i % kRing;
        if (i >= kRing && !ctl.wait_all(ring_empty0 + 8 * slot, ((i / kRing) & 1) ^ 1, WHERE_RING_EMPTY))
            return false;
        if (lane == 0) {
            const uint32_t a = ring0 + 4 * kRingWords * slot;
            const uint32_t v[12] = {static_cast<uint32_t>(w),        static_cast<uint32_t>(t.g),
                                    static_cast<uint32_t>(t.tm),     static_cast<uint32_t>(t.tn),
                                    static_cast<uint32_t>(t.n_off),  static_cast<uint32_t>(t.n_len),
                                    static_cast<uint32_t>(t.kb_begin), static_cast<uint32_t>(t.kb_end),
                                    static_cast<uint32_t>(t.ks),     static_cast<uint32_t>(t.idx), 0u, 0u};
#pragma unroll
            for (int q = 0; q < 3; ++q) {
                st_shared_v4(a + 16 * q, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                if constexpr (CG == 2)
                    st_cluster_v4(mapa(a + 16 * q, 1u), v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            }
            if constexpr (CG == 2) mbar_arrive_cluster(mapa(ring_full0 + 8 * slot, 1u));
            mbar_arrive(ring_full0 + 8 * slot);
        }
        __syncwarp();
        return true;
    };
    auto ring_read = [&](int i, int &w, WorkTile &t, bool whole_warp) -> bool {
        const int slot = i % kRing;
        const uint32_t par = (i / kRing) & 1;
        if (!(whole_warp ? ctl.wait_all(ring_full0 + 8 * slot, par, WHERE_RING_FULL)
                         : ctl.wait(ring_full0 + 8 * slot, par, WHERE_RING_FULL)))
            return false;
        const uint32_t a = ring0 + 4 * kRingWords * slot;
        const uint4 v0 = ld_shared_v4(a), v1 = ld_shared_v4(a + 16), v2 = ld_shared_v4(a + 32);
        w = static_cast<int>(v0.x);
        t.g = static_cast<int>(v0.y);
        t.tm = static_cast<int>(v0.z);
        t.tn = static_cast<int>(v0.w);
        t.n_off = static_cast<int>(v1.x);
        t.n_len = static_cast<int>(v1.y);
        t.kb_begin = static_cast<int>(v1.z);
        t.kb_end = static_cast<int>(v1.w);
        t.ks = static_cast<int>(v2.x);
        t.idx = static_cast<int>(v2.y);
        if (CG == 2 && !leader)
            mbar_arrive_cluster_if(one, mapa(ring_empty0 + 8 * slot, 0u));
        else
            mbar_arrive_if(one, ring_empty0 + 8 * slot);
        return true;
    };

    if (warp == 0) {
        // =============================== producer ==============================
        // All 32 lanes run this loop in step (every branch below is uniform
        // across the warp); lane 0 issues the loads.  Work items come from
        // the broadcast ring; on the leader CTA, the producer tells the
        // scheduler warp when it starts each one.
        int stage = 0;
        uint32_t phase = 0;
        long long issued = 0;
        bool ok = true;
        int maps_of = -1;   // grouped launch: the problem whose A and B maps this thread last acquired
        // Load k-blocks [kb_from, kb_to) of work item t (kb_from is the
        // item's first k-block or a stage boundary after it).
        auto load_tile = [&](const WorkTile &t, int kb_from, int kb_to) -> bool {
            int ya, yb;
            const CUtensorMap *ma;
            const CUtensorMap *mb = boxes(t, ya, yb, ma);
            if (grouped && t.g != maps_of) {
                tmap_acquire(one, ma);
                tmap_acquire(one, mb);
                maps_of = t.g;
            }
            // a stage holds KBS k-blocks (the last stage of an item may hold fewer)
            for (int kb = kb_from; kb < kb_to; kb += KBS) {
                if (!ctl.wait_all(empty0 + 8 * stage, phase ^ 1u, WHERE_EMPTY)) return false;
                const int nk = t.kb_end - kb < KBS ? t.kb_end - kb : KBS;
                const uint32_t tx =
                    static_cast<uint32_t>(CG * nk * (SA / KBS + (t.n_len / CG) * kKBlockBytes));
                const uint32_t fb = full0 + 8 * stage;
                // test hook: announce the stage's bytes but never load them,
                // so the MMA warp's bounded wait on this stage runs out
                const bool skip = FULL && (p.debug_flags & DBG_FAULT_SKIP_TMA) && issued == p.fault_arg;
                const uint32_t go = skip ? 0u : one;
                if constexpr (CG == 1) {
                    mbar_arrive_expect_tx_if(one, fb, tx);
                    for (int j = 0; j < nk; ++j) {
                        tma_load_2d(go, sA + stage * SA + j * (SA / KBS), ma, fb, (kb + j) * KELEMS, ya);
                        tma_load_2d(go, sB + stage * SB + j * (SB / KBS), mb, fb, (kb + j) * KELEMS, yb);
                    }
                } else {
                    mbar_arrive_expect_tx_if(leader ? one : 0u, fb, tx);
                    const uint32_t fbc = mapa(fb, 0u);
                    for (int j = 0; j < nk; ++j) {
                        tma_load_2d_pair(go, sA + stage * SA + j * (SA / KBS), ma, fbc, (kb + j) * KELEMS, ya);
                        tma_load_2d_pair(go, sB + stage * SB + j * (SB / KBS), mb, fbc, (kb + j) * KELEMS, yb);
                    }
                }
                // keep the k-block prefetch_kb ahead of this one on its way into
                // L2, so that a stage rarely waits on an HBM miss
                const int kp = kb + p.prefetch_kb;
                if (FULL && p.prefetch_kb > 0 && kp < t.kb_end) {
                    tma_prefetch_2d(one, ma, kp * KELEMS, ya);
                    tma_prefetch_2d(one, mb, kp * KELEMS, yb);
                }
                ++issued;
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            return true;
        };

        for (int i = 0;; ++i) {
            int w;
            WorkTile t;
            if (!ring_read(i, w, t, true)) {
                ok = false;
                break;
            }
            if (w < 0) break;
            if (leader) {
                mbar_arrive_if(one, started_bar);
                if (lane == 0) st_shared_u32(started_cnt, static_cast<uint32_t>(i + 1));
            }
            if (!load_tile(t, t.kb_begin, t.kb_end)) {
                ok = false;
                break;
            }
        }
        if (!ok) {
            // Stopped early: let the loads already issued land before the
            // CTA can exit (bounded).  The leader drains the full barriers of
            // its last stages, on which both CTAs' loads of those stages
            // complete.  The peer may have issued a stage the leader never
            // armed (the leader stopped first): that load completes on a
            // leader barrier whose phase can no longer finish, so nothing can
            // be waited on for it, and the peer instead lets a bounded 1 ms
            // pass, far longer than any load takes, before it goes on to the
            // teardown barrier.
            if (CG == 1 || leader) {
                const long long n = issued < S ? issued : S;
                for (long long j = 0; j < n; ++j) {
                    const long long g = issued - 1 - j;
                    ctl.drain(full0 + 8 * static_cast<int>(g % S), static_cast<uint32_t>((g / S) & 1),
                              10000000ull);
                }
            } else if (issued > 0) {
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 1000000ull) {
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================================ MMA ==================================
        // The leader CTA's whole warp runs the loop in step; lane 0 issues
        // the MMAs and the commits (a commit tracks the MMAs of its own lane).
        if (leader) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            int last_stage = -1;
            uint32_t last_phase = 0;
            for (int i = 0;; ++i) {
                int w;
                WorkTile t;
                if (!ring_read(i, w, t, true) || w < 0) break;
                if (!ctl.wait_all(acc_empty0 + 8 * acc, acc_phase ^ 1u, WHERE_ACC_EMPTY)) break;
                tc_fence_after();
                if (FULL && p.records != nullptr && lane == 0)
                    p.records[w].t_mma_start = static_cast<uint32_t>(globaltimer_ns());
                const uint32_t idesc = make_idesc<KIND, CG>(static_cast<uint32_t>(t.n_len));
                const uint32_t d = tmem_base + static_cast<uint32_t>(acc * BN);
                bool ok = true;
                for (int kb = t.kb_begin; kb < t.kb_end; kb += KBS) {
                    if (!ctl.wait_all(full0 + 8 * stage, phase, WHERE_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int nk = t.kb_end - kb < KBS ? t.kb_end - kb : KBS;
#pragma unroll
                    for (int j = 0; j < KBS; ++j) {
                        if (j >= nk) break;
                        const uint64_t ad = smem_desc_sw128(sA + stage * SA + j * (SA / KBS));
                        const uint64_t bd = smem_desc_sw128(sB + stage * SB + j * (SB / KBS));
#pragma unroll
                        for (int k = 0; k < 4; ++k)   // 32 bytes of K per instruction
                            umma<KIND, CG>(one, d, ad + 2 * k, bd + 2 * k, idesc,
                                           (kb + j != t.kb_begin || k != 0) ? 1u : 0u);
                    }
                    umma_commit<CG>(one, empty0 + 8 * stage, 0x3);
                    last_stage = stage;
                    last_phase = phase;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit<CG>(one, acc_full0 + 8 * acc, 0x3);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // the last stage release is the last asynchronous arrival this
            // warp caused; see it land before the CTA may exit
            if (last_stage >= 0) ctl.drain(empty0 + 8 * last_stage, last_phase, 10000000ull);
        }
        __syncwarp();
    } else if (warp < 2 + kEpiWarps) {
        // ============================== epilogue ===============================
        const uint32_t e = warp - 2;          // staging buffer owner index
        const uint32_t q = warp & 3u;         // TMEM lane quarter this warp may access
        const uint32_t stage_base = sEpi + e * (kEpiBufsPerWarp * kEpiBufBytes);
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t nstore = 0;
        int maps_of = -1;   // the problem whose C map this warp's lane 0 has acquired (grouped launch)
        for (int i = 0;; ++i) {
            int w = 0;
            WorkTile t{};
            int ok = 1;
            if (lane == 0) ok = ring_read(i, w, t, false) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            w = __shfl_sync(0xffffffffu, w, 0);
            if (!ok || w < 0) break;
            t.g = __shfl_sync(0xffffffffu, t.g, 0);
            t.tm = __shfl_sync(0xffffffffu, t.tm, 0);
            t.tn = __shfl_sync(0xffffffffu, t.tn, 0);
            t.n_off = __shfl_sync(0xffffffffu, t.n_off, 0);
            t.n_len = __shfl_sync(0xffffffffu, t.n_len, 0);
            t.kb_begin = __shfl_sync(0xffffffffu, t.kb_begin, 0);
            t.kb_end = __shfl_sync(0xffffffffu, t.kb_end, 0);
            t.ks = __shfl_sync(0xffffffffu, t.ks, 0);
            t.idx = __shfl_sync(0xffffffffu, t.idx, 0);
            const int g = t.g;
            // the item's output: its problem's C map, sizes and scale
            const CUtensorMap *mc = &tmC;
            int cM = p.M, cN = p.N;
            float oscale = p.out_scale;
            if (grouped) {
                const GroupDesc *d = p.groups + g;
                mc = &d->tmC;
                cM = __ldg(&d->M);
                cN = __ldg(&d->N);
                oscale = __ldg(&d->out_scale);
                if (g != maps_of) {
                    tmap_acquire(one, mc);
                    maps_of = g;
                }
            }
            // K = 0 (a grouped launch's empty problem): nothing was accumulated,
            // the tile is the empty sum
            const bool empty_sum = t.kb_begin == t.kb_end;
            if (lane == 0) ok = ctl.wait(acc_full0 + 8 * acc, acc_phase, WHERE_ACC_FULL) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            TileRecord *rec = (FULL && p.records != nullptr && e == 0 && lane == 0) ? p.records + w : nullptr;
            if (rec != nullptr) {
                atomicAdd(&rec->visits, 1u);
                if (leader) {
                    rec->tile = static_cast<uint32_t>(t.idx);
                    rec->group = grouped ? static_cast<uint32_t>(__ldg(&p.groups[g].index)) : 0u;
                    rec->n_off = static_cast<uint32_t>(t.n_off);
                    rec->n_len = static_cast<uint32_t>(t.n_len);
                    rec->kb_begin = static_cast<uint32_t>(t.kb_begin);
                    rec->kb_end = static_cast<uint32_t>(t.kb_end);
                    rec->owner = static_cast<uint32_t>(cluster_id);
                    rec->iter = static_cast<uint32_t>(i);
                    rec->smid = smid();
                    rec->t_acc_full = static_cast<uint32_t>(globaltimer_ns());
                }
            }
            const int row0 = t.tm * (kRowsPerCta * CG) + static_cast<int>(rank) * kRowsPerCta
                             + static_cast<int>(q) * kEpiRowsPerWarp;
            const uint32_t tbase = tmem_base + ((q * 32u) << 16) + static_cast<uint32_t>(acc * BN);
            const int chunks = t.n_len / kEpiChunkCols;

            // A stream-K piece of a cut tile: claim a part number for this
            // warp's rows.  Pieces other than the last claimed write their fp32
            // partial and raise a flag; the last claimed waits for those flags
            // (every such piece has already claimed, so it is past its
            // mainloop and never waits itself) and adds the partials before
            // storing C.
            constexpr int nparts = kSkMaxParts;   // pieces of a cut tile
            int part = -1;
            uint32_t *sync = nullptr;
            const float4 *partials = nullptr;
            if (kStreamK && t.ks >= 0) {
                const long long unit = (static_cast<long long>(t.ks) * CG + rank) * kEpiWarps + q;
                sync = p.ws_sync + unit * 4;
                partials = reinterpret_cast<const float4 *>(p.ws_partial)
                           + unit * (nparts - 1) * kPartialFloat4PerWarp;
                uint32_t mine = 0;
                if (lane == 0) mine = atomicAdd(sync, 1u);
                part = static_cast<int>(__shfl_sync(0xffffffffu, mine, 0));
                if (part == nparts - 1) {
                    uint32_t seen = 1u;
                    if (lane == 0) {
                        for (int sl = 0; sl < nparts - 1 && seen; ++sl) {
                            const uint64_t t0 = globaltimer_ns();
                            while (ld_acquire_gpu(sync + 1 + sl) == 0u) {
                                if (ld_shared_u32(abort_flag)) {
                                    seen = 0u;
                                    break;
                                }
                                if (globaltimer_ns() - t0 > p.timeout_ns) {
                                    ctl.fail(WHERE_FIXUP);
                                    seen = 0u;
                                    break;
                                }
                            }
                        }
                    }
                    seen = __shfl_sync(0xffffffffu, seen, 0);
                    // every lane acquires the raised flags itself before reading the partials
                    for (int sl = 0; sl < nparts - 1; ++sl) (void)ld_acquire_gpu(sync + 1 + sl);
                    __syncwarp();
                    // Every other piece has claimed and raised its flag: no one
                    // else touches these words again in this launch, so they go
                    // back to zero for the next one (which starts only after
                    // this grid has completed).
                    if (lane == 0 && seen) {
                        for (int sl = 0; sl < nparts - 1; ++sl) sync[1 + sl] = 0u;
                        sync[0] = 0u;
                    }
                }
            }
            const bool write_partial = part >= 0 && part < nparts - 1;
            // Chunks of 64 columns.  A TMEM read returns within a few dozen
            // cycles, so each chunk is read when it is needed.  The piece that
            // adds the partial keeps the next chunk's partial sums in flight
            // while the current chunk is converted and stored.
            const float4 *src = part > 0 ? partials + lane : nullptr;   // the one partial slot
            float4 pa[16];
            if (part > 0) {
#pragma unroll
                for (int g = 0; g < 16; ++g) pa[g] = __ldcg(src + g * 32);
            }
#pragma unroll
            for (int c = 0; c < BN / kEpiChunkCols; ++c) {
                if (c >= chunks) break;
                uint32_t v0[32], v1[32];
                tmem_ld_32x32b_x32(tbase + c * kEpiChunkCols, v0);
                tmem_ld_32x32b_x32(tbase + c * kEpiChunkCols + 32, v1);
                tmem_wait_ld();
                if (empty_sum) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v0[j] = v1[j] = 0u;
                }
                if (c + 1 == chunks) {
                    // accumulator fully read: hand it back to the MMA warp
                    tc_fence_before();
                    __syncwarp();
                    if (CG == 2 && !leader)
                        mbar_arrive_cluster_if(one, mapa(acc_empty0 + 8 * acc, 0u));
                    else
                        mbar_arrive_if(one, acc_empty0 + 8 * acc);
                }
                if (write_partial) {
                    float4 *dst = const_cast<float4 *>(partials) + c * 16 * 32 + lane;
#pragma unroll
                    for (int g = 0; g < 8; ++g)
                        __stcg(dst + g * 32, make_float4(__uint_as_float(v0[4 * g]), __uint_as_float(v0[4 * g + 1]),
                                                         __uint_as_float(v0[4 * g + 2]),
                                                         __uint_as_float(v0[4 * g + 3])));
#pragma unroll
                    for (int g = 0; g < 8; ++g)
                        __stcg(dst + (8 + g) * 32,
                               make_float4(__uint_as_float(v1[4 * g]), __uint_as_float(v1[4 * g + 1]),
                                           __uint_as_float(v1[4 * g + 2]), __uint_as_float(v1[4 * g + 3])));
                    continue;
                }
                if (part > 0) {   // the last piece of a cut tile: add the other's partial
#pragma unroll
                    for (int g = 0; g < 8; ++g) {
                        v0[4 * g] = __float_as_uint(__uint_as_float(v0[4 * g]) + pa[g].x);
                        v0[4 * g + 1] = __float_as_uint(__uint_as_float(v0[4 * g + 1]) + pa[g].y);
                        v0[4 * g + 2] = __float_as_uint(__uint_as_float(v0[4 * g + 2]) + pa[g].z);
                        v0[4 * g + 3] = __float_as_uint(__uint_as_float(v0[4 * g + 3]) + pa[g].w);
                        v1[4 * g] = __float_as_uint(__uint_as_float(v1[4 * g]) + pa[8 + g].x);
                        v1[4 * g + 1] = __float_as_uint(__uint_as_float(v1[4 * g + 1]) + pa[8 + g].y);
                        v1[4 * g + 2] = __float_as_uint(__uint_as_float(v1[4 * g + 2]) + pa[8 + g].z);
                        v1[4 * g + 3] = __float_as_uint(__uint_as_float(v1[4 * g + 3]) + pa[8 + g].w);
                    }
                    if (c + 1 < chunks) {   // the next chunk's partial, in flight from here on
#pragma unroll
                        for (int g = 0; g < 16; ++g) pa[g] = __ldcg(src + (c + 1) * 16 * 32 + g * 32);
                    }
                }
                uint32_t pk[32];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    pk[j] = pack2<KIND>(v0[2 * j], v0[2 * j + 1], oscale);
                    pk[16 + j] = pack2<KIND>(v1[2 * j], v1[2 * j + 1], oscale);
                }
                const int col = t.tn * BN + t.n_off + c * kEpiChunkCols;
                if (FULL && p.epi_direct) {
                    // this lane's row: 64 outputs = 8 x 16 bytes, straight to global
                    const int row = row0 + static_cast<int>(lane);
                    if (row < cM) {
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.c_ptr)
                                                               + static_cast<long long>(row) * cN + col);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            if (col + 8 * j < cN)
                                dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                    }
                    continue;
                }
                const uint32_t buf = stage_base + (nstore & 1u) * kEpiBufBytes;
                // the store that used this buffer has read it (only lane 0 has
                // stores in flight; the other lanes return at once)
                bulk_wait_read<1>();
                __syncwarp();
                // row `lane`, 16-byte chunk j stored at chunk j ^ (row % 8): the
                // layout the 128-byte-swizzled tensor map expects
                const uint32_t row_addr = buf + lane * 128u;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    st_shared_v4(row_addr + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4), pk[4 * j],
                                 pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                tma_store_2d_if((row0 < cM && col < cN) ? one : 0u, mc, buf, col, row0);
                bulk_commit();   // (an empty group in lanes 1-31)
                ++nstore;
            }
            if (write_partial) {
                // publish this part: every lane's stores, then the flag (release)
                __threadfence();
                __syncwarp();
                if (lane == 0) st_release_gpu(sync + 1 + part, 1u);
            }
            if (rec != nullptr && leader) rec->t_stored = static_cast<uint32_t>(globaltimer_ns());
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        // the last stores must have read their staging buffers before the
        // CTA's shared memory goes away (their writes to C complete with the
        // grid)
        bulk_wait_read<0>();
        __syncwarp();
    } else if (warp == kSchedWarp) {
        // ============================== scheduler ==============================
        // The leader CTA's whole warp runs this loop in step; lane 0 makes
        // the CLC requests.  It takes units (static arithmetic, CLC, or the
        // cluster's own for the non-persistent grid), splits each into its
        // work items, decodes them and publishes them into the broadcast
        // ring, so no other warp does scheduling or decoding work.  With CLC
        // it publishes item i + 1 only once the producer has started item i,
        // and claims the next unit when the producer starts a unit's first
        // item (as late as the producer's lead allows, so that CLC still
        // balances the last tiles); the unit is decoded while the producer
        // loads.  The static scheduler's units are fixed, so it runs as far
        // ahead as the ring allows.
        if (leader) {
            bool ok = true;
            bool clc_pending = false;
            bool may_request = p.sched == SCHED_CLC;
            uint32_t clc_phase = 0;
            int maps_of = -1;   // grouped launch: the problem whose maps this thread last acquired
            // The unit after `cur` (-1: none): static arithmetic, or the
            // answer to the CLC request made when `cur` started.  False on a
            // failed wait.
            auto next_unit = [&](int cur, int &next) -> bool {
                next = -1;
                if (p.sched == SCHED_STATIC) {
                    next = (cur + num_clusters < p.num_units) ? cur + num_clusters : -1;
                } else if (clc_pending) {
                    if (!ctl.wait_all(clc_bar, clc_phase, WHERE_CLC)) return false;
                    clc_phase ^= 1u;
                    clc_pending = false;
                    // only lane 0 reads the response slot (it alone re-arms it)
                    uint32_t x = 0, got = 0;
                    if (lane == 0) got = clc_decode(clc_resp, x) ? 1u : 0u;
                    got = __shfl_sync(0xffffffffu, got, 0);
                    x = __shfl_sync(0xffffffffu, x, 0);
                    if (got) {
                        next = static_cast<int>(x / CG);
                        if (next >= p.num_units) {   // cannot happen for a well-formed grid
                            ctl.fail(WHERE_BAD_TILE);
                            next = -1;
                        }
                    } else {
                        may_request = false;   // a failed request is never repeated
                    }
                }
                return true;
            };
            // Grouped launch: the next tile belongs to another problem, whose
            // tensor maps and operands are not on chip yet.  Bring its maps
            // (A and B, C) into the descriptor cache and its first stages'
            // k-blocks (both CTAs' boxes) into L2 before the producer needs them.
            auto warm = [&](const WorkTile &t) {
                int ya, yb;
                const CUtensorMap *ma;
                const CUtensorMap *mb = boxes(t, ya, yb, ma);
                const bool has_k = t.kb_end > t.kb_begin;   // (a problem with K = 0 has no A and B maps)
                if (t.g != maps_of && has_k) {
                    tmap_acquire(one, ma);
                    tmap_acquire(one, mb);
                    maps_of = t.g;
                }
                if (lane == 0) {
                    if (has_k) {
                        prefetch_tmap(ma);
                        prefetch_tmap(mb);
                    }
                    prefetch_tmap(&p.groups[t.g].tmC);
                }
                __syncwarp();
                const int kb_end = t.kb_end < t.kb_begin + S * KBS ? t.kb_end : t.kb_begin + S * KBS;
                for (int kb = t.kb_begin; kb < kb_end; ++kb) {
#pragma unroll
                    for (int r = 0; r < CG; ++r) {
                        tma_prefetch_2d(one, ma, kb * KELEMS, ya + r * kRowsPerCta);
                        tma_prefetch_2d(one, mb, kb * KELEMS, yb + r * (t.n_len / CG));
                    }
                }
            };
            // Grouped launch: the problem of the last tile decoded, its tiles
            // [gc_lo, gc_hi) and sizes, so that a tile of the same problem (or
            // of the next one) costs no search and no table read.
            int gc = -1, gc_lo = 0, gc_hi = 0, gc_tm = 0, gc_tn = 0, gc_kb = 0;
            auto item_of = [&](int w) -> WorkTile {
                if (!grouped) return work_tile<BN>(w, p);
                if (w < gc_lo || w >= gc_hi) {
                    int g;
                    if (gc >= 0 && w >= gc_hi && gc + 1 < p.num_groups && w < __ldg(p.group_start + gc + 2))
                        g = gc + 1;
                    else
                        g = group_of(w, p);
                    const GroupDesc *d = p.groups + g;
                    gc = g;
                    gc_lo = __ldg(p.group_start + g);
                    gc_hi = __ldg(p.group_start + g + 1);
                    gc_tm = __ldg(&d->tiles_m);
                    gc_tn = __ldg(&d->tiles_n);
                    gc_kb = __ldg(&d->num_kb);
                }
                WorkTile t;
                t.g = gc;
                t.n_off = 0;
                t.n_len = BN;
                t.kb_begin = 0;
                t.kb_end = gc_kb;
                t.ks = -1;
                tile_of(w - gc_lo, gc_tm, gc_tn, p.group_m, t.tm, t.tn);
                t.idx = t.tm * gc_tn + t.tn;
                return t;
            };
            // Only CLC waits for the producer before going on: it claims a unit
            // when the producer starts the unit `lead` - 1 units earlier, so
            // the producer finds the next `lead` - 1 units decoded in the ring
            // (lead 1: the claim is made as the producer starts the unit
            // before it; lead 2: one unit earlier, which hides a CLC response
            // behind a whole unit even when units are short, but leaves each
            // cluster holding one more claimed unit when the grid runs out).
            // Claims stay one at a time: a request is issued only after the
            // previous one's response was seen to succeed.  Static units are
            // fixed, so that scheduler runs as far ahead as the ring allows.
            const int lead = p.sched == SCHED_CLC ? p.clc_lead : 0;
            int u = cluster_id < p.num_units ? cluster_id : -1;
            int i = 0;   // ring slot sequence = work items published
            for (int n = 0; ok && u >= 0; ++n) {
                const int pieces = unit_items(u, p);
                for (int j = 0; ok && j < pieces; ++j) {
                    const int w = unit_item(u, j, pieces, p);
                    // Depth 1 waits for the producer to start item i on the started
                    // barrier, whose phase parity is unambiguous there (the producer
                    // cannot be past an item not yet published), and the hardware
                    // may suspend the waiting warp.  Depth 2 lets the producer run a
                    // further item ahead, past what a parity can tell apart, so it
                    // waits on the started-item counter instead.
                    ok = publish(i, w, item_of(w));
                    if (!grouped && i == 0) pdl_wait();   // before any time-limited wait or global access
                    ok = ok
                         && (lead == 0
                             || (lead == 1 ? ctl.wait_all(started_bar, static_cast<uint32_t>(i & 1), WHERE_STARTED)
                                           : ctl.wait_count_all(started_cnt, i + 2 - lead, WHERE_STARTED)));
                    ++i;
                    if (ok && j == 0 && may_request) {
                        // the producer has begun the item `lead` - 1 before this one: claim the next unit
                        if (FULL && (p.debug_flags & DBG_CLC_STOP_AT) && n == p.fault_arg) {
                            may_request = false;   // behave as if this request had failed
                        } else {
                            if (lane == 0) {
                                fence_proxy_async_smem();   // earlier reads of the slot before the async write
                                mbar_arrive_expect_tx(clc_bar, 16);
                                clc_try_cancel(clc_resp, clc_bar);
                            }
                            __syncwarp();
                            clc_pending = true;
                        }
                    }
                }
                int next = -1;
                if (!ok || !next_unit(u, next)) {
                    ok = false;
                    break;
                }
                if (grouped && next >= 0) warm(item_of(next));   // (a grouped launch's units are tiles)
                u = next;
            }
            if (ok) publish(i, -1, WorkTile{});
            if (clc_pending) ctl.drain(clc_bar, clc_phase, 10000000ull);
        }
        __syncwarp();
    }

    // ---- teardown ------------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    if constexpr (CG == 2) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<CG>(tmem_base, kAccCols);
    }
}

}  // namespace pts
