// Kernel parameters and compile-time tile geometry shared by the launcher
// and the kernels (host and device).
#pragma once
#include <cuda.h>

#include <cstdint>

namespace pts {

// One CTA owns 128 rows of the output tile and its TMEM accumulator holds
// 128 lanes x 256 fp32 columns (the wide tile, one CTA per SM) or 128 lanes x
// 128 columns (the narrow tile: single CTAs, whose smaller ring and
// accumulators let two of them share an SM, or CTA pairs, 256 x 128 per pair,
// one CTA per SM).  A k-block is 128 bytes of K per row (64 fp16/bf16 or 128
// e4m3 elements): one 128-byte swizzle atom row.
constexpr int kRowsPerCta = 128;
constexpr int kTileN = 256;             // columns of the wide tile
constexpr int kTileNNarrow = 128;       // columns of the narrow tile
constexpr int kKBlockBytes = 128;
constexpr int kThreads = 224;           // warp 0 producer, warp 1 MMA, warps 2-5 epilogue, warp 6 scheduler
constexpr int kEpiWarps = 4;
constexpr int kSchedWarp = 2 + kEpiWarps;
constexpr int kEpiChunkCols = 64;       // columns per epilogue TMA store (128 bytes of fp16/bf16)
constexpr int kEpiRowsPerWarp = 32;
constexpr int kEpiBufBytes = kEpiRowsPerWarp * kEpiChunkCols * 2;   // 4 KB
constexpr int kEpiBufsPerWarp = 2;
constexpr int kRing = 4;                // depth of the work-item broadcast ring
constexpr int kRingWords = 12;          // 32-bit words per ring slot (a decoded work item)
constexpr int kTmemCols = 512;          // two 256-column accumulators (the narrow tile: 2 x 128)
constexpr int kMaxStages = 8;
constexpr int kDefaultClcLead = 1;      // CLC claim depth when the caller leaves it to the library
constexpr int kDefaultPrefetchKb = 0;   // L2 prefetch of the operand loads: off (it costs more L2
                                        // traffic than it saves in miss latency on GB300)

enum : int32_t { SCHED_NONPERSISTENT = 0, SCHED_STATIC = 1, SCHED_CLC = 2 };

// Device status block: [0] first error code, [1] where, [2] block, [3] error count.
enum : int32_t { DEV_ERR_TIMEOUT = 1 };
enum : uint32_t { DBG_RECORDS = 0x1u, DBG_CLC_STOP_AT = 0x2u, DBG_FAULT_SKIP_TMA = 0x4u };

// Debug record of one work item (a whole tile, a column slice of one, or a
// stream-K piece: one tile's share of a unit's k-blocks).  Times are the low 32 bits of %globaltimer (ns): the
// MMA thread starting the item, the epilogue seeing its accumulator complete,
// the epilogue having issued the item's last store.
struct TileRecord {
    uint32_t visits, tile, n_off, n_len, owner, iter, smid, t_mma_start, t_acc_full, t_stored, kb_begin, kb_end,
        group;
};

// One problem of a grouped launch, in the device table the launcher fills:
// its tensor maps (A: boxes of 128 rows, B: boxes of 256/CG rows, C: the
// epilogue's 32 x 64 store box; A and B unused when K = 0), its sizes in
// tiles and k-blocks, and its output scale.  512 bytes (tensor maps are
// 128-byte aligned).
struct GroupDesc {
    CUtensorMap tmA, tmB, tmC;
    int32_t M, N, num_kb, tiles_m, tiles_n;
    float out_scale;
    int32_t index;   // the problem's position in the caller's list
};
static_assert(sizeof(GroupDesc) == 512, "problem table entry");

struct GemmParams {
    int32_t M, N, K;
    int32_t num_kb;             // k-blocks per tile
    int32_t tiles_m, tiles_n;   // output tiles (per cluster) along M and N
    int32_t num_tiles;
    int32_t split;              // column slices per tile (1, 2 or 4); 1 when sk_units > 0
    int32_t sk_tiles;           // tiles of the stream-K region (the first in grouped order); 0 = none
    int32_t sk_units;           // units sharing the region's k-blocks (0 = none)
    int32_t num_units;          // work ids the schedulers hand out
    int32_t num_work;           // work items (record slots); see work_tile()
    int32_t group_m;            // GROUP_SIZE_M
    int32_t sched;
    int32_t stages;
    int32_t prefetch_kb;        // L2 prefetch distance ahead of the operand loads, in k-blocks (0 = none)
    int32_t epi_direct;         // 1: the epilogue stores C rows straight from registers (no TMA store)
    int32_t clc_lead;           // CLC: units claimed ahead of the producer (1 or 2)
    int32_t tail_tiles;         // the last tail_tiles tiles (grouped order) run as two column halves
                                // each; 0 = none (not with split > 1 or a stream-K region)
    void *c_ptr;                // C (for the direct-store epilogue)
    float out_scale;            // 1, or 1/(scale_a*scale_b) for e4m3
    uint32_t debug_flags;
    int32_t fault_arg;
    uint64_t timeout_ns;
    int32_t *status;            // 4 ints
    float *ws_partial;          // stream-K partial accumulators (fixup workspace), or null
    uint32_t *ws_sync;          // stream-K claim counters and ready flags, 4 words per (tile, CTA, warp);
                                // zero between launches (each launch resets what it used)
    TileRecord *records;        // num_work entries, or null
    // Grouped launch (num_groups > 0): work id w is tile w - group_start[g] of
    // problem g, where group_start[g] <= w < group_start[g + 1], numbered in
    // grouped order within the problem; M, N, K, num_kb, tiles_m, tiles_n,
    // out_scale and the kernel's own tensor maps are then unused.  No
    // stream-K share and no column slices.
    int32_t num_groups;
    const GroupDesc *groups;    // num_groups entries (device)
    const int32_t *group_start; // num_groups + 1 entries (device), group_start[0] = 0
};

// Floats of one stream-K partial: a CTA's 128 x 256 fp32 accumulator.
constexpr int kPartialFloats = kRowsPerCta * kTileN;

// Stream-K share of the last waves.  With T tiles on G resident clusters and
// R = T mod G > 0, the first R + G tiles (grouped order) form the stream-K
// region of L = (R + G) * num_kb k-blocks, taken tile by tile.  Unit c
// (0 <= c < G) gets the k-blocks [floor(c*L/G), floor((c+1)*L/G)), at least
// num_kb and fewer than 2*num_kb of them: up to 3 pieces (one per tile it
// touches), and every tile gets at most 2 pieces.  The remaining tiles are
// whole-tile units G, G+1, ...  Every cluster then does the same number of
// k-blocks to within one, instead of some clusters running a whole extra
// tile in the last wave.  A tile cut in two is summed by a fixup: the piece
// whose accumulation ends first writes its fp32 partial, the other adds it
// and stores C.  The stream-K units come first, so that fixup overlaps the
// whole tiles that follow.
constexpr int kSkMaxPieces = 3;      // record slots per stream-K unit
constexpr int kSkMaxParts = 2;       // pieces per tile
__host__ __device__ inline int64_t sk_unit_begin(int64_t c, int64_t L, int64_t U) { return c * L / U; }

// The unit whose range holds k-block x of the region: the largest c with
// floor(c*L/U) <= x.
__host__ __device__ inline int64_t sk_unit_of(int64_t x, int64_t L, int64_t U) { return ((x + 1) * U - 1) / L; }

// Pieces of stream-K unit c: one per tile its k-block range touches (1..3).
__host__ __device__ inline int sk_pieces(int64_t c, int64_t L, int64_t U, int64_t num_kb)
{
    const int64_t a = sk_unit_begin(c, L, U), b = sk_unit_begin(c + 1, L, U);
    return static_cast<int>((b - 1) / num_kb - a / num_kb + 1);
}

// CTAs per SM: one for the wide tile and for any CTA pair; two for the narrow
// single CTA, whose ring, staging and accumulators fit twice in an SM (why
// pairs never get two, and when the library uses the narrow tile, is with
// choose_tile_n in gemm_plan.h).
__host__ __device__ constexpr int ctas_per_sm(int cg, int bn) { return (bn == kTileNNarrow && cg == 1) ? 2 : 1; }
constexpr int kNarrowStages = 2;        // ring stages of the narrow single CTA

// K-blocks per ring stage.  A stage's fixed costs (its barrier waits, the
// expect-tx arrival, the commit that frees it) are paid once per stage, so a
// CTA pair, whose 32 KB k-blocks leave room for 3 stages of 2, takes 2 per
// stage: measured on GB300 (fp16 4096^2 x 4096) 75.7 vs 79.0 us from the first
// MMA to the last store.  A single CTA keeps 1 (4 stages of 48 KB): with 2 per
// stage it would have only 2 stages in flight, too few to cover the loads
// (K = 768: 26.6 vs 24.8 us).
__host__ __device__ constexpr int kb_per_stage(int cg) { return cg == 2 ? 2 : 1; }
__host__ __device__ constexpr int stage_bytes_a(int cg) { return kRowsPerCta * kKBlockBytes * kb_per_stage(cg); }
__host__ __device__ constexpr int stage_bytes_b(int cg, int bn = kTileN)
{
    return (bn / cg) * kKBlockBytes * kb_per_stage(cg);
}
__host__ __device__ constexpr int epi_bytes() { return kEpiWarps * kEpiBufsPerWarp * kEpiBufBytes; }

// Dynamic shared memory needed for `stages` stages of a tile `bn` columns
// wide (plus 1 KB for aligning the base to the 1024-byte swizzle period).
__host__ __device__ constexpr int smem_bytes(int cg, int stages, int bn = kTileN)
{
    return 1024 + stages * (stage_bytes_a(cg) + stage_bytes_b(cg, bn)) + epi_bytes()
           + 8 * (2 * kMaxStages + 4 + 2 * kRing + 2)    // mbarriers
           + 16                                          // CLC response
           + 4 * kRingWords * kRing + 16;                // ring payload, TMEM base, abort flag, started count
}

}  // namespace pts
