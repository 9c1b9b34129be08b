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
// Use it when it saves each cluster at least this many k-blocks' time.  The
// price, measured on GB300 (fp16 4096^2, CTA pairs, per-item records): a
// writer piece's epilogue takes 5.5-5.8 us against 1.1-1.5 us for a whole
// tile (its 128 KB fp32 partial per CTA; staging that partial through shared
// memory and bulk copies measured slower still, 6.9-7.7 us), a reader's
// 3.5-4.7 us; hidden behind a long next tile, not behind a short one.
// Chained launches, without / with the share: K = 1536 (24 k-blocks, 15 saved
// per cluster) 38.2 / 38.8 us, K = 1792 (28, 18 saved) 42.5 / 43.2, K = 2048
// (32, 20 saved) 48.7 / 48.1, K = 3072 68.6 / 64.8, K = 4096 91.2 / 84.2.
constexpr int kSkMinSavedKb = 20;

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

// Tiles in the stream-K region for `tiles` tiles of `num_kb` k-blocks on
// `resident` clusters (0 = do not use it).  force: 1 = whenever the last wave
// is partial, -1 = never, 0 = when it saves kSkMinSavedKb k-blocks' time.
inline int64_t choose_stream_k(int64_t tiles, int64_t resident, int64_t num_kb, int force)
{
    if (force < 0 || num_kb < 1 || resident < 1 || tiles < resident) return 0;
    const int64_t r = tiles % resident;
    if (r == 0) return 0;
    if (force == 0 && num_kb * (resident - r) < kSkMinSavedKb * resident) return 0;
    return r + resident;
}

// CTA group when the caller leaves it to the library.  CTA pairs (cta_group
// 2) load a third less per SM for the same MMA work, so their mainloop runs
// faster under full load, but a pair costs more per launch to start, fill
// and finish.  Measured on GB300 on fp16 4096^2 with cold inputs (eight
// buffer sets in turn), single vs pair per launch, without the stream-K
// share: K = 640 22.9-23.1 vs 24.3-24.5 us, K = 768 25.5 vs 25.7, K = 896
// 27.8-28.3 vs 27.4-27.5, K = 1152 33.1-33.2 vs 32.7-32.8.  So pairs from
// 14 k-blocks per tile.
constexpr int kPairMinKb = 14;

inline int choose_cta_group(int64_t num_kb) { return num_kb >= kPairMinKb ? 2 : 1; }

// Column slices per tile for a problem of `tiles` tiles on `resident`
// clusters.  Only a problem smaller than one wave is sliced (quarters when it
// fits in a quarter wave, halves when it fits in half): there slicing puts
// idle SMs to work.  Past one wave the slices' smaller stages leave the
// latency-bound load pipeline with fewer bytes in flight, and a slice takes
// nearly as long as a whole tile, so later waves are not sliced.
inline int choose_split(int64_t tiles, int64_t resident)
{
    if (tiles >= resident) return 1;
    if (4 * tiles <= resident) return 4;
    if (2 * tiles <= resident) return 2;
    return 1;
}

// CTAs per SM: the wide tile's ring and staging take nearly all of an SM's
// shared memory; the narrow tile's fit twice (two stages of 32 KB, 32 KB of
// epilogue staging, about 97 KB per CTA), and its accumulators take 256 of
// the SM's 512 TMEM columns.  A second resident CTA gives the SM a second,
// independent load -> MMA -> epilogue pipeline: while one CTA waits for its
// operands or drains its output, the other computes.  That pays where tiles
// are short (few k-blocks) and the per-tile latencies dominate; for long
// tiles the narrow tile's two-stage ring and its 4/3 times higher operand
// traffic per flop lose to the wide tile.  ("[Persistent] Performance on
// 09-persistent-matmul on A100 worse than non-persistent": the best
// persistent configuration there was 128x128x64 tiles with twice as many
// programs as SMs.)
//
// Measured on GB300 (fp16 4096^2, 40 chained launches per point, microseconds
// per launch; wide = 128 x 256 single CTAs, narrow = 128 x 128, two per SM):
//   K     static wide / narrow   CLC wide / narrow   non-persistent wide / narrow
//   128   11.8 / 11.8            12.9 / 11.8         23.5 / 20.8
//   256   13.1 / 16.8            13.6 / 16.6         26.2 / 25.3
//   512   19.5 / 24.2            19.4 / 24.1         31.5 / 32.7
//   1024  29.6 / 38.9            29.7 / 39.0         41.9 / 47.0
// The persistent grids gain nothing: at small K a launch is bound by the
// latency of its operand loads, and the SM's operands in flight are what
// sets the pace -- four 48 KB stages for the wide tile, 2 x 2 stages of 32 KB
// for the narrow pair -- so the narrow tile ties at 2 k-blocks and loses
// beyond.  The non-persistent grid, which starts a CTA per tile, gains from
// two CTAs per SM up to 4 k-blocks.
//
// The narrow tile also comes as a CTA pair (256 x 128 per pair, tcgen05
// cta_group::2), but at one CTA per SM, with the deepest ring that fits: the
// two CTAs of a pair then sit on two SMs by construction.  Nothing available
// here documents where the hardware puts a pair's two CTAs when one SM could
// hold both, and a pair's MMA cannot run with both on one SM, so pairs are
// never given a second CTA per SM.
__host__ __device__ constexpr int ctas_per_sm(int cg, int bn) { return (bn == kTileNNarrow && cg == 1) ? 2 : 1; }
constexpr int kNarrowStages = 2;        // ring stages of the narrow single CTA
// Narrow tiles when the caller leaves both the tile and the CTA group to the
// library: for the non-persistent grid (sched 0) on tiles of at most this
// many k-blocks.
constexpr int kNarrowMaxKb = 4;

inline int choose_tile_n(int64_t num_kb, int cta_group_opt, int sched)
{
    return (cta_group_opt == 0 && sched == SCHED_NONPERSISTENT && num_kb <= kNarrowMaxKb) ? kTileNNarrow : kTileN;
}

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
