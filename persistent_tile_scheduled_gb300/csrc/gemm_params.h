// Kernel parameters and compile-time tile geometry shared by the launcher
// and the kernels (host and device).
#pragma once
#include <cstdint>

namespace pts {

// One CTA owns 128 rows of the output tile and its TMEM accumulator holds
// 128 lanes x 256 fp32 columns.  A k-block is 128 bytes of K per row (64
// fp16/bf16 or 128 e4m3 elements): one 128-byte swizzle atom row.
constexpr int kRowsPerCta = 128;
constexpr int kTileN = 256;
constexpr int kKBlockBytes = 128;
constexpr int kThreads = 192;           // warp 0 producer, warp 1 MMA, warps 2-5 epilogue
constexpr int kEpiWarps = 4;
constexpr int kEpiChunkCols = 64;       // columns per epilogue TMA store (128 bytes of fp16/bf16)
constexpr int kEpiRowsPerWarp = 32;
constexpr int kEpiBufBytes = kEpiRowsPerWarp * kEpiChunkCols * 2;   // 4 KB
constexpr int kEpiBufsPerWarp = 2;
constexpr int kRing = 4;                // depth of the tile-id broadcast ring
constexpr int kTmemCols = 512;          // two 256-column accumulators
constexpr int kMaxStages = 8;
constexpr int kDefaultPrefetchKb = 0;   // L2 prefetch of the operand loads: off (it costs more L2
                                        // traffic than it saves in miss latency on GB300)

enum : int32_t { SCHED_NONPERSISTENT = 0, SCHED_STATIC = 1, SCHED_CLC = 2 };

// Device status block: [0] first error code, [1] where, [2] block, [3] error count.
enum : int32_t { DEV_ERR_TIMEOUT = 1 };
enum : uint32_t { DBG_RECORDS = 0x1u, DBG_CLC_STOP_AT = 0x2u, DBG_FAULT_SKIP_TMA = 0x4u };

// Debug record of one work item (a tile, or a column slice of a tile of the
// last partial wave).  Times are the low 32 bits of %globaltimer (ns): the
// MMA thread starting the item, the epilogue seeing its accumulator complete,
// the epilogue having issued the item's last store.
struct TileRecord {
    uint32_t visits, tile, n_off, n_len, owner, iter, smid, t_mma_start, t_acc_full, t_stored, kb_begin, kb_end;
};

struct GemmParams {
    int32_t M, N, K;
    int32_t num_kb;             // k-blocks per tile
    int32_t tiles_m, tiles_n;   // output tiles (per cluster) along M and N
    int32_t num_tiles;
    int32_t full_work;          // work ids below this are whole tiles
    int32_t split;              // each later tile is cut into `split` parts (1..4)
    int32_t split_k;            // 0: parts are column slices; 1: parts are K ranges, reduced in a fixup
    int32_t part_kb;            // K ranges: k-blocks of each part but the last (the last gets the rest)
    uint32_t epoch;             // launch number (29 bits, never 0) tagging the fixup counters and flags
    int32_t num_work;           // full_work + split * (num_tiles - full_work)
    int32_t group_m;            // GROUP_SIZE_M
    int32_t sched;
    int32_t stages;
    int32_t prefetch_kb;        // L2 prefetch distance ahead of the operand loads, in k-blocks (0 = none)
    int32_t epi_direct;         // 1: the epilogue stores C rows straight from registers (no TMA store)
    void *c_ptr;                // C (for the direct-store epilogue)
    float out_scale;            // 1, or 1/(scale_a*scale_b) for e4m3
    uint32_t debug_flags;
    int32_t fault_arg;
    uint64_t timeout_ns;
    int32_t *status;            // 4 ints
    float *ws_partial;          // K-split partial accumulators (fixup workspace), or null
    uint32_t *ws_sync;          // K-split claim counters and ready flags, 4 words per (tile, CTA)
    TileRecord *records;        // num_work entries, or null
};

// Floats of one K-split partial: a CTA's 128 x 256 fp32 accumulator.
constexpr int kPartialFloats = kRowsPerCta * kTileN;

// K-split of the last partial wave.  The first split-1 parts get `part_kb`
// k-blocks each and the last part the rest, which is longer: the first parts
// finish early and write their fp32 partials while the last one still
// computes, so it finds them ready.  Measured on GB300 a writer needs about
// kFixupWriteKb k-blocks' time to publish its partial and the last part about
// kFixupReadKb per partial it adds.
constexpr int kFixupWriteKb = 13;
constexpr int kFixupReadKb = 5;

inline int64_t split_part_kb(int64_t num_kb, int split)
{
    const int64_t a = (num_kb - kFixupWriteKb) / split;
    return a < 1 ? 1 : a;
}

// K parts per leftover tile of the last partial wave (1 = no split): the
// count that shortens the wave most, if it saves more than 8 k-blocks' time;
// parts must fit the idle clusters of that wave.
inline int choose_split_k(int64_t tiles, int64_t resident, int64_t num_kb)
{
    const int64_t r = tiles % resident;
    if (tiles < resident || r == 0) return 1;
    int best = 1;
    int64_t best_tail = num_kb - 8;
    for (int s = 2; s <= 4; ++s) {
        if (s * r > resident || s > num_kb) break;
        const int64_t a = split_part_kb(num_kb, s);
        const int64_t last = num_kb - (s - 1) * a;
        const int64_t writers_done = a + kFixupWriteKb;
        const int64_t tail = (last > writers_done ? last : writers_done) + kFixupReadKb * (s - 1);
        if (tail < best_tail) {
            best_tail = tail;
            best = s;
        }
    }
    return best;
}

// CTA group when the caller leaves it to the library.  CTA pairs (cta_group
// 2) load a third less per SM for the same MMA work, so their mainloop runs
// faster under full load (fp16 4096^2 x 4096: 0.318 vs 0.326 us per k-block,
// 90 vs 94 us per launch), but a pair costs a few microseconds more to start
// and finish.  Measured over the fp16 4096^2 K sweep on GB300, pairs pay off
// from about 16 k-blocks per tile; single CTAs win below (K = 256: 21.5 vs
// 28.3 us).
constexpr int kPairMinKb = 16;

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

__host__ __device__ constexpr int stage_bytes_a() { return kRowsPerCta * kKBlockBytes; }
__host__ __device__ constexpr int stage_bytes_b(int cg) { return (kTileN / cg) * kKBlockBytes; }
__host__ __device__ constexpr int epi_bytes() { return kEpiWarps * kEpiBufsPerWarp * kEpiBufBytes; }

// Dynamic shared memory needed for `stages` stages (plus 1 KB for aligning
// the base to the 1024-byte swizzle period).
__host__ __device__ constexpr int smem_bytes(int cg, int stages)
{
    return 1024 + stages * (stage_bytes_a() + stage_bytes_b(cg)) + epi_bytes()
           + 8 * (2 * kMaxStages + 4 + 2 * kRing + 1)    // mbarriers
           + 16                                          // CLC response
           + 4 * kRing + 16;                             // ring payload, TMEM base, abort flag
}

}  // namespace pts
