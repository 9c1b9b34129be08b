// Launch-plan rules of the host: the CTA group, tile width, column slices,
// tail halves and stream-K share a problem gets when the caller leaves them
// to the library.
// Host-only (the kernels never read them); each threshold comes from the
// measurement on GB300 quoted beside it.
#pragma once
#include <cstdint>

#include "gemm_params.h"

namespace pts {

// Stream-K share of the last waves (its layout is with kSkMaxPieces in
// gemm_params.h).
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
// The non-persistent grid launches a cluster per tile (or stream-K unit), and
// a pair cluster costs more to start and finish than a single CTA, so single
// CTAs stay ahead much longer there.  Measured on GB300 (chained launches,
// the library's stream-K choice, single vs pairs, us per launch): fp16 4096^2
// K = 1024 41.6 vs 51.9, 2048 57.0 vs 61.8, 3072 77.6 vs 80.9, 3584 86.5 vs
// 88.4, 4096 95.5 vs 96.9; bf16 8192^2 K = 1024 141.3 vs 180.7, 2048 217.4 vs
// 247.3, 3072 290.5 vs 301.6, 4096 375.7 vs 368.2, 8192 726.5 vs 674.0.  So
// pairs from 64 k-blocks per tile for that grid.
constexpr int kPairMinKbNonPersistent = 64;

inline int choose_cta_group(int64_t num_kb, int sched = SCHED_STATIC)
{
    return num_kb >= (sched == SCHED_NONPERSISTENT ? kPairMinKbNonPersistent : kPairMinKb) ? 2 : 1;
}

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

// Column halves for the tail.  With T tiles on G resident clusters and
// R = T mod G, the last wave keeps only R clusters busy, each for a whole
// tile.  When 2R <= G the last R tiles (grouped order) are each cut into two
// column halves, run as 2R units: every cluster still busy in the last wave
// has half a tile.  A half tile takes about two thirds of a whole one (its
// k-blocks carry half the MMA work but not half the per-k-block cost) and
// needs no fixup, so it keeps the result's bits.  Measured on GB300 (fp16
// 4096^2, R = 28 of 76 pairs or 56 of 152 single CTAs, chained launches,
// whole / halves, us per launch): K = 384 16.1 / 14.8, 640 21.6 / 20.6,
// 1024 28.6 / 27.5, 1536 38.1 / 36.8, 1920 45.0 / 43.5; bf16 8192^2
// (R = 36) K = 1024 84.6 / 83.2, 2048 152.1 / 151.2.  Returns R, or 0.
inline int64_t choose_tail(int64_t tiles, int64_t resident)
{
    if (resident < 2 || tiles <= resident) return 0;
    const int64_t r = tiles % resident;
    return (r > 0 && 2 * r <= resident) ? r : 0;
}

// Where both apply, the halves are used below this many k-blocks per tile and
// the stream-K share from here (when it saves kSkMinSavedKb): the share
// evens the last wave out fully but pays its fixup, the halves leave the last
// wave at two thirds of a tile but pay nothing.  Measured on GB300 (fp16
// 4096^2, chained launches, share / halves, us per launch): K = 2048 47.1 /
// 45.4, 2560 54.9 / 54.3, 3072 63.7 / 63.8, 3584 72.7 / 73.5, 4096 81.9 /
// 83.0; bf16 8192^2 K = 3072 220.8 / 221.0, 4096 288.5 / 287.9.
constexpr int kTailMaxKb = 48;

// The partial last wave of `tiles` tiles of `num_kb` k-blocks on `resident`
// clusters (wide tile, no column slices): returns the stream-K region's tiles
// (0 = none) and sets `tail` to the tiles run as column halves (0 = none).
// split_auto: the caller left column slicing to the library (else no
// halves); sk_force as for choose_stream_k.  Halves only for the persistent
// schedulers: the non-persistent grid launches a cluster per half and gains
// nothing from them (measured on GB300, fp16 4096^2, chained, without /
// with halves: K = 1024 40.0 / 40.0 us, 1536 49.9 / 50.0; in place of the
// stream-K share K = 2048 57.1 / 59.6, 2560 65.9-71.5 / 75.7).
inline int64_t choose_last_wave(int64_t tiles, int64_t resident, int64_t num_kb, bool split_auto, int sk_force,
                                int sched, int64_t &tail)
{
    const int64_t r = (split_auto && sched != SCHED_NONPERSISTENT) ? choose_tail(tiles, resident) : 0;
    const bool halves_first = r > 0 && sk_force == 0 && num_kb < kTailMaxKb;
    const int64_t sk = halves_first ? 0 : choose_stream_k(tiles, resident, num_kb, sk_force);
    tail = sk > 0 ? 0 : r;
    return sk;
}

// The narrow tile (tile_n 128).  The wide tile's ring and staging take nearly
// all of an SM's shared memory; the narrow single CTA's fit twice (two stages of 32 KB, 32 KB of
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
//
// Narrow tiles when the caller leaves both the tile and the CTA group to the
// library: for the non-persistent grid (sched 0) on tiles of at most this
// many k-blocks.
constexpr int kNarrowMaxKb = 4;
// CLC is left on the wide tile even at 2 k-blocks, where the narrow tile's
// second CTA per SM hides the claim latency (fp16 4096^2 x 128, chained
// launches of that one shape, wide / narrow: 12.9 / 11.8 and 13.9 / 12.4 us on
// two boxes): in a sequence of GEMMs of different K, the first wide-tile launch
// after a narrow one pays about 3 us for the change of kernel, which takes the
// gain back (measured in the K sweep: CLC at K = 256 went from 436-442 to 381
// TFLOP/s when K = 128 before it took the narrow tile).

inline int choose_tile_n(int64_t num_kb, int cta_group_opt, int sched)
{
    return (cta_group_opt == 0 && sched == SCHED_NONPERSISTENT && num_kb <= kNarrowMaxKb) ? kTileNNarrow : kTileN;
}

}  // namespace pts
