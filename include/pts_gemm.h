/*
 * pts_gemm.h -- C ABI of the persistent, tile-scheduled GEMM for GB300 (sm_103a).
 *
 * Computes C = A . B with fp32 accumulation on the tensor cores:
 *   A  M x K, row-major (leading dimension K)
 *   B  stored N x K, row-major (leading dimension K), i.e. K x N column-major
 *   C  M x N, row-major (leading dimension N); fp16 for fp16 inputs, bf16 for
 *      bf16 and e4m3 inputs.  For e4m3, C = (A8 . B8) / (scale_a * scale_b).
 *
 * The output is cut into tiles (one tile per CTA, or per CTA pair with
 * cta_group 2); a scheduler hands the tiles to CTAs:
 *   - non-persistent: one CTA (pair) per tile, the hardware block scheduler
 *     assigns them (the question of "question about persistent kernel
 *     concept": one thread block per tile);
 *   - static: a grid sized to the resident capacity of the SMs, each CTA
 *     derives its later tiles in software ("Persistent Kernels with Cluster
 *     Launch Control", first paragraph; "Choosing between static and CLC
 *     scheduling", first bullet);
 *   - CLC: a grid of one CTA (pair) per tile; running CTAs cancel clusters
 *     that have not launched yet and take over their tiles
 *     (clusterlaunchcontrol.try_cancel; same page, second paragraph).
 * Tiles are visited in GROUP_SIZE_M-grouped order ("[Persistent] Performance
 * on 09-persistent-matmul on A100 worse than non-persistent", the
 * hyperparameter list: GROUP_SIZE_M 8).
 *
 * General rules for every call:
 *   - Device pointers are plain CUDA device addresses of the current process
 *     on the handle's device; host pointers are ordinary host memory (pinned
 *     memory makes the copies asynchronous).
 *   - Errors are reported only through the returned status; nothing aborts
 *     the process and no call falls back to the CPU.
 *   - Calls are asynchronous on the given stream unless stated otherwise.
 *   - A handle is not thread-safe; use one handle per host thread.  GEMMs
 *     that run at the same time on different streams need one handle each:
 *     a handle's workspace (stream-K partials, debug records) serves one
 *     launch at a time.
 */
#ifndef PTS_GEMM_H
#define PTS_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { GEMM_F16 = 0, GEMM_BF16 = 1, GEMM_E4M3 = 2 } gemm_dtype_t;

typedef enum {
    GEMM_SCHED_NONPERSISTENT = 0,
    GEMM_SCHED_STATIC = 1,
    GEMM_SCHED_CLC = 2
} gemm_sched_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment, enum or option */
    GEMM_ERR_UNSUPPORTED = 2,   /* device is not compute capability 10.3 */
    GEMM_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed */
    GEMM_ERR_TIMEOUT = 4,       /* a device-side wait hit its time limit */
    GEMM_ERR_COVERAGE = 5       /* tile records show a tile not visited exactly once */
} gemm_status_t;

/* debug_flags */
#define GEMM_DEBUG_RECORDS 0x1u   /* fill one gemm_tile_record_t per tile */
#define GEMM_DEBUG_CLC_STOP_AT 0x2u
/* with GEMM_SCHED_CLC: every CTA (pair) behaves as if its fault_arg-th
 * try_cancel request (0-based) had failed: it does not issue it and stops
 * after its current tile.  Clusters that were therefore not cancelled launch
 * and run their own tile, so coverage stays exact. */
#define GEMM_DEBUG_FAULT_SKIP_TMA 0x4u
/* test hook for the bounded waits: every producer announces its fault_arg-th
 * stage load (0-based) but does not issue it, so the MMA warp's wait on that
 * stage runs past timeout_ns.  The kernel records the time-out, stops every
 * role, frees its resources and returns; gemm_check then reports
 * GEMM_ERR_TIMEOUT and C is unspecified.  The context stays usable. */

typedef struct gemm_opts {
    int cta_group;                  /* 1 (128x256 tile per CTA) or 2 (256x256 per CTA pair);
                                       0 = per call: pairs when a tile has >= 14 k-blocks
                                       (the persistent schedulers) or >= 64 (the
                                       non-persistent grid) */
    int group_size_m;               /* tile-rows per group of the tile order; 0 = 8 */
    int stages;                     /* shared-memory ring depth in stages (a stage holds one
                                       k-block for single CTAs, two for CTA pairs); 0 = the
                                       most that fits (4 and 3) */
    int max_clusters;               /* static scheduler: cap on resident clusters; 0 = occupancy */
    unsigned debug_flags;           /* GEMM_DEBUG_*.  Any debug flag, epilogue 2 or an L2
                                       prefetch makes gemm_run use the kernel built with every
                                       feature; without them it uses a build with those paths
                                       compiled out, which gives the same bits and starts about
                                       1 us sooner per launch at small K (measured on GB300) */
    int fault_arg;                  /* argument of GEMM_DEBUG_CLC_STOP_AT / _FAULT_SKIP_TMA */
    unsigned long long timeout_ns;  /* limit of every device-side wait; 0 = 1 s */
    int split;                      /* column slices: 0 = automatic (a problem smaller than one
                                       wave; or, with the wide tile and a persistent scheduler,
                                       the tiles of a partial last wave when they fill at most
                                       half of it: two column halves each, unless the stream-K
                                       share is used instead); 1 = never; 2 or 4 = cut EVERY
                                       tile into that many column slices (testing) */
    int split_k;                    /* stream-K share of the last waves: 0 = automatic (when it
                                       saves time), 1 = whenever the tiles leave a partial last
                                       wave, -1 = never.  Not with split 2 or 4. */
    int prefetch;                   /* L2 prefetch of the operands, in k-blocks ahead of the
                                       loads (<= 64); 0 = default (none), -1 = none */
    int overlap_launch;             /* 0 = default (on): a launch may start while the previous
                                       kernel in the stream finishes (programmatic dependent
                                       launch; it waits for that kernel before touching memory);
                                       -1 = off */
    int epilogue;                   /* 0 = default (1); 1 = TMA stores from a swizzled shared-
                                       memory staging buffer; 2 = every lane stores its row's
                                       outputs straight from registers */
    int group_order;                /* gemm_run_grouped's order of the problems in the work-id
                                       list: 0 = default (1); 1 = most k-blocks first (stable:
                                       equal K keep the given order); 2 = as given */
    int tile_n;                     /* output tile columns of gemm_run: 0 = per call (128 for the
                                       non-persistent scheduler when a tile has <= 4 k-blocks and
                                       cta_group is 0, else 256);
                                       256 = the wide tile (one CTA, or CTA pair, per SM);
                                       128 = the narrow tile: 128 x 128 per CTA; with cta_group
                                       0 or 1 single CTAs, two resident per SM; with cta_group 2
                                       a 256 x 128 tile per CTA pair, one CTA per SM (a pair is
                                       never given a second CTA per SM: where the hardware puts
                                       the two CTAs of a pair then is not documented); no
                                       stream-K share and no column quarters (split 4) with it.
                                       gemm_run_grouped and gemm_run_noalloc use the wide tile. */
    int clc_depth;                  /* GEMM_SCHED_CLC: how far ahead of the producer a cluster
                                       claims work.  1 = the next unit is claimed when the producer
                                       starts the current one; 2 = one unit earlier (the response
                                       then has a whole unit to arrive in, but every cluster holds
                                       one more claimed unit at the end of the grid).  Requests
                                       stay one at a time either way: the next is issued only after
                                       the previous one was seen to succeed.  0 = default (1). */
} gemm_opts_t;

/* Work items.  Output tiles are numbered in grouped order (GROUP_SIZE_M tile-
 * rows per group, walked column by column).  The schedulers hand out units;
 * a unit is one or more work items, each computed in one accumulator:
 *   - Whole tiles: unit u = work item u = tile u.
 *   - Column slices (split 2 or 4; a problem smaller than one wave of
 *     resident clusters, so that more SMs take part): unit u = work item u =
 *     columns (u % split) * 256/split .. +256/split of tile u / split.
 *   - Stream-K share (split_k): with T tiles on G resident clusters and a
 *     partial last wave (R = T mod G > 0), the first R + G tiles form a region
 *     of L = (R + G) * num_kb k-blocks, taken tile by tile.  Unit c < G gets
 *     k-blocks floor(c*L/G) .. floor((c+1)*L/G) - 1 of it: one work item
 *     ("piece", record slot 3c + j) for each tile j = 0, 1, 2 the range
 *     touches, run last tile first (so every unit starts at k-block 0 of a
 *     tile).  A tile split between two units is summed by a fixup: the
 *     piece that finishes accumulating first writes its fp32 partial to a
 *     workspace the handle owns, the other adds it and stores C.  Units
 *     G, G+1, ... (record slots 3G, 3G+1, ...) are the remaining tiles,
 *     whole.  Every cluster then does the same number of k-blocks to within
 *     one, instead of some clusters running a whole extra tile in the last
 *     wave; the region comes first so that the fixup overlaps whole tiles.
 * Cutting tiles changes which CTA computes what, never the result beyond the
 * fp32 summation order.  The pages on persistent tile scheduling hand out
 * whole tiles only; the column slices and the stream-K share are this
 * library's additions for the tail of a grid.
 *
 * Per-work-item record written when GEMM_DEBUG_RECORDS is set (work-id order). */
typedef struct gemm_tile_record {
    uint32_t visits;   /* CTAs that stored this item; exactly cta_group when coverage is exact
                          (0 for the unused slots of a stream-K unit with fewer than 3 pieces) */
    uint32_t tile;     /* tile index tm * tiles_n + tn of the item */
    uint32_t n_off;    /* first column of the item within its tile */
    uint32_t n_len;    /* columns of the item (256, 128 or 64) */
    uint32_t owner;    /* cluster index (blockIdx.x / cta_group) that ran it */
    uint32_t iter;     /* how many items that cluster had run before it */
    uint32_t smid;     /* SM of the (leader) CTA */
    /* low 32 bits of the GPU global timer (ns) when: the MMA thread began the
     * item, the epilogue saw its accumulator complete, the epilogue issued the
     * item's last store (leader CTA) */
    uint32_t t_mma_start, t_acc_full, t_stored;
    uint32_t kb_begin, kb_end;  /* k-block range of the item */
    uint32_t group;    /* problem of the item in a grouped launch (its index in the caller's list;
                          0 otherwise); `tile` is then the tile index within that problem */
} gemm_tile_record_t;

/* Launch shape chosen for a problem. */
typedef struct gemm_launch_info {
    int tile_m, tile_n, tile_k;     /* output tile per cluster, k-block (elements; a CTA pair's
                                       ring stage holds two k-blocks) */
    int cta_group;
    int stages;
    int64_t tiles_m, tiles_n, tiles;
    int64_t grid_ctas;              /* gridDim.x */
    int max_active_clusters;        /* resident clusters the device holds for this kernel */
    int smem_bytes;                 /* dynamic shared memory per CTA */
    int threads;                    /* threads per CTA */
    int split;                      /* column slices per tile (1 = none, 2 or 4) */
    int split_k;                    /* 1 when the stream-K share is used */
    int64_t sk_tiles;               /* tiles of the stream-K region (0 = none) */
    int64_t sk_units;               /* units sharing it (the resident clusters G) */
    int64_t work_items;             /* work items = record slots (gemm_read_debug's n_work) */
    int64_t units;                  /* units the schedulers hand out */
    int ctas_per_sm;                /* CTAs the kernel keeps resident per SM (1 wide, 2 narrow) */
    int64_t tail_tiles;             /* tiles of the partial last wave run as two column halves
                                       each (the last in tile order; 0 = none); work ids
                                       tiles - tail_tiles + 2j and + 2j + 1 are the left and
                                       right half of tile tiles - tail_tiles + j */
} gemm_launch_info_t;

typedef struct gemm_ctx *gemm_handle_t;

/* Create a handle on `device` (made current for the call).  opts may be NULL
 * (all defaults).  Allocates a small device status block; the handle owns it.
 * Returns GEMM_ERR_UNSUPPORTED on anything but compute capability 10.3,
 * GEMM_ERR_CUDA if the device cannot be used, GEMM_ERR_INVALID_ARG for bad
 * options. */
gemm_status_t gemm_create(gemm_handle_t *out, int device, const gemm_opts_t *opts);

/* C = A . B on `stream` (a cudaStream_t; NULL = legacy default stream).
 * A, B, C: device pointers, 16-byte aligned, caller-owned, not overlapping C.
 * Sizes: M, N, K >= 0; K*elem_bytes and N*2 must be multiples of 16 bytes
 * (K % 8 == 0 for fp16/bf16, K % 16 == 0 for e4m3, N % 8 == 0); each of
 * M, N, K < 2^31.  M == 0 or N == 0 launches nothing; K == 0 writes zeros.
 * scale_a, scale_b: e4m3 per-tensor scales (> 0, finite); ignored otherwise.
 * Returns after the launch; device-side errors (wait time-outs) are read with
 * gemm_check or gemm_read_debug.
 * CUDA graphs: a gemm_run launch may be captured and the graph replayed any
 * number of times.  Each launch leaves the stream-K claim counters and ready
 * flags it used at zero, so a replay starts exactly like a fresh launch.
 * The workspace is grown (cudaMalloc, cudaMemset) by the first call that
 * needs more than the handle holds, which a capturing stream does not allow:
 * make one call of the same shape before capturing.  That growth may also
 * wait for work already queued on other streams of the device, so a call that
 * should overlap another stream's kernels is best preceded by one of the same
 * shape. */
gemm_status_t gemm_run(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                       const void *A, const void *B, void *C,
                       gemm_dtype_t dtype, gemm_sched_t sched,
                       float scale_a, float scale_b, void *stream);

/* gemm_run on HOST buffers: copies A and B to device memory the handle owns
 * (grown as needed), runs, copies C back to C_host, all on `stream`, then
 * synchronises the stream and returns the device status like gemm_check.
 * Same size rules as gemm_run; host pointers need no alignment. */
gemm_status_t gemm_run_host(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                            const void *A_host, const void *B_host, void *C_host,
                            gemm_dtype_t dtype, gemm_sched_t sched,
                            float scale_a, float scale_b, void *stream);

/* One GEMM of a host-buffer batch (see gemm_run_host_batch). */
typedef struct gemm_host_problem {
    int64_t M, N, K;
    const void *A;          /* host, M x K */
    const void *B;          /* host, N x K */
    void *C;                /* host, M x N */
    gemm_dtype_t dtype;
    float scale_a, scale_b; /* e4m3 only */
} gemm_host_problem_t;

/* Run n independent GEMMs on HOST buffers with the transfers overlapped:
 * while one GEMM computes on `stream`, the inputs of the next are copied in
 * (one copy stream) and the results of earlier ones are copied out (two copy
 * streams, alternating), all owned by the handle, through six device staging
 * slots the handle owns (grown as needed), so copy-in may run up to five GEMMs
 * ahead of copy-out.  The
 * problems are processed in an order the library picks (alternately the most
 * output-heavy and the most input-heavy remaining one), so that both
 * directions of the host link carry data at once; every C is written exactly
 * as if they ran in the given order.  Work already
 * queued on `stream` completes before the first copy starts.  Returns after
 * every result is in host memory (the call synchronises), with the device
 * status like gemm_check.  Pinned host memory is needed for the copies to
 * overlap.  Same size rules per problem as gemm_run; n == 0 does nothing. */
gemm_status_t gemm_run_host_batch(gemm_handle_t h, const gemm_host_problem_t *problems, int64_t n,
                                  gemm_sched_t sched, void *stream);

/* ---- grouped launch ----------------------------------------------------
 * One problem of gemm_run_grouped: C = A . B with device pointers and the
 * layouts, size rules and scales of gemm_run (M, N, K >= 0; M == 0 or N == 0
 * contributes no tiles; K == 0 makes C zero). */
typedef struct gemm_group_problem {
    int64_t M, N, K;
    const void *A;          /* device, M x K */
    const void *B;          /* device, N x K */
    void *C;                /* device, M x N */
    float scale_a, scale_b; /* e4m3 only */
} gemm_group_problem_t;

#define GEMM_GROUPED_MAX_PROBLEMS 65536

/* `count` independent GEMMs of one dtype in ONE launch.  The tiles of all
 * problems form one list of work ids (problem by problem, each problem's
 * tiles in GROUP_SIZE_M-grouped order) that the scheduler hands out as it
 * does one problem's tiles; a tile costs time in proportion to its problem's
 * K, so the tiles differ in cost and a scheduler that hands out work as
 * clusters finish (CLC, or the hardware's for the non-persistent grid) can
 * balance what the static stride cannot ("Choosing between static and CLC
 * scheduling": dynamic scheduling pays off when the work per tile varies).
 * The problems are listed most k-blocks first (opts.group_order 1, the
 * default; longest-processing-time-first list scheduling, so the last tiles
 * handed out are the short ones) or in the given order (group_order 2).
 * No stream-K share and no column slices.  CTA group (cta_group 0): pairs
 * when the mean k-blocks per tile, weighted by output size, is at least 14.
 * The handle keeps the problem table (tensor maps and tile counts, 512 bytes
 * per problem) in device memory it owns, in two slots: a call with the same
 * problems as the previous one reuses its table; a different list is copied
 * to the other slot on `stream`, after the host has waited for the launch
 * that last read that slot.  `problems` is host memory, read during the call
 * only.  A capturing stream is refused (GEMM_ERR_INVALID_ARG): a graph would
 * keep referring to a table later calls rewrite.  count in
 * [0, GEMM_GROUPED_MAX_PROBLEMS]; total tiles < 2^30.  Records
 * (GEMM_DEBUG_RECORDS) are per tile in work-id order with `group` set. */
gemm_status_t gemm_run_grouped(gemm_handle_t h, const gemm_group_problem_t *problems, int64_t count,
                               gemm_dtype_t dtype, gemm_sched_t sched, void *stream);

/* Launch shape gemm_run_grouped would use (no GPU work): tiles, work_items
 * and units are the total over all problems; tiles_m, tiles_n are 0. */
gemm_status_t gemm_query_grouped(gemm_handle_t h, const gemm_group_problem_t *problems, int64_t count,
                                 gemm_dtype_t dtype, gemm_sched_t sched, gemm_launch_info_t *info);

/* ---- tensor-pipe peak probe (a measurement aid, not a GEMM) -------------
 * Every SM (cta_group 1) or SM pair (cta_group 2) issues `mmas` back-to-back
 * tcgen05.mma of one k-step of the GEMM's tile (128 x 256 per CTA, 256 x 256
 * per pair; K = 16 for fp16/bf16, 32 for e4m3) on finite operands already in
 * shared memory: no loads, stores or epilogue, so only the tensor pipe limits
 * it.  It measures the dense FLOP per SM clock that the GEMM's "% of tensor
 * peak" assumes ("Persistent Kernels with Cluster Launch Control" names the
 * tcgen05 2-SM MMA; the rate is not on the pages).  Outputs: the median over
 * SMs of FLOP per SM clock, the aggregate FLOP/s over all SMs (TFLOP/s) and
 * the median SM clock it ran at (GHz).  mmas in [1, 2^20]; synchronous; the
 * device is made current.  GEMM_ERR_UNSUPPORTED off compute capability 10.3,
 * GEMM_ERR_TIMEOUT if the MMAs did not complete within 2 s. */
gemm_status_t gemm_tensor_peak_probe(int device, gemm_dtype_t dtype, int cta_group, int64_t mmas,
                                     double *flop_per_clk_per_sm, double *tflops, double *sm_ghz);

/* Launch shape gemm_run would use (no GPU work).  Same argument rules. */
gemm_status_t gemm_query(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                         gemm_dtype_t dtype, gemm_sched_t sched, gemm_launch_info_t *info);

/* Synchronise `stream`, read and clear the device status block.
 * device_status (may be NULL) receives the raw first error word (0 = none).
 * Returns GEMM_ERR_TIMEOUT if a device wait timed out since the last check.
 * After an error it also zeroes the handle's stream-K claim counters and
 * ready flags, which a launch that stopped early may have left set. */
gemm_status_t gemm_check(gemm_handle_t h, void *stream, int *device_status);

/* After a run with GEMM_DEBUG_RECORDS: synchronise `stream`, copy the
 * n_work records of the last run (work-id order; n_work must equal its
 * work_items) to host memory `records`, and do what gemm_check does.
 * Returns GEMM_ERR_COVERAGE if any visits count differs from the cta_group of
 * the last run. */
gemm_status_t gemm_read_debug(gemm_handle_t h, void *stream, gemm_tile_record_t *records,
                              int64_t n_work, int *device_status);

/* ---- allocation-free entry point ---------------------------------------
 * The paper has no counterpart to this call; it exists for callers that
 * cannot allocate device memory when they need a GEMM: runtimes that reserve
 * all device memory at start-up and refuse later allocations, and
 * latency-critical loops that cannot accept the implicit synchronisation
 * cudaMalloc / cudaFree may perform.  gemm_create allocates, so those callers
 * cannot use the handle API.
 *
 * gemm_run_noalloc computes C = A . B exactly like gemm_run (same layouts,
 * size and alignment rules, K == 0 writes zeros) on the CURRENT device, with
 * the default options (group_size_m 8, deepest ring, automatic last-wave
 * slicing, 1 s wait limit) and the given cta_group (1 or 2).  It allocates
 * nothing: no cudaMalloc, no cudaFree, no host heap.  The kernel's scratch --
 * a 4-word device status block and one gemm_tile_record_t per work item (the
 * coverage counters) -- lives in a file-scope __device__ array of
 * 256 + 52 * GEMM_NOALLOC_MAX_WORK_ITEMS bytes (832.25 KiB) that every GPU which
 * loads the library holds until the process exits.
 *   - Problems with more than GEMM_NOALLOC_MAX_WORK_ITEMS work items are
 *     rejected with GEMM_ERR_INVALID_ARG before anything is launched (work
 *     items = output tiles of 128x256 for cta_group 1 or 256x256 for
 *     cta_group 2, plus up to 3 per tile of a problem smaller than one
 *     wave, or 1 per tile of a partial last wave run as column halves; the
 *     stream-K share is never used here).
 *   - The first call on a device does a one-time set-up on that device (the
 *     scratch array's device address via cudaGetSymbolAddress, kernel
 *     attributes, occupancy); make that first call before any stream capture.
 *     Only a set-up that succeeds is kept: if it fails, that call returns
 *     the error and the next call on the device tries the set-up again.
 *   - Every call clears the status block and its work items' records with a
 *     cudaMemsetAsync on `stream`, then launches on `stream`.
 *   - All calls share the one scratch array, which keeps the last call's
 *     contents: calls whose kernels overlap on the GPU (different streams,
 *     or different host threads) race on it.  Order them on one stream.
 *   - device_status == NULL: asynchronous, returns after the launch (device
 *     errors are then not reported).  Otherwise the call synchronises
 *     `stream`, stores the raw first device error word (0 = none) and returns
 *     GEMM_ERR_TIMEOUT on a device wait time-out, GEMM_ERR_COVERAGE if a work
 *     item was not stored exactly once by its CTA (pair), else GEMM_OK. */
#define GEMM_NOALLOC_MAX_WORK_ITEMS 16384
gemm_status_t gemm_run_noalloc(int64_t M, int64_t N, int64_t K,
                               const void *A, const void *B, void *C,
                               gemm_dtype_t dtype, gemm_sched_t sched,
                               float scale_a, float scale_b, int cta_group,
                               void *stream, int *device_status);

/* Free the handle and everything it owns.  NULL is accepted. */
gemm_status_t gemm_destroy(gemm_handle_t h);

/* Static string for a status code (never NULL). */
const char *gemm_status_string(gemm_status_t s);

#ifdef __cplusplus
}
#endif

#endif /* PTS_GEMM_H */
