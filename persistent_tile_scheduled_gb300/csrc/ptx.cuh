// Inline-PTX wrappers for sm_103a: mbarrier, TMA (cp.async.bulk.tensor),
// tcgen05 (TMEM alloc, MMA, commit, loads, fences) and Cluster Launch Control.
// Every form is written against the PTX ISA for sm_100-family targets.
#pragma once
#include <cstdint>

namespace pts {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smid()
{
    uint32_t s;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(s));
    return s;
}

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory object in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank)
{
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(addr), "r"(rank));
    return out;
}

__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

__device__ __forceinline__ void st_cluster_v4(uint32_t cluster_addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(cluster_addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Arrive on a barrier given by its shared::cluster address (own or peer CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Predicated forms (`_if`, or a leading `pred` argument below): the
// instruction executes only in the lanes whose `pred` is non-zero.  The
// producer and MMA warps run their loops with all 32 lanes in step and issue
// from lane 0 through these, so the per-k-block path has no divergent branch.
__device__ __forceinline__ void mbar_arrive_if(uint32_t pred, uint32_t bar)
{
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %0, 0;\n\t"
                 "@q mbarrier.arrive.shared::cta.b64 _, [%1];\n\t}" ::"r"(pred), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster_if(uint32_t pred, uint32_t cluster_bar)
{
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %0, 0;\n\t"
                 "@q mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%1];\n\t}" ::"r"(pred),
                 "r"(cluster_bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx_if(uint32_t pred, uint32_t bar, uint32_t bytes)
{
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %0, 0;\n\t"
                 "@q mbarrier.arrive.expect_tx.shared::cta.b64 _, [%1], %2;\n\t}" ::"r"(pred), "r"(bar),
                 "r"(bytes)
                 : "memory");
}

// Non-blocking probe of phase `parity`; cluster-scope acquire so that arrivals
// and async writes made by the peer CTA of a pair are visible afterwards.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}

// --------------------------------------------------------------------- TMA

__device__ __forceinline__ void prefetch_tmap(const void *tmap)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// Order this thread's later uses of the 128-byte tensor map at `tmap` (in
// global memory) after the generic-proxy writes that filled it, such as a
// table the host rewrote between launches.  Only where `pred` is non-zero.
__device__ __forceinline__ void tmap_acquire(uint32_t pred, const void *tmap)
{
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %0, 0;\n\t"
                 "@q fence.proxy.tensormap::generic.acquire.gpu [%1], 128;\n\t}" ::"r"(pred),
                 "l"(tmap)
                 : "memory");
}

// 2-D tiled load into this CTA's shared memory; completion is signalled on
// `bar` (shared::cta address of this CTA).
// (Only in the lanes where `pred` is non-zero.)
__device__ __forceinline__ void tma_load_2d(uint32_t pred, uint32_t dst, const void *tmap, uint32_t bar,
                                            int x, int y)
{
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %0, 0;\n\t"
                 "@q cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%1], [%2, {%4, %5}], [%3];\n\t}" ::"r"(pred),
                 "r"(dst), "l"(tmap), "r"(bar), "r"(x), "r"(y)
                 : "memory");
}

// Same for a CTA pair: data lands in this CTA's shared memory, completion is
// signalled on `cluster_bar`, which may live in the peer CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t pred, uint32_t dst, const void *tmap,
                                                 uint32_t cluster_bar, int x, int y)
{
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %0, 0;\n\t"
                 "@q cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 ".cta_group::2 [%1], [%2, {%4, %5}], [%3];\n\t}" ::"r"(pred),
                 "r"(dst), "l"(tmap), "r"(cluster_bar), "r"(x), "r"(y)
                 : "memory");
}

// Bring a 2-D box of the tensor into L2 (no shared-memory destination, no
// completion); out-of-bounds parts are ignored.
__device__ __forceinline__ void tma_prefetch_2d(uint32_t pred, const void *tmap, int x, int y)
{
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %0, 0;\n\t"
                 "@q cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%1, {%2, %3}];\n\t}" ::"r"(pred),
                 "l"(tmap), "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// TMA store of a shared-memory box, only where `pred` is non-zero.
__device__ __forceinline__ void tma_store_2d_if(uint32_t pred, const void *tmap, uint32_t src, int x, int y)
{
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %0, 0;\n\t"
                 "@q cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%1, {%3, %4}], [%2];\n\t}"
                 ::"r"(pred), "l"(tmap), "r"(src), "r"(x), "r"(y)
                 : "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Order this thread's generic-proxy shared-memory accesses with later
// async-proxy accesses (TMA store source, CLC response slot reuse).
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------- tcgen05

template <int CG>
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    if constexpr (CG == 1)
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                     "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                     "r"(ncols)
                     : "memory");
}

template <int CG>
__device__ __forceinline__ void tmem_relinquish()
{
    if constexpr (CG == 1)
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    else
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

template <int CG>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    if constexpr (CG == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                     : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] . B[smem]^T, both operands K-major.  KIND 0/1: f16/bf16
// (kind::f16), KIND 2: e4m3 (kind::f8f6f4).  Issued only where `pred` is
// non-zero (one lane of the MMA warp).
template <int KIND, int CG>
__device__ __forceinline__ void umma(uint32_t pred, uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                     uint32_t idesc, uint32_t accumulate)
{
#define PTS_UMMA(K_, G_)                                                                              \
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %4, 0;\n\tsetp.ne.b32 q, %5, 0;\n\t"         \
                 "@q tcgen05.mma.cta_group::" #G_ ".kind::" #K_ " [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem), \
                 "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(pred)                       \
                 : "memory")
    if constexpr (KIND == 2 && CG == 1) PTS_UMMA(f8f6f4, 1);
    else if constexpr (KIND == 2 && CG == 2) PTS_UMMA(f8f6f4, 2);
    else if constexpr (CG == 1) PTS_UMMA(f16, 1);
    else PTS_UMMA(f16, 2);
#undef PTS_UMMA
}

// Arrive (once) on `bar` when every tcgen05 operation this thread issued so
// far has completed.  CG 2: the arrival is multicast to the barrier at the
// same offset in each CTA of `cta_mask`.  Only where `pred` is non-zero: the
// lane that issued the MMAs.
template <int CG>
__device__ __forceinline__ void umma_commit(uint32_t pred, uint32_t bar, uint16_t cta_mask)
{
    if constexpr (CG == 1)
        asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %0, 0;\n\t"
                     "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%1];\n\t}"
                     ::"r"(pred), "r"(bar)
                     : "memory");
    else
        asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %0, 0;\n\t"
                     "@q tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
                     " [%1], %2;\n\t}" ::"r"(pred),
                     "r"(bar), "h"(cta_mask)
                     : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t gets lane (base + t).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
                 "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
                   "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
                   "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
                   "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
                   "=r"(r[31])
                 : "r"(taddr)
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ------------------------------------------------ global-memory ordering

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ------------------------------------------ programmatic dependent launch

// Let the next grid in the stream (launched with programmatic stream
// serialization) be scheduled once every CTA of this grid has called this or
// exited.  It does not release any data: the next grid still waits below.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Block until the grids this one depends on have completed and their memory
// is visible; returns at once when there is no such dependency.
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------- Cluster Launch Control

// Ask the hardware to cancel a cluster of this grid that has not launched
// yet.  The 16-byte response is written asynchronously to `resp` and
// signalled on `bar` as a 16-byte transaction.
__device__ __forceinline__ void clc_try_cancel(uint32_t resp, uint32_t bar)
{
    asm volatile("clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128"
                 " [%0], [%1];" ::"r"(resp),
                 "r"(bar)
                 : "memory");
}

// Decode a response: returns true and the x index of the first CTA of the
// cancelled cluster, or false when the request failed.
__device__ __forceinline__ bool clc_decode(uint32_t resp_smem, uint32_t &first_ctaid_x)
{
    uint64_t lo, hi;
    asm volatile("ld.shared.v2.u64 {%0, %1}, [%2];" : "=l"(lo), "=l"(hi) : "r"(resp_smem) : "memory");
    uint32_t ok, x;
    asm volatile("{\n\t.reg .b128 r;\n\t.reg .pred p;\n\t"
                 "mov.b128 r, {%2, %3};\n\t"
                 "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t"
                 "clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, r;\n\t}"
                 : "=r"(ok), "=r"(x)
                 : "l"(lo), "l"(hi));
    first_ctaid_x = x;
    return ok != 0;
}

}  // namespace pts
