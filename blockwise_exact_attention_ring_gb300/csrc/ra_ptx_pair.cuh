// Inline-PTX helpers for kernels launched as clusters of two CTAs: the
// CTA-pair kernel, whose tcgen05 MMAs use cta_group::2 (one MMA spans both
// CTAs' tensor memory and shared memory), and the single-CTA kernel's
// cluster form, whose two CTAs share each key/value tile load by TMA
// multicast.  Builds on the single-CTA helpers of ra_ptx.cuh.
#pragma once

#include "ra_ptx.cuh"

namespace ra {

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Shared-memory address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Arrive on an mbarrier given by its shared::cluster address (any CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait with cluster-scope acquire (barriers that receive arrivals or
// copies from the peer CTA).
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, volatile int *abort,
                                                  uint64_t timeout_ns, unsigned int *status,
                                                  unsigned int site)
{
    if (mbar_try_wait_cluster(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_cluster(bar, parity))
            return true;
        if ((it & 63u) == 0) {
            if (*abort)
                return false;
            if (globaltimer_ns() - t0 > timeout_ns) {
                record_error(status, RA_DEV_TIMEOUT, site);
                *abort = 1;
                return false;
            }
        }
    }
}

// 2-D tiled TMA load into this CTA's shared memory whose completion is
// counted on `bar_cluster` (an mbarrier of either CTA of the pair).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void *tmap, int x, int y,
                                                 uint32_t bar_cluster, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(bar_cluster), "l"(policy)
        : "memory");
}

// 2-D tiled TMA load multicast to the CTAs in `mask`: the box lands at the
// same shared-memory offset `dst` in each of them and completes `bar` (same
// offset) in each.
__device__ __forceinline__ void tma_load_2d_mc(uint32_t dst, const void *tmap, int x, int y, uint32_t bar,
                                               uint16_t mask, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5, %6;"
        ::"r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(bar), "h"(mask), "l"(policy)
        : "memory");
}

// Arrive once on the mbarrier at offset `bar` in each CTA of `mask` when
// every tcgen05 operation this thread issued so far (cta_group::1) has
// completed.
__device__ __forceinline__ void mma_commit_mc(uint32_t bar, uint16_t mask)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
                 " [%0], %1;" ::"r"(bar), "h"(mask) : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(dst_smem), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;"
                 ::"r"(taddr), "r"(ncols) : "memory");
}

// D (+)= A[tmem] * B[smem desc] across the CTA pair (M = 256: each CTA holds
// 128 rows of A and D; B is split along N, half in each CTA).
__device__ __forceinline__ void mma_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// D (+)= A[smem desc] * B[smem desc] across the CTA pair (each CTA holds its
// 128 rows of A in its own shared memory at the same offset).
__device__ __forceinline__ void mma_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// Arrive once on the mbarrier at the same offset in both CTAs of the pair
// when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
                 " [%0], %1;" ::"r"(bar), "h"((uint16_t)3) : "memory");
}

// Cluster-wide barrier; every thread of both CTAs arrives individually.
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

}  // namespace ra
