// Inline-PTX helpers for the single-CTA kernel's cluster form, whose two CTAs
// share each key/value tile load by TMA multicast (within this GPU's own
// memory).  Builds on the single-CTA helpers of ra_ptx.cuh.
#pragma once

#include "ra_ptx.cuh"

namespace ra {

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
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

// Cluster-wide barrier; every thread of both CTAs arrives individually.
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

}  // namespace ra
