// Work order of the backward pass, shared by the kernels and the host export
// that tests check (ra_backward_tile_pairs).
//
// On a ring, key/value block j and its gradient accumulators travel: at ring
// step s they sit on device i = (j + s) mod N, which adds the contribution of
// its query block i ("Ring Attention" glossary page, ultralytics.com/tr,
// section "Halka Dikkati Nasil Calisir": blocks pass from each device to the
// next).  The dK/dV kernel follows that order for one 128-key tile; the dQ
// kernel walks the key blocks of one query tile in the forward's order
// j = (i - s) mod N.
#pragma once

#include "ra_schedule.h"

// Query tiles that meet key tile tb of block j, in ring order: step s, then
// the kv group's query heads hh, then the query tiles ta that see the key
// tile (all of them on a full block, ta >= tb on a diagonal block).
struct RaQWalk {
    int j, tb, N, layout, causal, ntiles, grp;
    int s, i, cls, hh, ta;

    RA_HD void start(int j_, int tb_, int N_, int layout_, int causal_, int ntiles_, int grp_)
    {
        j = j_, tb = tb_, N = N_, layout = layout_, causal = causal_, ntiles = ntiles_, grp = grp_;
        s = -1, i = 0, cls = 0, hh = 0, ta = 0;
        next_block();
    }
    RA_HD int ta_first() const { return cls == RA_CLS_FULL ? 0 : tb; }
    RA_HD void next_block()
    {
        while (++s < N) {
            i = (j + s) % N;
            cls = ra_block_class(layout, causal, i, j);
            if (cls != RA_CLS_SKIP && ta_first() < ntiles) {
                hh = 0, ta = ta_first();
                return;
            }
        }
    }
    RA_HD bool valid() const { return s < N; }
    RA_HD void advance()
    {
        if (++ta < ntiles)
            return;
        if (++hh < grp) {
            ta = ta_first();
            return;
        }
        next_block();
    }
};

// Key tiles one query tile meets, in the forward's ring order.
struct RaKWalk {
    int i, ta, N, layout, causal, ntiles;
    int s, j, cls, nt, tb;

    RA_HD void start(int i_, int ta_, int N_, int layout_, int causal_, int ntiles_)
    {
        i = i_, ta = ta_, N = N_, layout = layout_, causal = causal_, ntiles = ntiles_;
        s = -1, j = 0, cls = 0, nt = 0, tb = 0;
        next_block();
    }
    RA_HD void next_block()
    {
        tb = 0;
        while (++s < N) {
            j = ra_ring_block(i, s, N);
            cls = ra_block_class(layout, causal, i, j);
            nt = ra_kv_tiles(cls, ta, ntiles);
            if (nt > 0)
                return;
        }
    }
    RA_HD bool valid() const { return s < N; }
    RA_HD void advance()
    {
        if (++tb >= nt)
            next_block();
    }
};

// Unit u of the dK/dV kernel -> (batch * Hkv + kv head, block j, key tile tb),
// heaviest first: contiguous causal blocks are seen by every later block, so
// ascending (j, tb); otherwise tb ascending outermost (early key tiles of a
// block meet more query tiles on diagonal blocks).  With kv_outer (the K/V of
// all heads far exceed L2, as in the forward's dealing order) the kv head is
// the outermost index, so the units in flight stream one kv group's Q and dO
// together; otherwise it is the fastest one.
RA_HD void ra_bwd_dkdv_unit(int u, int B, int Hkv, int N, int ntiles, int layout, int kv_outer, int &bhkv, int &j,
                            int &tb)
{
    const int nkv = B * Hkv;
    int r;
    if (kv_outer) {
        const int per_kv = N * ntiles;
        bhkv = u / per_kv;
        r = u - bhkv * per_kv;
    } else {
        bhkv = u % nkv;
        r = u / nkv;
    }
    if (layout == 0) {
        j = r / ntiles, tb = r % ntiles;
    } else {
        tb = r / N, j = r % N;
    }
}

// Unit u of the dQ kernel -> (batch * H + head, block i, query tile ta),
// latest in the causal order (heaviest) first.  With kv_outer the kv group is
// the outermost index and its query heads the fastest, so the units in flight
// walk one kv head's K and V together; otherwise the head is the fastest
// index over all heads.
RA_HD void ra_bwd_dq_unit(int u, int B, int H, int Hkv, int N, int ntiles, int layout, int kv_outer, int &bh, int &i,
                          int &ta)
{
    const int nq = B * H;
    int r;
    if (kv_outer) {
        const int grp = H / Hkv;
        const int per_kv = grp * N * ntiles;
        const int kvi = u / per_kv;                   // batch * Hkv + kv head
        const int rem = u - kvi * per_kv;
        const int b = kvi / Hkv;
        bh = b * H + (kvi - b * Hkv) * grp + rem % grp;
        r = rem / grp;
    } else {
        bh = u % nq;
        r = u / nq;
    }
    if (layout == 0) {
        const int q = N * ntiles - 1 - r;
        i = q / ntiles, ta = q % ntiles;
    } else {
        ta = ntiles - 1 - r / N, i = N - 1 - r % N;
    }
}

// Whether the backward kernels deal their units by kv head (the forward's
// rule: B * Hkv * S key/value rows at or above RA_KV_OUTER_ROWS).
RA_HD int ra_bwd_kv_outer(int B, int Hkv, int S)
{
    return (long long)B * Hkv * S >= RA_KV_OUTER_ROWS ? 1 : 0;
}
