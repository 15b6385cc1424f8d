// Per-row pieces of the tensor-core forward kernel (ra_attn_sm103.cu): the
// walk over a unit's key tiles in ring order, the dealing order of units, one
// online-softmax step of a query row, and the epilogue that divides by the
// running sum and stores a row.
//
// Method ("Ring Attention" glossary page, ultralytics.com/tr, section "Halka
// Dikkati Nasil Calisir"): query block i meets key/value block
// j = (i - s) mod N at ring step s; each block's scores are exponentiated
// against a running maximum and folded into a running sum and a running
// score-weighted value sum, which are divided at the end.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "ra_ptx.cuh"
#include "ra_schedule.h"

namespace ra {

constexpr float RA_LAZY_RESCALE_LOG2 = 8.0f;
constexpr float RA_LN2 = 0.693147180559945309f;

// Walks the key tiles of one unit in ring order: steps s in [s_begin, s_end),
// block j = (i - s) mod N, tiles tb in [0, ra_kv_tiles(...)).  P is the
// kernel's parameter block (fields N, layout, causal, ntiles, s_begin, s_end).
struct KvWalk {
    int i, N, layout, causal, ntiles, ta_max, s_end;
    int s, j, cls, nt, tb;

    template <class P>
    __device__ void start(int rank, int tmax, const P &p)
    {
        i = rank, N = p.N, layout = p.layout, causal = p.causal, ntiles = p.ntiles;
        ta_max = tmax, s_end = p.s_end, s = p.s_begin - 1, j = 0, cls = 0, nt = 0;
        next_block();
    }
    __device__ void next_block()
    {
        tb = 0;
        while (++s < s_end) {
            j = ra_ring_block(i, s, N);
            cls = ra_block_class(layout, causal, i, j);
            nt = ra_kv_tiles(cls, ta_max, ntiles);
            if (nt > 0)
                return;
        }
    }
    __device__ bool valid() const { return s < s_end; }
    __device__ void advance()
    {
        if (++tb >= nt)
            next_block();
    }
    // Moves n key tiles ahead along the walk (a block at a time).
    __device__ void skip(int n)
    {
        while (n > 0 && valid()) {
            const int left = nt - tb;
            if (n < left) {
                tb += n;
                return;
            }
            n -= left;
            next_block();
        }
    }
};

// Units are dealt to CTAs (or clusters) in snake order over the
// heaviest-first enumeration.
__device__ __forceinline__ int unit_index(int round, int cta, int G)
{
    return round * G + ((round & 1) ? (G - 1 - cta) : cta);
}

// One online-softmax step for the query row this thread owns.  The row's 128
// scores of the current key tile are read from TMEM once (two 64-column
// loads, one wait); on unmasked tiles the loads also return each half row's
// maximum (tcgen05.ld.red), so no max pass over the registers is needed;
// columns at or past `lim` count as -inf when MASK.  The
// running max m (log2 domain, scores scaled by sl2 = log2e / sqrt(d)) only
// moves when the tile max exceeds it by more than 2^8, and then O (in TMEM,
// when has_o) and l are rescaled by 2^(m_old - m_new); the final division
// cancels the common factor, so the result is exact.  P = 2^(s sl2 - m) is
// packed to bf16 pairs over the first 64 columns of the tile (all scores are
// in registers by then) for the P V MMA, and l accumulates the fp32 P.
template <int D, bool MASK>
__device__ __forceinline__ void softmax_step(uint32_t tS, uint32_t tO, int lim, float sl2, bool has_o,
                                             float &m_run, float &l_run)
{
    const uint32_t ninf = __float_as_uint(-INFINITY);
    float ma = -INFINITY, mb = -INFINITY;
    uint32_t xa[64], xb[64];
    if (MASK) {
        tmem_ld64(tS, xa);
        tmem_ld64(tS + 64, xb);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 64; ++e) {
            xa[e] = e < lim ? xa[e] : ninf;
            xb[e] = e + 64 < lim ? xb[e] : ninf;
        }
#pragma unroll
        for (int e = 0; e < 64; e += 2) {
            ma = max3f(ma, __uint_as_float(xa[e]), __uint_as_float(xa[e + 1]));
            mb = max3f(mb, __uint_as_float(xb[e]), __uint_as_float(xb[e + 1]));
        }
    } else {
        // the tensor-memory load reduces each half row to its maximum itself
        tmem_ld64_max(tS, xa, ma);
        tmem_ld64_max(tS + 64, xb, mb);
        tmem_wait_ld();
        asm volatile("" : "+f"(ma), "+f"(mb));  // keep every use of the maxima after the wait
    }
    const float m_tile = fmaxf(ma, mb) * sl2;  // -inf stays -inf
    const bool resc = m_tile > m_run + RA_LAZY_RESCALE_LOG2;
    float alpha = 1.f;
    if (resc) {
        alpha = ex2_approx(m_run - m_tile);  // 0 when m_run = -inf
        m_run = m_tile;
        l_run *= alpha;
    }
    const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
    const float2 scale = make_float2(sl2, sl2), shift = make_float2(neg_m, neg_m);
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const uint32_t u0 = h ? xb[2 * e] : xa[2 * e];
            const uint32_t u1 = h ? xb[2 * e + 1] : xa[2 * e + 1];
            const float2 t2 = ffma2(make_float2(__uint_as_float(u0), __uint_as_float(u1)), scale, shift);
            const float2 pv = make_float2(ex2_approx(t2.x), ex2_approx(t2.y));
            if (e & 1)
                acc1 = fadd2(acc1, pv);
            else
                acc0 = fadd2(acc0, pv);
            pk[e] = pack_bf16x2(pv.x, pv.y);
        }
        tmem_st32(tS + h * 32, pk);
    }
    const float2 acc = fadd2(acc0, acc1);
    l_run += acc.x + acc.y;
    if (has_o && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e)
                o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tO + c * 32, o);
        }
    }
}

// The same step for one half of the row's 128 columns (64 keys) with its own
// running max m, sum l and accumulator O (D columns at tO): a query tile whose
// two column halves are handled by two threads, each an online softmax over
// its own key subset, merged at the end (merge_halves_store_row).  lim counts
// from the half's first column; P goes to the half's first 32 columns, which
// only this thread reads.
template <int D, bool MASK>
__device__ __forceinline__ void softmax_half(uint32_t tS, uint32_t tO, int lim, float sl2, bool has_o,
                                             float &m_run, float &l_run)
{
    const uint32_t ninf = __float_as_uint(-INFINITY);
    float ma = -INFINITY;
    uint32_t xa[64];
    if (MASK) {
        tmem_ld64(tS, xa);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 64; ++e)
            xa[e] = e < lim ? xa[e] : ninf;
#pragma unroll
        for (int e = 0; e < 64; e += 2)
            ma = max3f(ma, __uint_as_float(xa[e]), __uint_as_float(xa[e + 1]));
    } else {
        tmem_ld64_max(tS, xa, ma);
        tmem_wait_ld();
        asm volatile("" : "+f"(ma));  // keep every use of the maximum after the wait
    }
    const float m_tile = ma * sl2;
    const bool resc = m_tile > m_run + RA_LAZY_RESCALE_LOG2;
    float alpha = 1.f;
    if (resc) {
        alpha = ex2_approx(m_run - m_tile);
        m_run = m_tile;
        l_run *= alpha;
    }
    const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
    const float2 scale = make_float2(sl2, sl2), shift = make_float2(neg_m, neg_m);
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
    uint32_t pk[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        const float2 t2 = ffma2(make_float2(__uint_as_float(xa[2 * e]), __uint_as_float(xa[2 * e + 1])), scale, shift);
        const float2 pv = make_float2(ex2_approx(t2.x), ex2_approx(t2.y));
        if (e & 1)
            acc1 = fadd2(acc1, pv);
        else
            acc0 = fadd2(acc0, pv);
        pk[e] = pack_bf16x2(pv.x, pv.y);
    }
    tmem_st32(tS, pk);
    const float2 acc = fadd2(acc0, acc1);
    l_run += acc.x + acc.y;
    if (has_o && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e)
                o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tO + c * 32, o);
        }
    }
}

// Epilogue of one query row whose key columns were split between two threads
// (softmax_half): this thread, half h, holds (m_own, l_own) and knows the
// other half's (m_oth, l_oth); O of half g sits at tO + g D.  The halves merge
// like two blocks of the ring: m = max, weights 2^(m_g - m), l = sum of the
// weighted l_g, O = sum of the weighted O_g, out = O / l; thread h stores
// output columns [h D/2, (h + 1) D/2), half 0 the log-sum-exp.  Every thread
// of the warp must call it (the TMEM loads are warp-collective).
template <int D>
__device__ __forceinline__ void merge_halves_store_row(uint32_t tO, int h, bool valid, long long orow, float m_own,
                                                       float l_own, float m_oth, float l_oth, void *out, float *lse,
                                                       int out_f32)
{
    const float m = fmaxf(m_own, m_oth);
    float w_own = 0.f, w_oth = 0.f;
    if (m != -INFINITY) {
        w_own = ex2_approx(m_own - m);  // 0 for a half that saw no key
        w_oth = ex2_approx(m_oth - m);
    }
    const float w0 = h ? w_oth : w_own, w1 = h ? w_own : w_oth;
    const float l = h ? l_oth * w0 + l_own * w1 : l_own * w0 + l_oth * w1;  // the same sum in both threads
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float s0 = w0 * inv, s1 = w1 * inv;
#pragma unroll 1
    for (int c = 0; c < D / 64; ++c) {
        const int col = h * (D / 2) + c * 32;
        uint32_t o0[32], o1[32];
        __syncwarp();
        tmem_ld32(tO + col, o0);
        tmem_ld32(tO + D + col, o1);
        tmem_wait_ld();
        if (!valid)
            continue;
        float v[32];
#pragma unroll
        for (int e = 0; e < 32; ++e)
            v[e] = __uint_as_float(o0[e]) * s0 + __uint_as_float(o1[e]) * s1;
        if (out_f32) {
            float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(out) + orow * D + col);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                dst[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
        } else {
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(out) + orow * D + col);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                uint4 x;
                x.x = pack_bf16x2(v[8 * e + 0], v[8 * e + 1]);
                x.y = pack_bf16x2(v[8 * e + 2], v[8 * e + 3]);
                x.z = pack_bf16x2(v[8 * e + 4], v[8 * e + 5]);
                x.w = pack_bf16x2(v[8 * e + 6], v[8 * e + 7]);
                dst[e] = x;
            }
        }
    }
    if (valid && h == 0)
        lse[orow] = l > 0.f ? (m + log2f(l)) * RA_LN2 : -INFINITY;
}

// Epilogue of one query row: reads O (D fp32 columns at tO) from TMEM, divides
// by the running sum l_run and, when `valid`, stores the row (bf16 rounded to
// nearest even, or fp32 when out_f32) at row `orow` of `out` and its
// log-sum-exp (natural log; -inf for a row that saw no key) at lse[orow].
// Every thread of the warp must call it (the TMEM loads are warp-collective).
template <int D>
__device__ __forceinline__ void store_row(uint32_t tO, bool valid, long long orow, float m_run, float l_run,
                                          void *out, float *lse, int out_f32)
{
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        __syncwarp();
        tmem_ld32(tO + c * 32, o);
        tmem_wait_ld();
        if (!valid)
            continue;
        if (out_f32) {
            float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(out) + orow * D + c * 32);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                dst[e] = make_float4(__uint_as_float(o[4 * e]) * inv, __uint_as_float(o[4 * e + 1]) * inv,
                                     __uint_as_float(o[4 * e + 2]) * inv, __uint_as_float(o[4 * e + 3]) * inv);
        } else {
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(out) + orow * D + c * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                uint4 x;
                x.x = pack_bf16x2(__uint_as_float(o[8 * e + 0]) * inv, __uint_as_float(o[8 * e + 1]) * inv);
                x.y = pack_bf16x2(__uint_as_float(o[8 * e + 2]) * inv, __uint_as_float(o[8 * e + 3]) * inv);
                x.z = pack_bf16x2(__uint_as_float(o[8 * e + 4]) * inv, __uint_as_float(o[8 * e + 5]) * inv);
                x.w = pack_bf16x2(__uint_as_float(o[8 * e + 6]) * inv, __uint_as_float(o[8 * e + 7]) * inv);
                dst[e] = x;
            }
        }
    }
    if (valid)
        lse[orow] = l_run > 0.f ? (m_run + log2f(l_run)) * RA_LN2 : -INFINITY;
}

}  // namespace ra
