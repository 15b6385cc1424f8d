// Tensor-core ring-ordered blockwise attention on CTA pairs (cta_group::2),
// sm_103a, head dimension 128.
//
// Same method as ra_attn_sm103.cu ("Ring Attention" glossary page,
// ultralytics.com/tr, section "Halka Dikkati Nasil Calisir": query blocks stay
// in place, key/value blocks arrive in ring order j = (i - s) mod N, the
// running max / sum / weighted sum are merged per block and divided at the
// end), laid out for a pair of SMs:
//
//   * a cluster of two CTAs runs one work unit (two 128-row query tiles that
//     share a kv head); CTA r owns query tile r.  One tcgen05.mma with
//     cta_group::2 computes both tiles at once (M = 256): each CTA holds its
//     own Q tile in shared memory and its P in tensor memory (the A operand)
//     and HALF of every K and V tile in shared memory (the B operand is split
//     along N), so each SM stages only half the key/value bytes per FLOP;
//   * with one query tile per CTA, tensor memory has room for three S
//     buffers: S(j + 1) and S(j + 2) are computed while the softmax of S(j)
//     runs, and only P(j) -> O += P V waits for the softmax;
//   * eight softmax warps per CTA, two per TMEM lane quarter: each thread
//     owns half a row (64 scores) whose max comes with its tensor-memory
//     load (tcgen05.ld.red, except on masked tiles), and the two halves
//     exchange their row max through shared memory each step;
//   * the leader CTA (rank 0) issues all MMAs; its barriers receive the
//     peer's TMA bytes and softmax arrivals; MMA completions are multicast to
//     both CTAs;
//   * every wait is bounded, as in the single-CTA kernel.
//
// Measured on GB300 this layout is slower than the single-CTA kernel (about
// 0.6x): each CTA has a single query tile in flight, so its MMA warp waits
// for every P(j) before it can issue P V(j) and S(j + 3), and the pair MMAs
// take ~1.7x their isolated issue time in situ.  It is kept as a selectable,
// parity-tested alternative.
//
// TMEM columns per CTA: S/P buffers [0,128), [128,256), [256,384); O [384,512).
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "ra_internal.h"
#include "ra_ptx_pair.cuh"

namespace ra {


namespace {

constexpr int P_THREADS = 384;  // warps: 0 TMA, 1 MMA + TMEM, 2-3 spare, 4-11 softmax
constexpr int P_D = 128;
constexpr uint32_t P_TMEM_COLS = 512;
constexpr int NSB = 3;              // S / P buffers in TMEM
constexpr uint32_t COL_O = 384;
constexpr int KST = 4, VST = 4;
constexpr int K_HALF = 64 * 128 * 2;   // 64 keys x 128 d: two 8 KB swizzled slabs
constexpr int V_HALF = 128 * 64 * 2;   // 128 keys x 64 d: one 16 KB swizzled slab
constexpr int Q_TILE = 128 * 128 * 2;  // this CTA's query tile: two 16 KB swizzled slabs
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + Q_TILE;
constexpr int OFF_V = OFF_K + KST * K_HALF;
constexpr int OFF_X = OFF_V + VST * V_HALF;  // half-row exchange: 3 buffers x 2 halves x 128 floats
constexpr int OFF_CTRL = OFF_X + 3 * 2 * 128 * 4;
constexpr int P_SMEM = OFF_CTRL + 512 + 1024;
constexpr float P_LAZY_LOG2 = 8.0f;
constexpr float P_LN2 = 0.693147180559945309f;

enum : unsigned int {
    PS_K_EMPTY = 21, PS_V_EMPTY, PS_K_FULL, PS_V_FULL, PS_P_FULL, PS_O_FREE, PS_S_FULL,
    PS_Q_EMPTY, PS_Q_FULL,
    PS_O_DONE, PS_XCH, PS_DRAIN
};

struct PairCtrl {
    uint64_t k_full[KST], k_empty[KST], v_full[VST], v_empty[VST];
    uint64_t s_full[NSB], p_full[NSB], o_done[NSB], o_free, q_full, q_empty, xch[3], final_bar;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(PairCtrl) <= 512, "control block");

struct PairParams {
    CUtensorMap tm_q, tm_k, tm_v;
    RaUnitSpace sp;
    void *out;
    float *lse;
    long long q_rows;  // B * H * S
    int n_units, H, Hkv, S, L, N, layout, causal, s_begin, s_end, out_f32, ntiles;
    float scale_log2;
    unsigned long long timeout_ns;
    unsigned int *status;  // the library's device status word
};

struct Walk {
    int i, N, layout, causal, ntiles, ta_max, s_end;
    int s, j, cls, nt, tb;
    __device__ void start(int rank, int tmax, const PairParams &p)
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
};

__device__ __forceinline__ int pair_unit_index(int round, int cluster, int G)
{
    return round * G + ((round & 1) ? (G - 1 - cluster) : cluster);
}

// Waits record a timeout in the library's status word, whose device address
// the launch passes in (`st`).
__device__ __forceinline__ bool pwait(unsigned int *st, uint32_t bar, uint32_t parity, volatile int *abort,
                                      uint64_t tmo, unsigned int site)
{
    return mbar_wait_cluster(bar, parity, abort, tmo, st, site);
}

__device__ __forceinline__ bool pwait_warp(unsigned int *st, uint32_t bar, uint32_t parity,
                                           volatile int *abort, uint64_t tmo, unsigned int site)
{
    return __all_sync(0xffffffffu, pwait(st, bar, parity, abort, tmo, site));
}

__device__ __forceinline__ void pdrain(unsigned int *st, uint32_t bar, uint32_t parity, uint64_t tmo)
{
    int never = 0;
    mbar_wait_cluster(bar, parity, &never, tmo, st, PS_DRAIN);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(P_THREADS, 1)
ra_attn_pair_kernel(const __grid_constant__ PairParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);
    PairCtrl *ctrl = reinterpret_cast<PairCtrl *>(smem + OFF_CTRL);
    float *xch = reinterpret_cast<float *>(smem + OFF_X);  // [2 buffers][2 halves][128 rows]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t crank = cluster_ctarank();
    const bool leader = crank == 0;
    const int cluster = blockIdx.x >> 1, G = gridDim.x >> 1;
    auto bar = [&](uint64_t &b) { return smem_u32(&b); };
    auto lbar = [&](uint64_t &b) { return mapa_shared(smem_u32(&b), 0); };  // leader's copy

    if (threadIdx.x == 0) {
        for (int s = 0; s < KST; ++s) {
            mbar_init(bar(ctrl->k_full[s]), 1);
            mbar_init(bar(ctrl->k_empty[s]), 1);
        }
        for (int s = 0; s < VST; ++s) {
            mbar_init(bar(ctrl->v_full[s]), 1);
            mbar_init(bar(ctrl->v_empty[s]), 1);
        }
        for (int b = 0; b < NSB; ++b) {
            mbar_init(bar(ctrl->s_full[b]), 1);
            mbar_init(bar(ctrl->p_full[b]), 16);  // 8 softmax warps x 2 CTAs
            mbar_init(bar(ctrl->o_done[b]), 1);   // P V of key tiles j with j % NSB == b
        }
        for (int b = 0; b < 3; ++b)
            mbar_init(bar(ctrl->xch[b]), 8);      // this CTA's softmax warps
        mbar_init(bar(ctrl->o_free), 16);  // epilogues of both CTAs read O
        mbar_init(bar(ctrl->q_full), 1);
        mbar_init(bar(ctrl->q_empty), 1);
        mbar_init(bar(ctrl->final_bar), 1);
        ctrl->abort = 0;
        fence_mbar_init();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(&ctrl->tmem_base), P_TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers and TMEM exist before any remote use
    tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    volatile int *abort = &ctrl->abort;
    const uint64_t tmo = p.timeout_ns;
    const int group = p.H / p.Hkv;

    if (warp == 0) {
        // ------------------------------------------------------------ producer (both CTAs)
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_last();
            const uint64_t pol_q = l2_policy_evict_first();
            uint32_t kcnt = 0, vcnt = 0, qcnt = 0;
            bool ok = true;
            for (int r = 0; ok; ++r) {
                const int u = pair_unit_index(r, cluster, G);
                if (u >= p.n_units)
                    break;
                const RaUnit U = ra_unit_decode(p.sp, u);
                // this CTA's query tile, once the previous unit's S MMAs are done
                if (qcnt > 0 && !(ok = pwait(p.status, bar(ctrl->q_empty), (qcnt - 1) & 1, abort, tmo, PS_Q_EMPTY)))
                    break;
                if (leader)
                    mbar_arrive_expect_tx(bar(ctrl->q_full), 2 * Q_TILE);
                {
                    const int qbh = crank ? U.bh1 : U.bh0, qta = crank ? U.ta1 : U.ta0;
                    const int qrow = qbh * p.S + U.rank * p.L + qta * RA_TILE;
                    tma_load_2d_pair(sb + OFF_Q, &p.tm_q, 0, qrow, lbar(ctrl->q_full), pol_q);
                    tma_load_2d_pair(sb + OFF_Q + Q_TILE / 2, &p.tm_q, 64, qrow, lbar(ctrl->q_full), pol_q);
                }
                ++qcnt;
                const int b = U.bh0 / p.H;
                const int kvbh = b * p.Hkv + (U.bh0 - b * p.H) / group;
                Walk w;
                w.start(U.rank, max(U.ta0, U.ta1), p);
                for (; w.valid(); w.advance()) {
                    const int row = kvbh * p.S + w.j * p.L + w.tb * RA_TILE;
                    const int ks = kcnt % KST;
                    if (!(ok = pwait(p.status, bar(ctrl->k_empty[ks]), ((kcnt / KST) & 1) ^ 1, abort, tmo, PS_K_EMPTY)))
                        break;
                    if (leader)
                        mbar_arrive_expect_tx(bar(ctrl->k_full[ks]), 2 * K_HALF);
                    // keys [64 crank, 64 crank + 64) of the tile, all 128 d (two 64-column slabs)
                    const uint32_t dk = sb + OFF_K + ks * K_HALF;
                    tma_load_2d_pair(dk, &p.tm_k, 0, row + 64 * (int)crank, lbar(ctrl->k_full[ks]), pol);
                    tma_load_2d_pair(dk + K_HALF / 2, &p.tm_k, 64, row + 64 * (int)crank,
                                     lbar(ctrl->k_full[ks]), pol);
                    ++kcnt;
                    const int vs = vcnt % VST;
                    if (!(ok = pwait(p.status, bar(ctrl->v_empty[vs]), ((vcnt / VST) & 1) ^ 1, abort, tmo, PS_V_EMPTY)))
                        break;
                    if (leader)
                        mbar_arrive_expect_tx(bar(ctrl->v_full[vs]), 2 * V_HALF);
                    // all 128 keys of the tile, d columns [64 crank, 64 crank + 64)
                    tma_load_2d_pair(sb + OFF_V + vs * V_HALF, &p.tm_v, 64 * (int)crank, row,
                                     lbar(ctrl->v_full[vs]), pol);
                    ++vcnt;
                }
            }
            if (!ok && leader) {
                // both CTAs' copies count on the leader's barriers: let them land
                for (int s = 0; s < KST; ++s) {
                    const uint32_t n = kcnt > (uint32_t)s ? (kcnt - s + KST - 1) / KST : 0;
                    if (n)
                        pdrain(p.status, bar(ctrl->k_full[s]), (n - 1) & 1, tmo);
                }
                for (int s = 0; s < VST; ++s) {
                    const uint32_t n = vcnt > (uint32_t)s ? (vcnt - s + VST - 1) / VST : 0;
                    if (n)
                        pdrain(p.status, bar(ctrl->v_full[s]), (n - 1) & 1, tmo);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader)
        if (lane == 0 && leader) {
            constexpr uint32_t IDESC_S = idesc_bf16_f32(256, 128, 0);
            constexpr uint32_t IDESC_PV = idesc_bf16_f32(256, P_D, 1);
            auto issue_s = [&](int buf, int ks) {
                const uint32_t kb = sb + OFF_K + ks * K_HALF;
                const uint32_t qb = sb + OFF_Q;
#pragma unroll
                for (int kk = 0; kk < P_D / 16; ++kk)
                    mma_ss_pair(tmem + buf * 128,
                                smem_desc_sw128(qb + (kk >> 2) * (Q_TILE / 2) + (kk & 3) * 32, 16, 1024),
                                smem_desc_sw128(kb + (kk >> 2) * (K_HALF / 2) + (kk & 3) * 32, 16, 1024),
                                IDESC_S, kk > 0);
            };
            auto issue_pv = [&](int buf, int vs, bool acc) {
                const uint32_t vb = sb + OFF_V + vs * V_HALF;
#pragma unroll
                for (int kk = 0; kk < RA_TILE / 16; ++kk)
                    mma_ts_pair(tmem + COL_O, tmem + buf * 128 + kk * 8,
                                smem_desc_sw128(vb + kk * 2048, V_HALF, 1024), IDESC_PV,
                                (acc || kk > 0) ? 1u : 0u);
            };
            uint32_t kcnt = 0, vcnt = 0, qcnt = 0, pcnt[NSB] = {0, 0, 0};
            bool ok = true;
            for (int r = 0; ok; ++r) {
                const int u = pair_unit_index(r, cluster, G);
                if (u >= p.n_units)
                    break;
                const int n = ra_unit_decode(p.sp, u).cost;
                // both CTAs' query tiles are in shared memory
                if (!(ok = pwait(p.status, bar(ctrl->q_full), qcnt & 1, abort, tmo, PS_Q_FULL)))
                    break;
                tc_fence_after();
                const int pre = n < NSB ? n : NSB;
                for (int jj = 0; jj < pre && ok; ++jj) {
                    const int ks = kcnt % KST;
                    if (!(ok = pwait(p.status, bar(ctrl->k_full[ks]), (kcnt / KST) & 1, abort, tmo, PS_K_FULL)))
                        break;
                    tc_fence_after();
                    issue_s(jj, ks);
                    mma_commit_pair(bar(ctrl->s_full[jj]));
                    mma_commit_pair(bar(ctrl->k_empty[ks]));
                    ++kcnt;
                }
                if (n <= NSB)
                    mma_commit_pair(bar(ctrl->q_empty));  // last S of the unit issued
                // the previous unit's O has been read by both epilogues
                if (ok && qcnt > 0 && !(ok = pwait(p.status, bar(ctrl->o_free), (qcnt - 1) & 1, abort, tmo, PS_O_FREE)))
                    break;
                ++qcnt;
                for (int j = 0; j < n && ok; ++j) {
                    const int buf = j % NSB;
                    const int vs = vcnt % VST;
                    if (!(ok = pwait(p.status, bar(ctrl->v_full[vs]), (vcnt / VST) & 1, abort, tmo, PS_V_FULL)))
                        break;
                    if (!(ok = pwait(p.status, bar(ctrl->p_full[buf]), pcnt[buf] & 1, abort, tmo, PS_P_FULL)))
                        break;
                    ++pcnt[buf];
                    tc_fence_after();
                    issue_pv(buf, vs, j > 0);
                    mma_commit_pair(bar(ctrl->o_done[buf]));
                    mma_commit_pair(bar(ctrl->v_empty[vs]));
                    ++vcnt;
                    if (j + NSB < n) {
                        // S(j + NSB) reuses this buffer; the tensor pipe runs in
                        // issue order, so P(j) is read before it is overwritten
                        const int ks = kcnt % KST;
                        if (!(ok = pwait(p.status, bar(ctrl->k_full[ks]), (kcnt / KST) & 1, abort, tmo, PS_K_FULL)))
                            break;
                        tc_fence_after();
                        issue_s(buf, ks);
                        mma_commit_pair(bar(ctrl->s_full[buf]));
                        mma_commit_pair(bar(ctrl->k_empty[ks]));
                        ++kcnt;
                        if (j + NSB + 1 == n)
                            mma_commit_pair(bar(ctrl->q_empty));  // last S of the unit issued
                    }
                }
            }
            mma_commit_pair(bar(ctrl->final_bar));
            pdrain(p.status, bar(ctrl->final_bar), 0, tmo);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax (both CTAs)
        const int qw = warp & 3;                  // TMEM lane quarter
        const int h = (warp - 4) >> 2;            // column half of the row
        const int row = qw * 32 + lane;           // query row within the tile
        const uint32_t tbase = tmem + ((uint32_t)(qw * 32) << 16);
        const float sl2 = p.scale_log2;
        // s_full[b] completes once per S into buffer b; o_done[b] once per P V
        // of a key tile j with j % NSB == b; xch[0..1] alternate over all
        // steps, xch[2] serves the epilogue
        uint32_t scnt[NSB] = {0, 0, 0}, pvdone[NSB] = {0, 0, 0}, gstep = 0, ecnt = 0;
        bool ok = true;
        // Exchange one float per half row with the partner thread (the other
        // column half of the same row, in warp w +- 4); returns the partner's.
        auto exchange = [&](int slot, uint32_t parity, float mine, float &theirs) -> bool {
            float *xb = xch + slot * 256;
            xb[h * 128 + row] = mine;
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(ctrl->xch[slot]));
            if (!pwait_warp(p.status, bar(ctrl->xch[slot]), parity, abort, tmo, PS_XCH))
                return false;
            theirs = xb[(1 - h) * 128 + row];
            return true;
        };
        int u = pair_unit_index(0, cluster, G);
        for (int rr = 0; ok && u < p.n_units; ++rr, u = pair_unit_index(rr, cluster, G)) {
            const RaUnit U = ra_unit_decode(p.sp, u);
            const int bh = crank ? U.bh1 : U.bh0;
            const int ta = crank ? U.ta1 : U.ta0;
            const bool store = (crank == 0) || U.tile1_valid;
            const int a = ta * RA_TILE + row;
            float m_run = -INFINITY, l_run = 0.f;
            Walk w;
            w.start(U.rank, max(U.ta0, U.ta1), p);
            int jj = 0;
            for (; w.valid(); w.advance(), ++jj, ++gstep) {
                const int buf = jj % NSB;
                if (!(ok = pwait_warp(p.status, bar(ctrl->s_full[buf]), scnt[buf] & 1, abort, tmo, PS_S_FULL)))
                    break;
                ++scnt[buf];
                tc_fence_after();
                uint32_t x[64];
                const uint32_t tS = tbase + buf * 128;
                float mine;
                tmem_ld64_max(tS + h * 64, x, mine);  // the load also reduces the half row to its max
                tmem_wait_ld();
                asm volatile("" : "+f"(mine));  // keep every use of the max after the wait
                const int lim = ra_key_limit(w.cls, a, p.L) - w.tb * RA_TILE - h * 64;
                if (!__all_sync(0xffffffffu, lim >= 64)) {
                    // masked tile: the max must skip the hidden columns
                    const uint32_t ninf = __float_as_uint(-INFINITY);
#pragma unroll
                    for (int e = 0; e < 64; ++e)
                        x[e] = e < lim ? x[e] : ninf;
                    float ma = -INFINITY, mb = -INFINITY;
#pragma unroll
                    for (int e = 0; e < 64; e += 4) {
                        ma = max3f(ma, __uint_as_float(x[e]), __uint_as_float(x[e + 1]));
                        mb = max3f(mb, __uint_as_float(x[e + 2]), __uint_as_float(x[e + 3]));
                    }
                    mine = fmaxf(ma, mb);
                }
                float theirs;
                if (!(ok = exchange(gstep & 1, (gstep >> 1) & 1, mine, theirs)))
                    break;
                const float m_tile = fmaxf(mine, theirs) * sl2;
                const bool resc = m_tile > m_run + P_LAZY_LOG2;
                float alpha = 1.f;
                if (resc) {
                    alpha = ex2_approx(m_run - m_tile);
                    m_run = m_tile;
                    l_run *= alpha;
                }
                __syncwarp();
                if (jj > 0 && __any_sync(0xffffffffu, resc)) {
                    // O must hold P V of the previous key tile before it is
                    // rescaled.  S(jj) completing implies P V(jj - NSB) did, so
                    // o_done[(jj - 1) % NSB] is either one completion short or
                    // done: a parity wait is unambiguous.
                    const int pb = (jj - 1) % NSB;
                    const uint32_t idx = pvdone[pb] + (uint32_t)((jj - 1) / NSB);
                    if (!(ok = pwait_warp(p.status, bar(ctrl->o_done[pb]), idx & 1, abort, tmo, PS_O_DONE)))
                        break;
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < 2; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tbase + COL_O + h * 64 + c * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(tbase + COL_O + h * 64 + c * 32, o);
                    }
                }
                const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
                const float2 scale = make_float2(sl2, sl2), shift = make_float2(neg_m, neg_m);
                float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
                uint32_t pk[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float2 t2 = ffma2(make_float2(__uint_as_float(x[2 * e]), __uint_as_float(x[2 * e + 1])),
                                            scale, shift);
                    const float2 pv = make_float2(ex2_approx(t2.x), ex2_approx(t2.y));
                    if (e & 1)
                        acc1 = fadd2(acc1, pv);
                    else
                        acc0 = fadd2(acc0, pv);
                    pk[e] = pack_bf16x2(pv.x, pv.y);
                }
                // P for keys [64h, 64h + 64) -> columns [32h, 32h + 32) of the
                // buffer; the partner read its scores before the exchange
                tmem_st32(tS + h * 32, pk);
                const float2 acc = fadd2(acc0, acc1);
                l_run += acc.x + acc.y;
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_cluster(lbar(ctrl->p_full[buf]));
            }
            if (!ok)
                break;
            // ------------------------------------------------ epilogue
            const int n = jj;
            {
                const int pb = (n - 1) % NSB;
                const uint32_t idx = pvdone[pb] + (uint32_t)((n - 1) / NSB);
                if (!(ok = pwait_warp(p.status, bar(ctrl->o_done[pb]), idx & 1, abort, tmo, PS_O_DONE)))
                    break;
            }
            for (int b2 = 0; b2 < NSB; ++b2)
                pvdone[b2] += (uint32_t)((n - b2 + NSB - 1) / NSB);  // j < n with j % NSB == b2
            tc_fence_after();
            float l_other;
            if (!(ok = exchange(2, ecnt & 1, l_run, l_other)))
                break;
            ++ecnt;
            const float l_row = l_run + l_other;
            const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
            const bool valid = store && a < p.L;
            const long long orow = (long long)bh * p.S + (long long)U.rank * p.L + a;
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
                uint32_t o[32];
                __syncwarp();
                tmem_ld32(tbase + COL_O + h * 64 + c * 32, o);
                tmem_wait_ld();
                if (!valid)
                    continue;
                const int col = h * 64 + c * 32;
                if (p.out_f32) {
                    float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + orow * P_D + col);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        dst[e] = make_float4(__uint_as_float(o[4 * e]) * inv, __uint_as_float(o[4 * e + 1]) * inv,
                                             __uint_as_float(o[4 * e + 2]) * inv, __uint_as_float(o[4 * e + 3]) * inv);
                } else {
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.out) + orow * P_D + col);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        uint4 v;
                        v.x = pack_bf16x2(__uint_as_float(o[8 * e + 0]) * inv, __uint_as_float(o[8 * e + 1]) * inv);
                        v.y = pack_bf16x2(__uint_as_float(o[8 * e + 2]) * inv, __uint_as_float(o[8 * e + 3]) * inv);
                        v.z = pack_bf16x2(__uint_as_float(o[8 * e + 4]) * inv, __uint_as_float(o[8 * e + 5]) * inv);
                        v.w = pack_bf16x2(__uint_as_float(o[8 * e + 6]) * inv, __uint_as_float(o[8 * e + 7]) * inv);
                        dst[e] = v;
                    }
                }
            }
            if (valid && h == 0)
                p.lse[orow] = l_row > 0.f ? (m_run + log2f(l_row)) * P_LN2 : -INFINITY;
            // O has been read: the next unit's first P V may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive_cluster(lbar(ctrl->o_free));
        }
    }
    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem, P_TMEM_COLS);
    }
}

}  // namespace
}  // namespace ra

namespace ra {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 pair_encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

bool encode_box(CUtensorMap *tm, const void *base, long long rows, int box_rows)
{
    auto enc = pair_encode_fn();
    if (!enc)
        return false;
    cuuint64_t dims[2] = {(cuuint64_t)P_D, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)P_D * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_attn_pair(const TcLaunch &a, cudaStream_t st)
{
    if (a.d != P_D)
        return cudaErrorInvalidValue;
    static std::atomic<int> attr_set[RA_MAX_DEVICES];
    cudaError_t e0 = once_per_device(attr_set, [] {
        return cudaFuncSetAttribute(ra_attn_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM);
    });
    if (e0 != cudaSuccess)
        return e0;
    PairParams p;
    memset(&p, 0, sizeof(p));
    const long long kv_rows = (long long)a.B * a.Hkv * a.S;
    if (!encode_box(&p.tm_q, a.q, (long long)a.B * a.H * a.S, RA_TILE) ||
        !encode_box(&p.tm_k, a.k, kv_rows, 64) || !encode_box(&p.tm_v, a.v, kv_rows, RA_TILE))
        return cudaErrorInvalidValue;
    p.sp = ra_unit_space_ranks(ra_unit_space(a.B, a.H, a.Hkv, a.S, a.N, a.layout, a.causal, a.s_begin, a.s_end),
                               a.rank_lo, a.rank_hi);
    const long long n_units = ra_unit_count(p.sp);
    if (n_units > 0x7fffffffll)
        return cudaErrorInvalidValue;
    p.out = a.out;
    p.lse = a.lse;
    p.q_rows = (long long)a.B * a.H * a.S;
    p.n_units = (int)n_units;
    p.H = a.H, p.Hkv = a.Hkv, p.S = a.S, p.N = a.N, p.L = a.S / a.N;
    p.layout = a.layout, p.causal = a.causal, p.s_begin = a.s_begin, p.s_end = a.s_end;
    p.out_f32 = a.out_f32;
    p.ntiles = (p.L + RA_TILE - 1) / RA_TILE;
    p.scale_log2 = 1.4426950408889634f / sqrtf((float)P_D);
    p.timeout_ns = a.timeout_ns;
    p.status = device_status_ptr();
    if (!p.status)
        return cudaErrorInvalidValue;
    if (p.n_units <= 0)
        return cudaSuccess;
    const int clusters = p.n_units < a.sm_count / 2 ? p.n_units : a.sm_count / 2;
    if (clusters < 1)
        return cudaErrorInvalidValue;
    ra_attn_pair_kernel<<<2 * clusters, P_THREADS, P_SMEM, st>>>(p);
    return cudaGetLastError();
}

}  // namespace ra
