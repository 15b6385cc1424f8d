// Tensor-core ring-ordered blockwise attention for sm_103a (GB300).
//
// Method ("Ring Attention" glossary page, ultralytics.com/tr, section "Halka
// Dikkati Nasil Calisir"): query block i stays in place while key/value
// blocks arrive in ring order j = (i - s) mod N; each block's scores are
// exponentiated and folded into a running sum of exponentials and a running
// score-weighted value sum that are divided at the end, with a running
// maximum subtracted before exponentiation for stability; causal masking
// skips key blocks that hold no visible key, and the striped layout changes
// only which tiles are masked.  The page notes that ring attention uses a
// flash-attention style blockwise kernel per device; this is that kernel,
// written for Blackwell:
//
//   * one persistent CTA per SM (512 TMEM columns, ~193 KB shared memory);
//     where every kv head serves four or more query heads, the CTAs run as
//     clusters of two whose units walk the same key/value tiles (the two
//     head pairs of a group), and each K and V tile is loaded once for both
//     by TMA multicast (CTA 0 issues K, CTA 1 issues V);
//   * a unit of work is a PAIR of 128-row query tiles that share a kv head
//     (two heads of one grouped-query group, or two adjacent tiles of one
//     head), so every key/value tile staged in shared memory feeds two tiles;
//   * warp 0 issues TMA loads (Q once per unit, K and V per 128-key tile, in
//     128-byte swizzled 64-column slabs), warp 1 issues tcgen05.mma (each
//     a whole warp on warp-uniform values, one elected lane issuing),
//     warps 4-7 and 8-11 run the online softmax for query tile 0 and 1 (at
//     d = 64, warps 4-11 and 12-19, two threads per row, one per 64-key
//     half of each key tile, each half with its own running max, sum and O,
//     merged in the epilogue);
//   * S = Q K^T goes to TMEM (fp32, 128 lanes x 128 columns per tile); each
//     softmax thread reads its row once (two 64-column loads, one wait; the
//     loads of an unmasked tile also reduce the row to its max, a Blackwell
//     Ultra form of tcgen05.ld),
//     writes P = exp2(S log2e/sqrt(d) - m) back over the same columns as
//     packed bf16, and O += P V reads P from TMEM as the A operand and V from
//     shared memory (MN-major);
//   * the running max is rescaled lazily: O and l are only corrected when a
//     row's max grows by more than 2^8, which the final division makes exact;
//   * every mbarrier wait is bounded; a wait that runs out records an error
//     word, raises a CTA-wide abort flag, drains in-flight copies and MMAs,
//     frees TMEM and returns.
//
// TMEM columns: S/P tile 0 [0,128), S/P tile 1 [128,256), O tile 0
// [256,256+d), O tile 1 [384,384+d); at d = 64 the two halves' O of tile t
// are [256+128t, 320+128t) and [320+128t, 384+128t).
#include <atomic>
#include <cstdint>
#include <mutex>
#include <type_traits>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "ra_attn_common.cuh"
#include "ra_internal.h"
#include "ra_ptx_pair.cuh"

namespace ra {

__device__ unsigned int g_ra_status = 0;

namespace {

constexpr uint32_t TMEM_COLS = 512;

enum Site : unsigned int {
    SITE_Q_EMPTY = 1, SITE_K_EMPTY, SITE_V_EMPTY, SITE_Q_FULL, SITE_K_FULL, SITE_V_FULL,
    SITE_P_FULL, SITE_O_FREE, SITE_S_FULL, SITE_O_DONE, SITE_FINAL, SITE_DRAIN, SITE_PROBE
};

template <int D>
struct Cfg {
    // softmax threads per query row: at d = 128 one thread takes the row's 128
    // key columns; at d = 64 (where a tile's MMAs are half as long and cover
    // half as much of the softmax) two threads take 64 columns each, with
    // their own running max, sum and O (TMEM: 2 tiles x (128 S + 2 x 64 O))
    static constexpr int HALVES = D == 64 ? 2 : 1;
    static constexpr int THREADS = 128 + 2 * 128 * HALVES;  // TMA, MMA, 2 spare warps, softmax
    static constexpr int KSTAGES = 2;
    static constexpr int VSTAGES = 2;
    static constexpr int SLAB = 128 * 64 * 2;  // 128 rows x 64 bf16 (128 B swizzled rows)
    static constexpr int NSLAB = D / 64;
    static constexpr int TILE = SLAB * NSLAB;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + 2 * TILE;
    static constexpr int OFF_V = OFF_K + KSTAGES * TILE;
    static constexpr int OFF_CTRL = OFF_V + VSTAGES * TILE;
    static constexpr int OFF_XCH = OFF_CTRL + 256;  // (m, l) of each row's halves: [unit parity][tile][half][row]
    static constexpr int XCH = HALVES == 2 ? 2 * 2 * 2 * 128 * 8 : 0;
    static constexpr int SMEM = OFF_XCH + XCH + 1024;  // + alignment slack
};

struct Ctrl {
    uint64_t q_full, q_empty;
    uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
    uint64_t s_full[2], p_full[2], o_done[2], o_free[2];  // o_done: once per unit, after its last P V
    uint64_t x_full[2];  // both halves of a tile's rows have posted (m, l)
    uint64_t final_bar;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Ctrl) <= 256, "control block");

struct TcParams {
    CUtensorMap tm_q, tm_k, tm_v;
    RaUnitSpace sp;  // the launch's work units, decoded on the fly
    void *out;
    float *lse;
    int n_items, H, Hkv, S, L, N, layout, causal, s_begin, s_end, out_f32, ntiles;
    // Work items: unit u, piece k of its key tiles in ring order.  nsplit = 1:
    // one item per unit (the whole walk).  nsplit > 1: item k of a unit walks
    // tiles [k c / nsplit, (k + 1) c / nsplit) of its c tiles and writes its
    // own fp32 partial at out + k split_out_bytes, lse + k split_lse_stride.
    // pair_items keeps the items of units 2m and 2m + 1 next to each other.
    int nsplit, pair_items;
    long long split_out_bytes, split_lse_stride;
    float scale_log2;
    unsigned long long timeout_ns;
};

// Work item w: its unit's description, piece index k and tile range
// [t0, t0 + cnt).
__device__ __forceinline__ RaUnit item_decode(const TcParams &p, int w, int &k, int &t0, int &cnt)
{
    int u = w;
    k = 0;
    if (p.nsplit > 1) {
        if (p.pair_items) {
            const int m = w / (2 * p.nsplit), rem = w - m * 2 * p.nsplit;
            k = rem >> 1;
            u = 2 * m + (rem & 1);
        } else {
            u = w / p.nsplit;
            k = w - u * p.nsplit;
        }
    }
    const RaUnit U = ra_unit_decode(p.sp, u);
    t0 = (int)((long long)k * U.cost / p.nsplit);
    cnt = (int)((long long)(k + 1) * U.cost / p.nsplit) - t0;
    return U;
}

__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int *abort,
                                          uint64_t timeout, unsigned int site)
{
    const bool ok = mbar_wait(bar, parity, abort, timeout, &g_ra_status, site);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ bool wait1(uint32_t bar, uint32_t parity, volatile int *abort,
                                      uint64_t timeout, unsigned int site)
{
    return mbar_wait(bar, parity, abort, timeout, &g_ra_status, site);
}

// Waits on barriers that the peer CTA of a cluster also feeds (multicast
// copies and MMA-completion arrivals): cluster-scope acquire.
__device__ __forceinline__ bool wait1c(uint32_t bar, uint32_t parity, volatile int *abort,
                                       uint64_t timeout, unsigned int site)
{
    return mbar_wait_cluster(bar, parity, abort, timeout, &g_ra_status, site);
}

// Wait that ignores the abort flag: used to drain work already in flight.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, uint64_t timeout)
{
    int never = 0;
    mbar_wait(bar, parity, &never, timeout, &g_ra_status, SITE_DRAIN);
}

template <int D>
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap *tm, int row, uint32_t bar,
                                          uint64_t pol)
{
#pragma unroll
    for (int h = 0; h < D / 64; ++h)
        tma_load_2d(dst + h * Cfg<D>::SLAB, tm, h * 64, row, bar, pol);
}

// The same tile into both CTAs of a cluster (same offsets, same barrier).
template <int D>
__device__ __forceinline__ void load_tile_both(uint32_t dst, const CUtensorMap *tm, int row, uint32_t bar,
                                               uint64_t pol)
{
#pragma unroll
    for (int h = 0; h < D / 64; ++h)
        tma_load_2d_mc(dst + h * Cfg<D>::SLAB, tm, h * 64, row, bar, (uint16_t)3, pol);
}

// CL = 1: one CTA per SM.  CL = 2: clusters of two CTAs whose units have the
// same kv head, rank and query tile slot (the two head pairs of a group of
// four or more query heads), so both walk the same key/value tiles: CTA 0
// loads each K tile and CTA 1 each V tile into BOTH CTAs' shared memory by
// TMA multicast, and a stage is reloaded only after both CTAs' MMAs have
// consumed it (each MMA warp commits to the empty barrier of both CTAs).
template <int D, int CL, bool SPLIT>
__global__ void __launch_bounds__(Cfg<D>::THREADS, 1) ra_attn_tc_kernel(const __grid_constant__ TcParams p)
{
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);
    Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem + C::OFF_CTRL);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    auto bar = [&](uint64_t &b) { return smem_u32(&b); };
    const uint32_t sQ = sb + C::OFF_Q, sK = sb + C::OFF_K, sV = sb + C::OFF_V;

    if (threadIdx.x == 0) {
        mbar_init(bar(ctrl->q_full), 1);
        mbar_init(bar(ctrl->q_empty), 1);
        for (int s = 0; s < C::KSTAGES; ++s) {
            mbar_init(bar(ctrl->k_full[s]), 1);
            mbar_init(bar(ctrl->k_empty[s]), CL);
        }
        for (int s = 0; s < C::VSTAGES; ++s) {
            mbar_init(bar(ctrl->v_full[s]), 1);
            mbar_init(bar(ctrl->v_empty[s]), CL);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(ctrl->s_full[t]), 1);
            mbar_init(bar(ctrl->p_full[t]), 128 * C::HALVES);
            mbar_init(bar(ctrl->o_done[t]), 1);
            mbar_init(bar(ctrl->o_free[t]), 128 * C::HALVES);
            if (C::HALVES == 2)
                mbar_init(bar(ctrl->x_full[t]), 128 * C::HALVES);
        }
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
        tmem_alloc(smem_u32(&ctrl->tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    if (CL == 2)
        cluster_sync_all();  // the peer's barriers exist before any multicast reaches them
    tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    volatile int *abort = &ctrl->abort;
    const uint64_t tmo = p.timeout_ns;
    const int group = p.H / p.Hkv;
    const int crank = CL == 2 ? (int)cluster_ctarank() : 0;
    // unit of round r: clusters are dealt unit pairs (2m, 2m + 1) in snake order
    auto unit_of = [&](int r) { return CL * unit_index(r, blockIdx.x / CL, gridDim.x / CL) + crank; };
    auto kv_wait = [&](uint32_t b, uint32_t parity, unsigned int site) {
        return CL == 2 ? wait1c(b, parity, abort, tmo, site) : wait1(b, parity, abort, tmo, site);
    };
    auto kv_release = [&](uint32_t b) {
        if (CL == 2)
            mma_commit_mc(b, (uint16_t)3);
        else
            mma_commit(b);
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // The whole warp runs the loop on warp-uniform values, its waits
        // included (a wait costs less in converged code, and each one sits on
        // the path from a freed stage to its next copy); one lane, elected
        // once, arms the barriers and issues the copies.
        const bool leader = elect_one();
        const uint64_t pol_q = l2_policy_evict_first();
        const uint64_t pol_kv = l2_policy_evict_last();
        auto pwait = [&](uint32_t b, uint32_t parity, unsigned int site) -> bool {
            return __all_sync(0xffffffffu, kv_wait(b, parity, site)) != 0;
        };
        uint32_t kcnt = 0, vcnt = 0, qcnt = 0;
        bool ok = true;
        for (int r = 0; ok; ++r) {
            const int wi = unit_of(r);
            if (wi >= p.n_items)
                break;
            int k = 0, t0 = 0, cnt = 0;
            const RaUnit U = SPLIT ? item_decode(p, wi, k, t0, cnt) : ra_unit_decode(p.sp, wi);
            if (SPLIT && cnt == 0)
                continue;  // an empty piece: nothing to load
            if (qcnt > 0 && !(ok = wait_warp(bar(ctrl->q_empty), (qcnt - 1) & 1, abort, tmo, SITE_Q_EMPTY)))
                break;
            if (leader) {
                mbar_arrive_expect_tx(bar(ctrl->q_full), 2 * C::TILE);
                const int qrow0 = U.bh0 * p.S + U.rank * p.L + U.ta0 * RA_TILE;
                const int qrow1 = U.bh1 * p.S + U.rank * p.L + U.ta1 * RA_TILE;
                load_tile<D>(sQ, &p.tm_q, qrow0, bar(ctrl->q_full), pol_q);
                load_tile<D>(sQ + C::TILE, &p.tm_q, qrow1, bar(ctrl->q_full), pol_q);
            }
            __syncwarp();
            ++qcnt;
            const int b = U.bh0 / p.H;
            const int kvbh = b * p.Hkv + (U.bh0 - b * p.H) / group;
            KvWalk w;
            w.start(U.rank, max(U.ta0, U.ta1), p);
            if (SPLIT)
                w.skip(t0);
            for (int c = 0; SPLIT ? c < cnt : w.valid(); ++c, w.advance()) {
                const int row = kvbh * p.S + w.j * p.L + w.tb * RA_TILE;
                const int ks = kcnt % C::KSTAGES;
                if (!(ok = pwait(bar(ctrl->k_empty[ks]), ((kcnt / C::KSTAGES) & 1) ^ 1, SITE_K_EMPTY)))
                    break;
                if (leader) {
                    mbar_arrive_expect_tx(bar(ctrl->k_full[ks]), C::TILE);
                    if (CL == 1)
                        load_tile<D>(sK + ks * C::TILE, &p.tm_k, row, bar(ctrl->k_full[ks]), pol_kv);
                    else if (crank == 0)
                        load_tile_both<D>(sK + ks * C::TILE, &p.tm_k, row, bar(ctrl->k_full[ks]), pol_kv);
                }
                __syncwarp();
                ++kcnt;
                const int vs = vcnt % C::VSTAGES;
                if (!(ok = pwait(bar(ctrl->v_empty[vs]), ((vcnt / C::VSTAGES) & 1) ^ 1, SITE_V_EMPTY)))
                    break;
                if (leader) {
                    mbar_arrive_expect_tx(bar(ctrl->v_full[vs]), C::TILE);
                    if (CL == 1)
                        load_tile<D>(sV + vs * C::TILE, &p.tm_v, row, bar(ctrl->v_full[vs]), pol_kv);
                    else if (crank == 1)
                        load_tile_both<D>(sV + vs * C::TILE, &p.tm_v, row, bar(ctrl->v_full[vs]), pol_kv);
                }
                __syncwarp();
                ++vcnt;
            }
        }
        if (!ok) {
            // let every issued copy land before shared memory is released
            for (int s = 0; s < C::KSTAGES; ++s) {
                const uint32_t n = kcnt > (uint32_t)s ? (kcnt - s + C::KSTAGES - 1) / C::KSTAGES : 0;
                if (n)
                    wait_drain(bar(ctrl->k_full[s]), (n - 1) & 1, tmo);
            }
            for (int s = 0; s < C::VSTAGES; ++s) {
                const uint32_t n = vcnt > (uint32_t)s ? (vcnt - s + C::VSTAGES - 1) / C::VSTAGES : 0;
                if (n)
                    wait_drain(bar(ctrl->v_full[s]), (n - 1) & 1, tmo);
            }
            if (qcnt)
                wait_drain(bar(ctrl->q_full), (qcnt - 1) & 1, tmo);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop on warp-uniform values, waits included,
        // and one lane, elected once, issues every MMA and commit (a commit
        // tracks the MMAs of the thread that executes it).  A tcgen05.mma issue
        // returns only once the tensor pipe takes it, about one MMA ahead, so
        // whatever the issuing thread does between MMAs leaves the pipe idle; a
        // barrier wait costs far less in converged, uniform code than inside a
        // one-lane branch.
        const bool leader = elect_one();
        const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
        constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 128, 0);
        constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, D, 1);
        auto issue_s = [&](int t, int ks) {
            const uint32_t qa = sQ + t * C::TILE, ka = sK + ks * C::TILE;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * C::SLAB + (kk & 3) * 32;
                mma_ss(tm + t * 128, smem_desc_sw128(qa + off, 16, 1024), smem_desc_sw128(ka + off, 16, 1024),
                       IDESC_S, kk > 0);
            }
        };
        auto issue_pv = [&](int t, int vs, bool acc) {
            const uint32_t va = sV + vs * C::TILE;
#pragma unroll
            for (int kk = 0; kk < RA_TILE / 16; ++kk) {
                if constexpr (C::HALVES == 2) {
                    // keys [0, 64) and [64, 128) go to the two halves' own O,
                    // each reading P from the first 32 columns of its half
                    const int hh = kk >> 2;
                    mma_ts(tm + 256 + t * 128 + hh * D, tm + t * 128 + hh * 64 + (kk & 3) * 8,
                           smem_desc_sw128(va + kk * 2048, C::SLAB, 1024), IDESC_PV, (acc || (kk & 3) > 0) ? 1u : 0u);
                } else {
                    mma_ts(tm + 256 + t * 128, tm + t * 128 + kk * 8, smem_desc_sw128(va + kk * 2048, C::SLAB, 1024),
                           IDESC_PV, (acc || kk > 0) ? 1u : 0u);
                }
            }
        };
        auto wwait = [&](uint32_t b, uint32_t parity, unsigned int site) {
            return wait_warp(b, parity, abort, tmo, site);
        };
        auto kv_wwait = [&](uint32_t b, uint32_t parity, unsigned int site) -> bool {
            if (CL == 2)
                return __all_sync(0xffffffffu, wait1c(b, parity, abort, tmo, site)) != 0;
            return wait_warp(b, parity, abort, tmo, site);
        };
        uint32_t kcnt = 0, vcnt = 0, qcnt = 0, pcnt = 0;
        bool ok = true;
        for (int r = 0; ok; ++r) {
            const int wi = unit_of(r);
            if (wi >= p.n_items)
                break;
            int k = 0, t0 = 0, n = 0;
            if (SPLIT)
                item_decode(p, wi, k, t0, n);
            else
                n = ra_unit_decode(p.sp, wi).cost;
            if (SPLIT && n == 0)
                continue;  // an empty piece: no MMA
            if (!(ok = wwait(bar(ctrl->q_full), qcnt & 1, SITE_Q_FULL)))
                break;
            int ks = kcnt % C::KSTAGES;
            if (!(ok = kv_wwait(bar(ctrl->k_full[ks]), (kcnt / C::KSTAGES) & 1, SITE_K_FULL)))
                break;
            tc_fence_after();
            if (leader) {
                issue_s(0, ks);
                mma_commit(bar(ctrl->s_full[0]));
                issue_s(1, ks);
                mma_commit(bar(ctrl->s_full[1]));
                kv_release(bar(ctrl->k_empty[ks]));
                if (n == 1)
                    mma_commit(bar(ctrl->q_empty));
            }
            __syncwarp();
            ++kcnt;
            // One key tile per step.  Inside a unit's walk K runs one tile ahead
            // of V (kcnt = vcnt + 1), so with two stages each the K stage is
            // the other one: the step is specialised on V's stage and every
            // shared-memory address below is the base plus a constant.
            static_assert(C::KSTAGES == 2 && C::VSTAGES == 2, "stage parity specialisation");
            auto step = [&](auto vs_c, int jj) -> bool {
                constexpr int VS = decltype(vs_c)::value, KS = 1 - VS;
                const bool more = jj + 1 < n;
                if (!kv_wwait(bar(ctrl->v_full[VS]), (vcnt >> 1) & 1, SITE_V_FULL))
                    return false;
                if (jj == 0 && qcnt > 0 && !wwait(bar(ctrl->o_free[0]), (qcnt - 1) & 1, SITE_O_FREE))
                    return false;
                if (!wwait(bar(ctrl->p_full[0]), pcnt & 1, SITE_P_FULL))
                    return false;
                tc_fence_after();
                if (leader) {
                    issue_pv(0, VS, jj > 0);
                    if (!more)
                        mma_commit(bar(ctrl->o_done[0]));  // O of tile 0 complete for the unit
                }
                __syncwarp();
                if (more) {
                    if (!kv_wwait(bar(ctrl->k_full[KS]), (kcnt >> 1) & 1, SITE_K_FULL))
                        return false;
                    tc_fence_after();
                    if (leader) {
                        issue_s(0, KS);
                        mma_commit(bar(ctrl->s_full[0]));
                    }
                    __syncwarp();
                }
                if (jj == 0 && qcnt > 0 && !wwait(bar(ctrl->o_free[1]), (qcnt - 1) & 1, SITE_O_FREE))
                    return false;
                if (!wwait(bar(ctrl->p_full[1]), pcnt & 1, SITE_P_FULL))
                    return false;
                tc_fence_after();
                if (leader) {
                    issue_pv(1, VS, jj > 0);
                    if (!more)
                        mma_commit(bar(ctrl->o_done[1]));  // O of tile 1 complete for the unit
                    kv_release(bar(ctrl->v_empty[VS]));
                    if (more) {
                        issue_s(1, KS);
                        mma_commit(bar(ctrl->s_full[1]));
                        kv_release(bar(ctrl->k_empty[KS]));
                        if (jj + 2 == n)
                            mma_commit(bar(ctrl->q_empty));
                    }
                }
                __syncwarp();
                ++vcnt;
                if (more)
                    ++kcnt;
                ++pcnt;
                return true;
            };
            for (int jj = 0; ok && jj < n; ++jj)
                ok = (vcnt & 1) ? step(std::integral_constant<int, 1>{}, jj) : step(std::integral_constant<int, 0>{}, jj);
            ++qcnt;
        }
        // every MMA issued so far completes before TMEM and shared memory go
        if (leader)
            mma_commit(bar(ctrl->final_bar));
        __syncwarp();
        wait_drain(bar(ctrl->final_bar), 0, tmo);
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax
        // warps 4 + 4 HALVES t + 4 h + qw: tile t, column half h, rows 32 qw..
        const int t = (warp - 4) >> (C::HALVES == 2 ? 3 : 2);
        const int h = C::HALVES == 2 ? ((warp - 4) >> 2) & 1 : 0;
        const int qw = warp & 3;
        const int r = qw * 32 + lane;
        const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
        const uint32_t tS = tmem + lane_off + t * 128;
        const uint32_t tO = tmem + lane_off + 256 + t * 128;
        const float sl2 = p.scale_log2;
        uint32_t scnt = 0, ocnt = 0;
        bool ok = true;
        for (int rr = 0; ok; ++rr) {
            const int wi = unit_of(rr);
            if (wi >= p.n_items)
                break;
            int k = 0, t0 = 0, cnt = 0;
            const RaUnit U = SPLIT ? item_decode(p, wi, k, t0, cnt) : ra_unit_decode(p.sp, wi);
            const int bh = t ? U.bh1 : U.bh0;
            const int ta = t ? U.ta1 : U.ta0;
            const bool store = (t == 0) || U.tile1_valid;
            const int a = ta * RA_TILE + r;
            if (SPLIT && cnt == 0) {
                // an empty piece: its partial holds no key (lse = -inf)
                if (store && a < p.L && h == 0)
                    p.lse[k * p.split_lse_stride + (long long)bh * p.S + (long long)U.rank * p.L + a] = -INFINITY;
                continue;
            }
            float m_run = -INFINITY, l_run = 0.f;
            KvWalk w;
            w.start(U.rank, max(U.ta0, U.ta1), p);
            if (SPLIT)
                w.skip(t0);
            for (int jj = 0; SPLIT ? jj < cnt : w.valid(); w.advance(), ++jj) {
                // S(t, jj) was issued after P V(t, jj - 1), and the commit that
                // signals S tracks every earlier MMA of the issuing thread: once
                // S is here, the previous P V has read P and written O, so P may
                // be overwritten and O rescaled without a wait of its own
                if (!(ok = wait_warp(bar(ctrl->s_full[t]), scnt & 1, abort, tmo, SITE_S_FULL)))
                    break;
                ++scnt;
                tc_fence_after();
                const int lim = ra_key_limit(w.cls, a, p.L) - w.tb * RA_TILE;
                // masked only where some column of the warp's rows lies past
                // its visibility bound (diagonal and ragged tiles)
                if constexpr (C::HALVES == 2) {
                    const int limh = lim - 64 * h;
                    if (!__all_sync(0xffffffffu, limh >= 64))
                        softmax_half<D, true>(tS + 64 * h, tO + D * h, limh, sl2, jj > 0, m_run, l_run);
                    else
                        softmax_half<D, false>(tS + 64 * h, tO + D * h, limh, sl2, jj > 0, m_run, l_run);
                } else {
                    const bool masked = !__all_sync(0xffffffffu, lim >= RA_TILE);
                    if (masked)
                        softmax_step<D, true>(tS, tO, lim, sl2, jj > 0, m_run, l_run);
                    else
                        softmax_step<D, false>(tS, tO, lim, sl2, jj > 0, m_run, l_run);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar(ctrl->p_full[t]));
            }
            if (!ok)
                break;
            // ------------------------------------------------ epilogue
            if (!(ok = wait_warp(bar(ctrl->o_done[t]), ocnt & 1, abort, tmo, SITE_O_DONE)))
                break;
            ++ocnt;
            tc_fence_after();
            const bool valid = store && a < p.L;
            const long long orow = (long long)bh * p.S + (long long)U.rank * p.L + a;
            if constexpr (C::HALVES == 2) {
                // post this half's (m, l), wait (bounded) for the other half's
                const uint32_t par = (ocnt - 1) & 1;
                float2 *xch = reinterpret_cast<float2 *>(smem + C::OFF_XCH) + (par * 2 + t) * 256;
                xch[h * 128 + r] = make_float2(m_run, l_run);
                mbar_arrive(bar(ctrl->x_full[t]));
                if (!(ok = wait_warp(bar(ctrl->x_full[t]), par, abort, tmo, SITE_O_DONE)))
                    break;
                const float2 oth = xch[(h ^ 1) * 128 + r];
                if (SPLIT)
                    merge_halves_store_row<D>(tO, h, valid, orow, m_run, l_run, oth.x, oth.y,
                                              static_cast<char *>(p.out) + k * p.split_out_bytes,
                                              p.lse + k * p.split_lse_stride, 1);
                else
                    merge_halves_store_row<D>(tO, h, valid, orow, m_run, l_run, oth.x, oth.y, p.out, p.lse,
                                              p.out_f32);
            } else {
                if (SPLIT)
                    store_row<D>(tO, valid, orow, m_run, l_run, static_cast<char *>(p.out) + k * p.split_out_bytes,
                                 p.lse + k * p.split_lse_stride, 1);
                else
                    store_row<D>(tO, valid, orow, m_run, l_run, p.out, p.lse, p.out_f32);
            }
            __syncwarp();
            tc_fence_before();
            mbar_arrive(bar(ctrl->o_free[t]));
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (CL == 2)
        cluster_sync_all();  // no CTA leaves while the peer may still signal or fill it
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn()
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

bool encode_rows(CUtensorMap *tm, const void *base, long long rows, int d)
{
    auto enc = get_encode_fn();
    if (!enc)
        return false;
    cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)d * 2};
    cuuint32_t box[2] = {64, RA_TILE};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int D, int CL, bool SPLIT>
cudaError_t set_smem_attr()
{
    static std::atomic<int> done[RA_MAX_DEVICES];
    return once_per_device(done, [] {
        return cudaFuncSetAttribute(ra_attn_tc_kernel<D, CL, SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    Cfg<D>::SMEM);
    });
}

// Clusters of two that can be resident at once on the current device (one
// CTA per SM), queried once per device.
template <int D>
int max_pair_clusters()
{
    static std::atomic<int> known[RA_MAX_DEVICES];  // clusters + 1; 0 = not queried yet
    const int dev = current_device_slot();
    if (dev < 0)
        return 0;
    const int have = known[dev].load(std::memory_order_acquire);
    if (have > 0)
        return have - 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(Cfg<D>::THREADS);
    cfg.dynamicSmemBytes = Cfg<D>::SMEM;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int c = 0;
    if (cudaOccupancyMaxActiveClusters(&c, ra_attn_tc_kernel<D, 2, false>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;  // not cached: asked again on the next launch
    }
    known[dev].store(c + 1, std::memory_order_release);
    return c;
}

// One launch of the kernel: clusters of two (CL = 2) or one CTA per SM.
template <int D, bool SPLIT>
cudaError_t launch_grid(const TcParams &p, bool clusters, int sm_count, cudaStream_t st)
{
    using C = Cfg<D>;
    cudaError_t e;
    if (clusters) {
        if ((e = set_smem_attr<D, 2, SPLIT>()) != cudaSuccess)
            return e;
        const int max_cl = max_pair_clusters<D>();
        if (max_cl >= 1) {
            const int pairs = p.n_items / 2;
            const int n_cl = pairs < max_cl ? pairs : max_cl;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2 * n_cl);
            cfg.blockDim = dim3(C::THREADS);
            cfg.dynamicSmemBytes = C::SMEM;
            cfg.stream = st;
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = 2;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            e = cudaLaunchKernelEx(&cfg, ra_attn_tc_kernel<D, 2, SPLIT>, p);
            return e != cudaSuccess ? e : cudaGetLastError();
        }
    }
    if ((e = set_smem_attr<D, 1, SPLIT>()) != cudaSuccess)
        return e;
    const int grid = p.n_items < sm_count ? p.n_items : sm_count;
    ra_attn_tc_kernel<D, 1, SPLIT><<<grid, C::THREADS, C::SMEM, st>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const TcLaunch &a, cudaStream_t st)
{
    TcParams p;
    memset(&p, 0, sizeof(p));
    if (!encode_rows(&p.tm_q, a.q, (long long)a.B * a.H * a.S, D) ||
        !encode_rows(&p.tm_k, a.k, (long long)a.B * a.Hkv * a.S, D) ||
        !encode_rows(&p.tm_v, a.v, (long long)a.B * a.Hkv * a.S, D))
        return cudaErrorInvalidValue;
    p.sp = ra_unit_space_ranks(ra_unit_space(a.B, a.H, a.Hkv, a.S, a.N, a.layout, a.causal, a.s_begin, a.s_end),
                               a.rank_lo, a.rank_hi);
    const long long n_units = ra_unit_count(p.sp);
    const int nsplit = a.nsplit > 1 ? a.nsplit : 1;
    if (n_units * nsplit > 0x7fffffffll || (nsplit > 1 && !a.out_f32))
        return cudaErrorInvalidValue;
    p.out = a.out;
    p.lse = a.lse;
    p.n_items = (int)(n_units * nsplit);
    p.nsplit = nsplit;
    p.pair_items = n_units % 2 == 0 ? 1 : 0;
    p.split_out_bytes = nsplit > 1 ? a.split_out_bytes : 0;
    p.split_lse_stride = nsplit > 1 ? a.split_lse_stride : 0;
    p.H = a.H, p.Hkv = a.Hkv, p.S = a.S, p.N = a.N, p.L = a.S / a.N;
    p.layout = a.layout, p.causal = a.causal;
    p.s_begin = a.s_begin, p.s_end = a.s_end, p.out_f32 = a.out_f32;
    p.ntiles = (p.L + RA_TILE - 1) / RA_TILE;
    p.scale_log2 = 1.4426950408889634f / sqrtf((float)D);
    p.timeout_ns = a.timeout_ns;
    if (p.n_items <= 0)
        return cudaSuccess;
    // Clusters need units (2m, 2m + 1) with one key/value walk: two head
    // pairs of one kv head next to each other in the order, i.e. an even
    // number of head pairs per kv head (the pieces of a split walk keep the
    // two units' pieces k next to each other).
    const int pairs_per_kv = p.sp.head_pairs ? (a.H / a.Hkv) / 2 : 0;
    const bool clusters = a.cluster == 2 && pairs_per_kv >= 2 && pairs_per_kv % 2 == 0 && n_units % 2 == 0;
    return nsplit > 1 ? launch_grid<D, true>(p, clusters, a.sm_count, st)
                      : launch_grid<D, false>(p, clusters, a.sm_count, st);
}

}  // namespace

cudaError_t launch_attn_tc(const TcLaunch &a, cudaStream_t st)
{
    if (a.d == 128)
        return launch_d<128>(a, st);
    if (a.d == 64)
        return launch_d<64>(a, st);
    return cudaErrorInvalidValue;
}

// The failure path under test: the same bounded wait, on an mbarrier that no
// thread or copy ever arrives at.
__global__ void ra_wait_probe_kernel(unsigned long long timeout_ns)
{
    __shared__ uint64_t bar;
    __shared__ int abort;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    abort = 0;
    fence_mbar_init();
    mbar_wait(b, 0, &abort, timeout_ns, &g_ra_status, SITE_PROBE);
}

cudaError_t launch_wait_probe(unsigned long long timeout_ns, cudaStream_t st)
{
    ra_wait_probe_kernel<<<1, 1, 0, st>>>(timeout_ns);
    return cudaGetLastError();
}

unsigned int *device_status_ptr()
{
    constexpr int kMax = 64;
    static std::mutex mu;
    static unsigned int *ptr[kMax] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMax)
        return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptr[dev]) {
        void *a = nullptr;
        if (cudaGetSymbolAddress(&a, g_ra_status) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        ptr[dev] = static_cast<unsigned int *>(a);
    }
    return ptr[dev];
}

cudaError_t read_and_clear_device_status(unsigned int *status)
{
    cudaError_t e = cudaMemcpyFromSymbol(status, g_ra_status, sizeof(unsigned int));
    if (e != cudaSuccess)
        return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_ra_status, &zero, sizeof(unsigned int));
}

}  // namespace ra
