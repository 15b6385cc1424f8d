// Backward pass of ring-ordered blockwise exact attention, sm_103a (GB300).
//
// The pages train through ring attention ("Context Parallelism" glossary
// page, ultralytics.com/tr, section "Pratik Kullanim ve Odunlesimler": the
// example calls backward on the attention output), and the ring computes
// exact attention ("Ring Attention" page, section "Halka Dikkati Nasil
// Calisir"), so the gradients are those of exact attention.  With the scale
// c = 1/sqrt(d), the forward's log-sum-exp lse and delta = rowsum(dO * O):
//
//   P = exp(c Q K^T - lse)      dP = dO V^T      dS = P * (dP - delta)
//   dV = P^T dO                 dK = c dS^T Q    dQ = c dS K
//
// computed blockwise in the ring's order.  On a ring, key/value block j and
// its gradient accumulators travel: at step s they sit on device i = (j + s)
// mod N, which adds the contribution of its query block i.  ra_bwd_dkdv_kernel
// follows that order for one 128-key tile of block j (all query heads of the
// kv group, query tiles that see the tile); ra_bwd_dq_kernel gives one
// 128-row query tile its dQ over the key blocks j = (i - s) mod N, as the
// forward walks them.  Both recompute P from lse instead of storing it.
//
// Per tile pair, on the tensor cores (tcgen05, fp32 accumulators in TMEM):
//   dK/dV kernel: S^T = K Q^T and dP^T = V dO^T (SMEM x SMEM, keys on TMEM
//     lanes); the elementwise warps turn them into P^T and dS^T (packed bf16,
//     written back over the consumed columns); dV += P^T dO and
//     dK += dS^T Q read them from TMEM as the A operand.
//   dQ kernel: S = Q K^T and dP = dO V^T (queries on lanes); dS in TMEM;
//     dQ += dS K.
// Roles: warp 0 issues TMA loads (and stages lse / delta rows), warp 1 issues
// MMAs and owns TMEM, warps 2-9 (two per TMEM lane quarter, each on half of
// the columns) do the elementwise work and the epilogue.  Every wait is bounded, as in the
// forward kernel.
//
// TMEM columns: S [0,128), dP [128,256), then the accumulators: dV and dK
// (dK/dV kernel) or dQ (dQ kernel) from column 256.
#include <cstdint>
#include <cstring>
#include <type_traits>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "ra_bwd_schedule.h"
#include "ra_internal.h"
#include "ra_ptx.cuh"

namespace ra {

namespace {

constexpr int BWD_THREADS = 320;  // warp 0 TMA, warp 1 MMA, warps 2-9 elementwise (2 per lane quarter)
constexpr int BWD_EW = 256;       // elementwise threads
constexpr uint32_t BWD_TMEM_COLS = 512;
constexpr float LOG2E = 1.4426950408889634f;

enum BwdSite : unsigned int {
    BS_KV_FULL = 32, BS_ST_FULL, BS_ST_EMPTY, BS_S_FULL, BS_P_FULL, BS_FINAL, BS_Q_FULL, BS_KV_EMPTY,
    BS_DRAIN
};

template <int D>
struct BwdCfg {
    static constexpr int SLAB = 128 * 64 * 2;
    static constexpr int TILE = SLAB * (D / 64);
    // dK/dV kernel: K, V once; Q and dO in two stages; lse/delta rows per stage
    static constexpr int KV_OFF_K = 0;
    static constexpr int KV_OFF_V = TILE;
    static constexpr int KV_OFF_Q = 2 * TILE;
    static constexpr int KV_OFF_DO = 4 * TILE;
    static constexpr int KV_OFF_ROWS = 6 * TILE;           // [stage][nl | dl][128] floats
    static constexpr int KV_OFF_CTRL = KV_OFF_ROWS + 2 * 2 * 128 * 4;
    static constexpr int KV_SMEM = KV_OFF_CTRL + 256 + 1024;
    // dQ kernel: Q, dO once; K in three stages (held until dQ), V in two
    // (free once dP has read it)
    static constexpr int Q_KST = 3;
    static constexpr int Q_OFF_Q = 0;
    static constexpr int Q_OFF_DO = TILE;
    static constexpr int Q_OFF_K = 2 * TILE;
    static constexpr int Q_OFF_V = (2 + Q_KST) * TILE;
    static constexpr int Q_OFF_CTRL = (4 + Q_KST) * TILE;
    static constexpr int Q_SMEM = Q_OFF_CTRL + 256 + 1024;
    // Both kernels allocate all 512 TMEM columns: ask for enough shared
    // memory that a second CTA never lands on the same SM (it would block in
    // tcgen05.alloc until the first one exits).
    static constexpr int ONE_PER_SM = 120 * 1024;
    static constexpr int KV_LAUNCH_SMEM = KV_SMEM > ONE_PER_SM ? KV_SMEM : ONE_PER_SM;
    static constexpr int Q_LAUNCH_SMEM = Q_SMEM > ONE_PER_SM ? Q_SMEM : ONE_PER_SM;
};

struct BwdCtrl {
    uint64_t once_full;            // K, V (dK/dV) or Q, dO (dQ)
    uint64_t st_full[2], st_empty[2];  // dK/dV: Q, dO stages; dQ: V stages
    uint64_t kf[3], ke[3];         // dQ: K stages
    uint64_t s_full[2];            // S (per S buffer)
    uint64_t dp_full;              // dP
    uint64_t p_full;               // dK/dV: P^T written; dQ: dS written (256 arrivals)
    uint64_t ds_full;              // dK/dV: dS^T written (256 arrivals)
    uint64_t final_bar;
    uint32_t tmem_base;
    int abort;
};

static_assert(sizeof(BwdCtrl) <= 256, "control block");

struct BwdParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_do;
    const float *lse;    // [B H S] natural log, rank-major rows
    const float *delta;  // [B H S]
    __nv_bfloat16 *dq, *dk, *dv;
    int B, H, Hkv, S, L, N, layout, causal, ntiles, n_units;
    float scale, scale_log2;
    unsigned long long timeout_ns;
    unsigned int *status;  // the library's device status word
};

// Waits record a timeout in the library's status word (`st`, passed in by
// the launch).
__device__ __forceinline__ bool bwait_warp(unsigned int *st, uint32_t bar, uint32_t parity, volatile int *abort,
                                           uint64_t tmo, unsigned int site)
{
    const bool ok = mbar_wait(bar, parity, abort, tmo, st, site);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void bdrain(unsigned int *st, uint32_t bar, uint32_t parity, uint64_t tmo)
{
    int never = 0;
    mbar_wait(bar, parity, &never, tmo, st, BS_DRAIN);
}

// Bring one [128 rows][D] tile into L2 ahead of its TMA load (no shared
// memory, no barrier).
template <int D>
__device__ __forceinline__ void bprefetch_tile(const CUtensorMap *tm, int row)
{
#pragma unroll
    for (int h = 0; h < D / 64; ++h)
        asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
                     ::"l"(tm), "r"(h * 64), "r"(row) : "memory");
}

template <int D>
__device__ __forceinline__ void bload_tile(uint32_t dst, const CUtensorMap *tm, int row, uint32_t bar,
                                           uint64_t pol)
{
#pragma unroll
    for (int h = 0; h < D / 64; ++h)
        tma_load_2d(dst + h * BwdCfg<D>::SLAB, tm, h * 64, row, bar, pol);
}

// D (+)= A B^T over the head dimension: A, B are [128 rows][D] K-major tiles.
template <int D>
__device__ __forceinline__ void issue_rows_dot(uint32_t d_tmem, uint32_t a, uint32_t b)
{
    constexpr uint32_t ID = idesc_bf16_f32(128, 128, 0);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * BwdCfg<D>::SLAB + (kk & 3) * 32;
        mma_ss(d_tmem, smem_desc_sw128(a + off, 16, 1024), smem_desc_sw128(b + off, 16, 1024), ID, kk > 0);
    }
}

// D (+)= A[tmem, 128 x 128 bf16] B, B a [128 rows = K][D] tile read MN-major.
// A is packed by the two halves of the elementwise warps: K columns
// [64h, 64h + 64) of A (32 TMEM columns of bf16 pairs) sit at TMEM columns
// [64h + 32, 64h + 64) of the 128-column region at a_tmem, the upper half of
// the columns that half h itself loaded its inputs from.
__device__ __forceinline__ uint32_t packed_col(int kk)
{
    return (uint32_t)((kk >> 2) * 64 + 32 + (kk & 3) * 8);
}

template <int D>
__device__ __forceinline__ void issue_tmem_times_tile(uint32_t d_tmem, uint32_t a_tmem, uint32_t b,
                                                      bool accumulate)
{
    constexpr uint32_t ID = idesc_bf16_f32(128, D, 1);
#pragma unroll
    for (int kk = 0; kk < RA_TILE / 16; ++kk)
        mma_ts(d_tmem, a_tmem + packed_col(kk), smem_desc_sw128(b + kk * 2048, BwdCfg<D>::SLAB, 1024), ID,
               (accumulate || kk > 0) ? 1u : 0u);
}

// Iterations of one unit (tile pairs it visits), counted per ring step.
__device__ __forceinline__ int dkdv_count(int j, int tb, const BwdParams &p)
{
    int n = 0;
    for (int s = 0; s < p.N; ++s) {
        const int cls = ra_block_class(p.layout, p.causal, (j + s) % p.N, j);
        const int first = cls == RA_CLS_FULL ? 0 : tb;
        if (cls != RA_CLS_SKIP && first < p.ntiles)
            n += (p.H / p.Hkv) * (p.ntiles - first);
    }
    return n;
}

__device__ __forceinline__ int dq_count(int i, int ta, const BwdParams &p)
{
    int n = 0;
    for (int s = 0; s < p.N; ++s)
        n += ra_kv_tiles(ra_block_class(p.layout, p.causal, i, ra_ring_block(i, s, p.N)), ta, p.ntiles);
    return n;
}

__device__ __forceinline__ void bwd_init_barriers(BwdCtrl *ctrl)
{
    mbar_init(smem_u32(&ctrl->once_full), 1);
    for (int s = 0; s < 2; ++s) {
        mbar_init(smem_u32(&ctrl->st_full[s]), 1);
        mbar_init(smem_u32(&ctrl->st_empty[s]), 1);
        mbar_init(smem_u32(&ctrl->s_full[s]), 1);
    }
    for (int s = 0; s < 3; ++s) {
        mbar_init(smem_u32(&ctrl->kf[s]), 1);
        mbar_init(smem_u32(&ctrl->ke[s]), 1);
    }
    mbar_init(smem_u32(&ctrl->dp_full), 1);
    mbar_init(smem_u32(&ctrl->p_full), BWD_EW);
    mbar_init(smem_u32(&ctrl->ds_full), BWD_EW);
    mbar_init(smem_u32(&ctrl->final_bar), 1);
    ctrl->abort = 0;
    fence_mbar_init();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint4 pack8(const uint32_t (&o)[32], int e, float mul, bool zero)
{
    uint4 v;
    v.x = zero ? 0u : pack_bf16x2(__uint_as_float(o[8 * e + 0]) * mul, __uint_as_float(o[8 * e + 1]) * mul);
    v.y = zero ? 0u : pack_bf16x2(__uint_as_float(o[8 * e + 2]) * mul, __uint_as_float(o[8 * e + 3]) * mul);
    v.z = zero ? 0u : pack_bf16x2(__uint_as_float(o[8 * e + 4]) * mul, __uint_as_float(o[8 * e + 5]) * mul);
    v.w = zero ? 0u : pack_bf16x2(__uint_as_float(o[8 * e + 6]) * mul, __uint_as_float(o[8 * e + 7]) * mul);
    return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// ------------------------------------------------------------------ dK, dV
// Per query tile n the elementwise warps release P^T before they compute dS^T,
// so the tensor pipe runs dV(n) and S^T(n + 1) while dS^T(n) is formed, and
// dK(n), dP^T(n + 1) while P^T(n + 1) is formed.  dS^T takes P from the bf16
// values just packed for the dV product (kept in registers).
template <int D>
__global__ void __launch_bounds__(BWD_THREADS, 1) ra_bwd_dkdv_kernel(const __grid_constant__ BwdParams p)
{
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);
    BwdCtrl *ctrl = reinterpret_cast<BwdCtrl *>(smem + C::KV_OFF_CTRL);
    float *rows = reinterpret_cast<float *>(smem + C::KV_OFF_ROWS);  // [st][nl|dl][128]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto bar = [&](uint64_t &b) { return smem_u32(&b); };

    int bhkv, j, tb;
    ra_bwd_dkdv_unit(blockIdx.x, p.B, p.Hkv, p.N, p.ntiles, p.layout, ra_bwd_kv_outer(p.B, p.Hkv, p.S), bhkv, j,
                     tb);
    const int b = bhkv / p.Hkv, g = bhkv % p.Hkv, grp = p.H / p.Hkv;
    const int kvrow = bhkv * p.S + j * p.L + tb * RA_TILE;

    if (threadIdx.x == 0)
        bwd_init_barriers(ctrl);
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctrl->tmem_base), BWD_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    volatile int *abort = &ctrl->abort;
    const uint64_t tmo = p.timeout_ns;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        const uint64_t pol_kv = l2_policy_evict_first();
        const uint64_t pol_q = l2_policy_evict_last();
        if (lane == 0) {
            mbar_arrive_expect_tx(bar(ctrl->once_full), 2 * C::TILE);
            bload_tile<D>(sb + C::KV_OFF_K, &p.tm_k, kvrow, bar(ctrl->once_full), pol_kv);
            bload_tile<D>(sb + C::KV_OFF_V, &p.tm_v, kvrow, bar(ctrl->once_full), pol_kv);
        }
        uint32_t n = 0;
        bool ok = true;
        RaQWalk w;
        w.start(j, tb, p.N, p.layout, p.causal, p.ntiles, grp);
        for (; w.valid(); w.advance(), ++n) {
            const int st = n & 1;
            const int bh = b * p.H + g * grp + w.hh;
            const long long row0 = (long long)bh * p.S + (long long)w.i * p.L + w.ta * RA_TILE;
            // the tile's -lse log2e and delta rows: loaded before the stage
            // wait, so that their latency overlaps it
            float nlv[4], dlv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = lane + 32 * e;
                const bool valid = w.ta * RA_TILE + r < p.L;
                nlv[e] = valid ? -p.lse[row0 + r] * LOG2E : 0.f;
                dlv[e] = valid ? p.delta[row0 + r] : 0.f;
            }
            if (n >= 2) {
                if (lane == 0) {
                    // the stage frees only after dK(n - 2): have the tiles in L2 by then
                    bprefetch_tile<D>(&p.tm_q, (int)row0);
                    bprefetch_tile<D>(&p.tm_do, (int)row0);
                }
                if (!(ok = bwait_warp(p.status, bar(ctrl->st_empty[st]), ((n >> 1) - 1) & 1, abort, tmo,
                                      BS_ST_EMPTY)))
                    break;
            }
            // the copies go out first; the stage's one arrival follows the row
            // stores, so the phase completes with both the bytes and the rows
            const uint32_t full = bar(ctrl->st_full[st]);
            if (lane == 0) {
                mbar_expect_tx(full, 2 * C::TILE);
                bload_tile<D>(sb + C::KV_OFF_Q + st * C::TILE, &p.tm_q, (int)row0, full, pol_q);
                bload_tile<D>(sb + C::KV_OFF_DO + st * C::TILE, &p.tm_do, (int)row0, full, pol_q);
            }
            float *nl = rows + st * 256, *dl = nl + 128;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                nl[lane + 32 * e] = nlv[e];
                dl[lane + 32 * e] = dlv[e];
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(full);
            __syncwarp();
        }
        if (lane == 0) {
            // every issued copy lands before shared memory is released
            bdrain(p.status, bar(ctrl->once_full), 0, tmo);
            for (uint32_t m = n > 2 ? n - 2 : 0; m < n; ++m)
                bdrain(p.status, bar(ctrl->st_full[m & 1]), (m >> 1) & 1, tmo);
        }
        (void)ok;
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop on warp-uniform values, waits included;
        // one lane, elected once, issues every MMA and commit (as in the
        // forward kernel: the pipe idles while the issuing thread does
        // anything else, and waits cost least in converged, uniform code).
        const bool leader = elect_one();
        const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
        const uint32_t sK = sb + C::KV_OFF_K, sV = sb + C::KV_OFF_V;
        const int T = dkdv_count(j, tb, p);
        auto sQ = [&](int n) { return sb + C::KV_OFF_Q + (n & 1) * C::TILE; };
        auto sDO = [&](int n) { return sb + C::KV_OFF_DO + (n & 1) * C::TILE; };
        auto ww = [&](uint32_t bb, uint32_t parity, unsigned int site) {
            return bwait_warp(p.status, bb, parity, abort, tmo, site);
        };
        bool ok = ww(bar(ctrl->once_full), 0, BS_KV_FULL);
        if (ok && T > 0) {
            if ((ok = ww(bar(ctrl->st_full[0]), 0, BS_ST_FULL))) {
                tc_fence_after();
                if (leader) {
                    issue_rows_dot<D>(tm, sK, sQ(0));        // S^T(0) = K Q^T
                    mma_commit(bar(ctrl->s_full[0]));
                    issue_rows_dot<D>(tm + 128, sV, sDO(0));  // dP^T(0) = V dO^T
                    mma_commit(bar(ctrl->dp_full));
                }
                __syncwarp();
            }
        }
        // One query tile per step, specialised on the stage parity (Q and dO
        // in two stages): every address below is a base plus a constant.
        auto step = [&](auto st_c, int n) -> bool {
            constexpr uint32_t ST = decltype(st_c)::value, ST1 = ST ^ 1u;
            const uint32_t sQn = sb + C::KV_OFF_Q + ST * C::TILE, sDOn = sb + C::KV_OFF_DO + ST * C::TILE;
            const uint32_t sQ1 = sb + C::KV_OFF_Q + ST1 * C::TILE, sDO1 = sb + C::KV_OFF_DO + ST1 * C::TILE;
            const bool next = n + 1 < T;
            if (!ww(bar(ctrl->p_full), n & 1, BS_P_FULL))
                return false;
            tc_fence_after();
            if (leader)
                issue_tmem_times_tile<D>(tm + 256, tm, sDOn, n > 0);  // dV += P^T dO
            __syncwarp();
            if (next) {
                if (!ww(bar(ctrl->st_full[ST1]), ((n + 1) >> 1) & 1, BS_ST_FULL))
                    return false;
                tc_fence_after();
                if (leader) {
                    issue_rows_dot<D>(tm, sK, sQ1);  // S^T(n+1): P^T(n) consumed in order
                    mma_commit(bar(ctrl->s_full[0]));
                }
                __syncwarp();
            }
            if (!ww(bar(ctrl->ds_full), n & 1, BS_S_FULL))
                return false;
            tc_fence_after();
            if (leader) {
                issue_tmem_times_tile<D>(tm + 256 + D, tm + 128, sQn, n > 0);  // dK += dS^T Q
                mma_commit(bar(ctrl->st_empty[ST]));
                if (next) {
                    issue_rows_dot<D>(tm + 128, sV, sDO1);  // dP^T(n+1): dS^T(n) consumed in order
                    mma_commit(bar(ctrl->dp_full));
                }
            }
            __syncwarp();
            return true;
        };
        for (int n = 0; ok && n < T; ++n)
            ok = (n & 1) ? step(std::integral_constant<uint32_t, 1>{}, n) : step(std::integral_constant<uint32_t, 0>{}, n);
        if (leader)
            mma_commit(bar(ctrl->final_bar));
        __syncwarp();
        bdrain(p.status, bar(ctrl->final_bar), 0, tmo);
    } else {
        // ------------------------------------------------------------ elementwise
        // Two warps per TMEM lane quarter: half h takes query columns
        // [64h, 64h + 64).  Its packed P^T / dS^T land in columns
        // [64h + 32, 64h + 64) of the S^T / dP^T region, inside the columns it
        // loaded itself, so the halves never wait for each other.
        const int qw = warp & 3;
        const int h = (warp - 2) >> 2;
        const int r = qw * 32 + lane;                 // key row of the tile
        const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
        const uint32_t tS = tmem + lane_off, tP = tS + 128;
        const int bl = tb * RA_TILE + r;              // key local index in block j
        const bool key_ok = bl < p.L;
        const float sl2 = p.scale_log2;
        uint32_t n = 0;
        bool ok = true;
        RaQWalk w;
        w.start(j, tb, p.N, p.layout, p.causal, p.ntiles, grp);
        for (; w.valid(); w.advance(), ++n) {
            if (!(ok = bwait_warp(p.status, bar(ctrl->s_full[0]), n & 1, abort, tmo, BS_S_FULL)))
                break;
            // the producer's lse / delta stores for this stage, made visible by
            // the stage's own barrier (complete: S^T waited for it)
            if (!(ok = bwait_warp(p.status, bar(ctrl->st_full[n & 1]), (n >> 1) & 1, abort, tmo, BS_ST_FULL)))
                break;
            tc_fence_after();
            const float *nl = rows + (n & 1) * 256 + 64 * h, *dl = nl + 128;
            // visible iff lo <= a < L for the query local index a
            const int lo = !key_ok ? p.L : (w.cls == RA_CLS_FULL ? 0 : bl + (w.cls == RA_CLS_DIAG_EXCL ? 1 : 0));
            const int a0 = w.ta * RA_TILE + 64 * h;
            uint32_t xs[64], pp[32];
            tmem_ld64(tS + 64 * h, xs);
            tmem_wait_ld();
            // P^T = 2^(S^T c log2e - lse log2e), masked where some query of the
            // warp's half-tile does not see the warp's keys
            const float2 sl2x2 = make_float2(sl2, sl2);
            const float2 *nl2 = reinterpret_cast<const float2 *>(nl);
            if (__all_sync(0xffffffffu, lo <= a0 && a0 + 64 <= p.L)) {
#pragma unroll
                for (int e = 0; e < 64; e += 2) {
                    const float2 t = ffma2(make_float2(__uint_as_float(xs[e]), __uint_as_float(xs[e + 1])), sl2x2,
                                           nl2[e >> 1]);
                    pp[e >> 1] = pack_bf16x2(ex2_approx(t.x), ex2_approx(t.y));
                }
            } else {
#pragma unroll
                for (int e = 0; e < 64; e += 2) {
                    const float2 t = ffma2(make_float2(__uint_as_float(xs[e]), __uint_as_float(xs[e + 1])), sl2x2,
                                           nl2[e >> 1]);
                    float p0 = ex2_approx(t.x), p1 = ex2_approx(t.y);
                    p0 = (a0 + e >= lo && a0 + e < p.L) ? p0 : 0.f;
                    p1 = (a0 + e + 1 >= lo && a0 + e + 1 < p.L) ? p1 : 0.f;
                    pp[e >> 1] = pack_bf16x2(p0, p1);
                }
            }
            tmem_st32(tS + 64 * h + 32, pp);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(ctrl->p_full));
            // dS^T = P^T (dP^T - delta), P^T as packed for the dV product
            if (!(ok = bwait_warp(p.status, bar(ctrl->dp_full), n & 1, abort, tmo, BS_S_FULL)))
                break;
            tc_fence_after();
            uint32_t xd[64], pd[32];
            tmem_ld64(tP + 64 * h, xd);
            tmem_wait_ld();
            const float2 *dl2 = reinterpret_cast<const float2 *>(dl);
            const float2 zero2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < 64; e += 2) {
                const uint32_t pk = pp[e >> 1];
                const float2 nd = dl2[e >> 1];
                const float2 t = fadd2(make_float2(__uint_as_float(xd[e]), __uint_as_float(xd[e + 1])),
                                       make_float2(-nd.x, -nd.y));
                const float2 ds = ffma2(make_float2(bf16_lo(pk), bf16_hi(pk)), t, zero2);
                pd[e >> 1] = pack_bf16x2(ds.x, ds.y);
            }
            tmem_st32(tP + 64 * h + 32, pd);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(ctrl->ds_full));
        }
        // ------------------------------------------------------------ epilogue
        // half 0 writes dV, half 1 dK
        if (ok)
            ok = bwait_warp(p.status, bar(ctrl->final_bar), 0, abort, tmo, BS_FINAL);
        if (ok) {
            tc_fence_after();
            const long long orow = (long long)kvrow + r;
            __nv_bfloat16 *dst = h == 0 ? p.dv : p.dk;
            const float mul = h == 0 ? 1.f : p.scale;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                __syncwarp();
                tmem_ld32(tS + 256 + h * D + c * 32, o);
                tmem_wait_ld();
                if (!key_ok)
                    continue;
                uint4 *out = reinterpret_cast<uint4 *>(dst + orow * D + c * 32);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    out[e] = pack8(o, e, mul, n == 0);  // n == 0: no query tile met this key tile
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, BWD_TMEM_COLS);
    }
}

// ------------------------------------------------------------------ dQ
// Two S buffers (columns [0,128) and [384,512)): S(n + 2) is computed while
// the elementwise warps work on tile n + 1, and dP(n + 1) is issued before
// dQ(n), so the elementwise work of one key tile waits only for its dP.
template <int D>
__global__ void __launch_bounds__(BWD_THREADS, 1) ra_bwd_dq_kernel(const __grid_constant__ BwdParams p)
{
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);
    BwdCtrl *ctrl = reinterpret_cast<BwdCtrl *>(smem + C::Q_OFF_CTRL);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto bar = [&](uint64_t &b) { return smem_u32(&b); };

    int bh, i, ta;
    ra_bwd_dq_unit(blockIdx.x, p.B, p.H, p.Hkv, p.N, p.ntiles, p.layout, ra_bwd_kv_outer(p.B, p.Hkv, p.S), bh, i,
                   ta);
    const int b = bh / p.H, h = bh % p.H;
    const int kvbh = b * p.Hkv + h / (p.H / p.Hkv);
    const int qrow = bh * p.S + i * p.L + ta * RA_TILE;

    if (threadIdx.x == 0)
        bwd_init_barriers(ctrl);
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctrl->tmem_base), BWD_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    volatile int *abort = &ctrl->abort;
    const uint64_t tmo = p.timeout_ns;

    if (warp == 0) {
        // producer: the whole warp on uniform values (its waits sit on the path
        // from a freed stage to the next copy), one elected lane issues
        const bool leader = elect_one();
        const uint64_t pol_q = l2_policy_evict_first();
        const uint64_t pol_kv = l2_policy_evict_last();
        if (leader) {
            mbar_arrive_expect_tx(bar(ctrl->once_full), 2 * C::TILE);
            bload_tile<D>(sb + C::Q_OFF_Q, &p.tm_q, qrow, bar(ctrl->once_full), pol_q);
            bload_tile<D>(sb + C::Q_OFF_DO, &p.tm_do, qrow, bar(ctrl->once_full), pol_q);
        }
        __syncwarp();
        uint32_t n = 0;
        bool ok = true;
        RaKWalk w;
        w.start(i, ta, p.N, p.layout, p.causal, p.ntiles);
        uint32_t nk = 0, nv = 0;  // K and V loads issued
        for (; w.valid(); w.advance(), ++n) {
            const int ks = n % C::Q_KST, vs = n & 1;
            const int row = kvbh * p.S + w.j * p.L + w.tb * RA_TILE;
            if (n >= (uint32_t)C::Q_KST) {
                // K's stage frees after dQ(n - 3): have the tile in L2 by then
                if (leader)
                    bprefetch_tile<D>(&p.tm_k, row);
                if (!(ok = bwait_warp(p.status, bar(ctrl->ke[ks]), (n / C::Q_KST - 1) & 1, abort, tmo,
                                      BS_KV_EMPTY)))
                    break;
            }
            if (leader) {
                mbar_arrive_expect_tx(bar(ctrl->kf[ks]), C::TILE);
                bload_tile<D>(sb + C::Q_OFF_K + ks * C::TILE, &p.tm_k, row, bar(ctrl->kf[ks]), pol_kv);
            }
            __syncwarp();
            ++nk;
            if (n >= 2) {
                // V's stage frees once dP(n - 2) has read it
                if (leader)
                    bprefetch_tile<D>(&p.tm_v, row);
                if (!(ok = bwait_warp(p.status, bar(ctrl->st_empty[vs]), ((n >> 1) - 1) & 1, abort, tmo,
                                      BS_KV_EMPTY)))
                    break;
            }
            if (leader) {
                mbar_arrive_expect_tx(bar(ctrl->st_full[vs]), C::TILE);
                bload_tile<D>(sb + C::Q_OFF_V + vs * C::TILE, &p.tm_v, row, bar(ctrl->st_full[vs]), pol_kv);
            }
            __syncwarp();
            ++nv;
        }
        // every issued copy lands before shared memory is released
        bdrain(p.status, bar(ctrl->once_full), 0, tmo);
        for (uint32_t m = nk > (uint32_t)C::Q_KST ? nk - C::Q_KST : 0; m < nk; ++m)
            bdrain(p.status, bar(ctrl->kf[m % C::Q_KST]), (m / C::Q_KST) & 1, tmo);
        for (uint32_t m = nv > 2 ? nv - 2 : 0; m < nv; ++m)
            bdrain(p.status, bar(ctrl->st_full[m & 1]), (m >> 1) & 1, tmo);
        (void)ok;
    } else if (warp == 1) {
        // MMA issuer: the whole warp on uniform values, one elected lane issues
        const bool leader = elect_one();
        const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
        const uint32_t sQ = sb + C::Q_OFF_Q, sDO = sb + C::Q_OFF_DO;
        const int T = dq_count(i, ta, p);
        auto sK = [&](int n) { return sb + C::Q_OFF_K + (n % C::Q_KST) * C::TILE; };
        auto sV = [&](int n) { return sb + C::Q_OFF_V + (n & 1) * C::TILE; };
        auto ww = [&](uint32_t bb, uint32_t parity, unsigned int site) {
            return bwait_warp(p.status, bb, parity, abort, tmo, site);
        };
        auto wait_k = [&](int n) { return ww(bar(ctrl->kf[n % C::Q_KST]), (n / C::Q_KST) & 1, BS_ST_FULL); };
        auto wait_v = [&](int n) { return ww(bar(ctrl->st_full[n & 1]), (n >> 1) & 1, BS_ST_FULL); };
        bool ok = ww(bar(ctrl->once_full), 0, BS_Q_FULL);
        // S(0), dP(0), S(1)
        for (int n = 0; ok && n < 2 && n < T; ++n) {
            if (!(ok = wait_k(n)))
                break;
            tc_fence_after();
            if (leader)
                issue_rows_dot<D>(tm + (n ? 384u : 0u), sQ, sK(n));  // S(n): tracked by dP(n)'s commit
            __syncwarp();
            if (n == 0) {
                if (!(ok = wait_v(0)))
                    break;
                tc_fence_after();
                if (leader) {
                    issue_rows_dot<D>(tm + 128, sDO, sV(0));
                    mma_commit(bar(ctrl->dp_full));
                    mma_commit(bar(ctrl->st_empty[0]));
                }
                __syncwarp();
            }
        }
        // One key tile per step, specialised on n mod 6 (K in three stages,
        // V and the S buffers in two), so every address below is a base plus a
        // constant.
        static_assert(C::Q_KST == 3, "dQ step specialisation assumes three K stages");
        auto step = [&](auto ph_c, int n) -> bool {
            constexpr int PH = decltype(ph_c)::value;
            constexpr uint32_t KS = PH % 3, KS2 = (PH + 2) % 3, VS1 = (PH + 1) & 1;
            constexpr uint32_t SBUF = (PH & 1) ? 384u : 0u;
            if (!ww(bar(ctrl->p_full), n & 1, BS_P_FULL))
                return false;
            tc_fence_after();
            if (n + 1 < T) {
                if (!ww(bar(ctrl->st_full[VS1]), ((n + 1) >> 1) & 1, BS_ST_FULL))
                    return false;
                tc_fence_after();
                if (leader) {
                    issue_rows_dot<D>(tm + 128, sDO, sb + C::Q_OFF_V + VS1 * C::TILE);  // dP(n+1): dP(n) was read
                    mma_commit(bar(ctrl->dp_full));
                    mma_commit(bar(ctrl->st_empty[VS1]));
                }
                __syncwarp();
            }
            if (leader) {
                issue_tmem_times_tile<D>(tm + 256, tm + SBUF, sb + C::Q_OFF_K + KS * C::TILE, n > 0);  // dQ += dS K
                mma_commit(bar(ctrl->ke[KS]));
            }
            __syncwarp();
            if (n + 2 < T) {
                if (!ww(bar(ctrl->kf[KS2]), ((n + 2) / 3) & 1, BS_ST_FULL))
                    return false;
                tc_fence_after();
                if (leader)  // dS(n) consumed in order; S(n + 2) is tracked by dP(n + 2)'s commit
                    issue_rows_dot<D>(tm + SBUF, sQ, sb + C::Q_OFF_K + KS2 * C::TILE);
                __syncwarp();
            }
            return true;
        };
        using std::integral_constant;
        for (int n = 0; ok && n < T; ++n) {
            switch (n % 6) {
            case 0: ok = step(integral_constant<int, 0>{}, n); break;
            case 1: ok = step(integral_constant<int, 1>{}, n); break;
            case 2: ok = step(integral_constant<int, 2>{}, n); break;
            case 3: ok = step(integral_constant<int, 3>{}, n); break;
            case 4: ok = step(integral_constant<int, 4>{}, n); break;
            default: ok = step(integral_constant<int, 5>{}, n); break;
            }
        }
        if (leader)
            mma_commit(bar(ctrl->final_bar));
        __syncwarp();
        bdrain(p.status, bar(ctrl->final_bar), 0, tmo);
    } else {
        // Two warps per TMEM lane quarter, half h on key columns [64h, 64h + 64);
        // packed dS goes to columns [64h + 32, 64h + 64) of the S buffer, inside
        // the columns half h loaded its scores from: the halves never wait for
        // each other.
        const int qw = warp & 3;
        const int h = (warp - 2) >> 2;
        const int r = qw * 32 + lane;
        const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
        const uint32_t tP = tmem + lane_off + 128;
        const int a = ta * RA_TILE + r;
        const bool row_ok = a < p.L;
        const long long grow = (long long)qrow + r;
        const float nl = row_ok ? -p.lse[grow] * LOG2E : 0.f;
        const float dl = row_ok ? p.delta[grow] : 0.f;
        const float sl2 = p.scale_log2;
        uint32_t n = 0;
        bool ok = true;
        RaKWalk w;
        w.start(i, ta, p.N, p.layout, p.causal, p.ntiles);
        for (; w.valid(); w.advance(), ++n) {
            const uint32_t tS = tmem + lane_off + ((n & 1) ? 384u : 0u);
            // S(n) was issued before dP(n) by the same thread, and the commit
            // that signals dP(n) tracks every earlier MMA: one wait covers both
            if (!(ok = bwait_warp(p.status, bar(ctrl->dp_full), n & 1, abort, tmo, BS_S_FULL)))
                break;
            tc_fence_after();
            const int lim = (row_ok ? ra_key_limit(w.cls, a, p.L) - w.tb * RA_TILE : 0) - 64 * h;
            uint32_t xs[64];
            tmem_ld64(tS + 64 * h, xs);
            tmem_wait_ld();
            uint32_t pd[32];
            const float2 sl2x2 = make_float2(sl2, sl2), nl2 = make_float2(nl, nl), ndl2 = make_float2(-dl, -dl);
            const float2 zero2 = make_float2(0.f, 0.f);
            const bool full = __all_sync(0xffffffffu, lim >= 64);  // no key of the half-tile masked
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t xd[32];
                tmem_ld32(tP + 64 * h + 32 * c, xd);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const int x = 32 * c + e;
                    const float2 t = ffma2(make_float2(__uint_as_float(xs[x]), __uint_as_float(xs[x + 1])), sl2x2, nl2);
                    float2 pr = make_float2(ex2_approx(t.x), ex2_approx(t.y));
                    if (!full) {
                        pr.x = x < lim ? pr.x : 0.f;
                        pr.y = x + 1 < lim ? pr.y : 0.f;
                    }
                    const float2 g = fadd2(make_float2(__uint_as_float(xd[e]), __uint_as_float(xd[e + 1])), ndl2);
                    const float2 ds = ffma2(pr, g, zero2);
                    pd[x >> 1] = pack_bf16x2(ds.x, ds.y);
                }
            }
            tmem_st32(tS + 64 * h + 32, pd);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(ctrl->p_full));
        }
        if (ok)
            ok = bwait_warp(p.status, bar(ctrl->final_bar), 0, abort, tmo, BS_FINAL);
        if (ok) {
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < D / 64; ++c) {
                uint32_t o[32];
                __syncwarp();
                tmem_ld32(tmem + lane_off + 256 + h * (D / 2) + c * 32, o);
                tmem_wait_ld();
                if (!row_ok)
                    continue;
                uint4 *out = reinterpret_cast<uint4 *>(p.dq + grow * D + h * (D / 2) + c * 32);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    out[e] = pack8(o, e, p.scale, n == 0);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, BWD_TMEM_COLS);
    }
}

// ------------------------------------------------------------------ delta
// delta[row] = sum_c dO[row, c] O[row, c] in fp32; each thread takes 8
// columns (16 bytes), D / 8 threads per row reduce with shuffles.
template <int D>
__global__ void ra_bwd_delta_kernel(const __nv_bfloat16 *__restrict__ o, const __nv_bfloat16 *__restrict__ dout,
                                    float *__restrict__ delta, long long rows)
{
    constexpr int G = D / 8;  // threads per row
    const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long row = t / G;
    const int part = (int)(t % G);
    float acc = 0.f;
    if (row < rows) {
        const uint4 x = reinterpret_cast<const uint4 *>(o + row * D)[part];
        const uint4 y = reinterpret_cast<const uint4 *>(dout + row * D)[part];
        const __nv_bfloat162 *xa = reinterpret_cast<const __nv_bfloat162 *>(&x);
        const __nv_bfloat162 *ya = reinterpret_cast<const __nv_bfloat162 *>(&y);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 fx = __bfloat1622float2(xa[e]), fy = __bfloat1622float2(ya[e]);
            acc = fmaf(fx.x, fy.x, acc);
            acc = fmaf(fx.y, fy.y, acc);
        }
    }
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1)
        acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (row < rows && part == 0)
        delta[row] = acc;
}

PFN_cuTensorMapEncodeTiled_v12000 bwd_encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

bool bwd_encode_rows(CUtensorMap *tm, const void *base, long long rows, int d)
{
    auto enc = bwd_encode_fn();
    if (!enc)
        return false;
    cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)d * 2};
    cuuint32_t box[2] = {64, RA_TILE};
    cuuint32_t estr[2] = {1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_bwd_d(const BwdLaunch &a, cudaStream_t st)
{
    using C = BwdCfg<D>;
    static std::atomic<int> attr_set[RA_MAX_DEVICES];
    cudaError_t e0 = once_per_device(attr_set, [] {
        cudaError_t e = cudaFuncSetAttribute(ra_bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::KV_LAUNCH_SMEM);
        if (e != cudaSuccess)
            return e;
        return cudaFuncSetAttribute(ra_bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    C::Q_LAUNCH_SMEM);
    });
    if (e0 != cudaSuccess)
        return e0;
    const long long rows = (long long)a.B * a.H * a.S;
    {
        const long long threads = rows * (D / 8);
        const int block = 256;
        ra_bwd_delta_kernel<D><<<(unsigned)((threads + block - 1) / block), block, 0, st>>>(
            static_cast<const __nv_bfloat16 *>(a.out), static_cast<const __nv_bfloat16 *>(a.dout), a.delta, rows);
    }
    BwdParams p;
    memset(&p, 0, sizeof(p));
    if (!bwd_encode_rows(&p.tm_q, a.q, rows, D) ||
        !bwd_encode_rows(&p.tm_k, a.k, (long long)a.B * a.Hkv * a.S, D) ||
        !bwd_encode_rows(&p.tm_v, a.v, (long long)a.B * a.Hkv * a.S, D) ||
        !bwd_encode_rows(&p.tm_do, a.dout, rows, D))
        return cudaErrorInvalidValue;
    p.lse = a.lse, p.delta = a.delta;
    p.dq = static_cast<__nv_bfloat16 *>(a.dq);
    p.dk = static_cast<__nv_bfloat16 *>(a.dk);
    p.dv = static_cast<__nv_bfloat16 *>(a.dv);
    p.B = a.B, p.H = a.H, p.Hkv = a.Hkv, p.S = a.S, p.N = a.N, p.L = a.S / a.N;
    p.layout = a.layout, p.causal = a.causal;
    p.ntiles = (p.L + RA_TILE - 1) / RA_TILE;
    p.scale = 1.0f / sqrtf((float)D);
    p.scale_log2 = LOG2E / sqrtf((float)D);
    p.timeout_ns = a.timeout_ns;
    p.status = device_status_ptr();
    if (!p.status)
        return cudaErrorInvalidValue;
    const long long kv_units = (long long)a.B * a.Hkv * a.N * p.ntiles;
    const long long q_units = (long long)a.B * a.H * a.N * p.ntiles;
    if (kv_units > 0x7fffffffll || q_units > 0x7fffffffll)
        return cudaErrorInvalidValue;
    p.n_units = (int)kv_units;
    ra_bwd_dkdv_kernel<D><<<(unsigned)kv_units, BWD_THREADS, C::KV_LAUNCH_SMEM, st>>>(p);
    p.n_units = (int)q_units;
    ra_bwd_dq_kernel<D><<<(unsigned)q_units, BWD_THREADS, C::Q_LAUNCH_SMEM, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdLaunch &a, cudaStream_t st)
{
    if (a.d == 128)
        return launch_bwd_d<128>(a, st);
    if (a.d == 64)
        return launch_bwd_d<64>(a, st);
    return cudaErrorInvalidValue;
}

}  // namespace ra
