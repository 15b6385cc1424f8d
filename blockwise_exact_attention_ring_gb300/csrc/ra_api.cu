// C-ABI layer of libra.so: argument validation, workspace layout, the host
// ring-step scheduler, and the stream-ordered launch sequence.  See
// include/ra.h for the contract of every entry point.
#include <cstdio>
#include <nvtx3/nvToolsExt.h>
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/ra.h"
#include "ra_bwd_schedule.h"
#include "ra_internal.h"
#include "ra_schedule.h"

namespace {



constexpr unsigned long long kDefaultTimeoutNs = 4000000000ull;  // 4 s per wait
unsigned long long g_timeout_ns = kDefaultTimeoutNs;
std::atomic<unsigned long long> g_launches{0};
// Host-side NVTX range around the enqueue of one phase (permute, attention,
// ring step, merge, finalise).  A no-op unless a profiler or tracing tool is
// attached; with one, timelines show the library's phases by name.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

// 0 automatic (= 3), 1 single-CTA, 3 single-CTA kernel in clusters of two
// sharing each K/V load where the heads allow it (2 is not a valid value)
std::atomic<int> g_kernel_variant{0};

void count_launch(unsigned long long n = 1) { g_launches.fetch_add(n, std::memory_order_relaxed); }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Largest number of pieces a unit's ring walk is split into (split_count).
constexpr int kMaxSplit = 16;

int sm_count_current()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        return 1;
    return n;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A caller buffer: its first byte and its size.
struct Span {
    const void *p;
    size_t bytes;
};

// True when every buffer starts in device memory of the current device.
// The kernels' tensor maps (TMA copies, which the default forward launch
// multicasts to both CTAs of a cluster) must cover this GPU's own memory
// only, so pinned or plain host memory, managed memory and a peer GPU's
// memory reached through unified addressing are refused.  One
// cudaPointerGetAttributes per buffer (its first byte: an allocation lies in
// one memory).  Null pointers and empty buffers are skipped (the callers
// reject or allow them before this check).
bool resident_here(std::initializer_list<Span> bufs)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    for (const Span &b : bufs) {
        if (!b.p || b.bytes == 0)
            continue;
        cudaPointerAttributes at{};
        if (cudaPointerGetAttributes(&at, b.p) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        if (at.type != cudaMemoryTypeDevice || at.device != dev)
            return false;
    }
    return true;
}

struct Problem {
    int B, H, Hkv, S, d, N, layout, causal, dtype, mode;
    bool rank_major = false;  // inputs/outputs already in the layout's rank order
    long long L() const { return S / N; }
    size_t esz() const { return dtype == RA_DTYPE_F32 ? 4 : 2; }
    size_t q_elems() const { return (size_t)B * H * S * d; }
    size_t kv_elems() const { return (size_t)B * Hkv * S * d; }
    size_t rows() const { return (size_t)B * H * S; }
};

// Validation shared by every forward entry point.  Returns RA_OK or the
// status to report.
ra_status check_problem(const Problem &p)
{
    if (p.B < 1 || p.H < 1 || p.Hkv < 1 || p.S < 1 || p.d < 1 || p.N < 1)
        return RA_ERR_INVALID_ARG;
    if (p.H % p.Hkv != 0 || p.S % p.N != 0)
        return RA_ERR_INVALID_ARG;
    if (p.layout != RA_LAYOUT_CONTIGUOUS && p.layout != RA_LAYOUT_STRIPED)
        return RA_ERR_INVALID_ARG;
    if (p.causal != 0 && p.causal != 1)
        return RA_ERR_INVALID_ARG;
    if (p.dtype != RA_DTYPE_BF16 && p.dtype != RA_DTYPE_F32)
        return RA_ERR_INVALID_ARG;
    if (p.mode != RA_MODE_FUSED && p.mode != RA_MODE_PER_STEP && p.mode != RA_MODE_RING)
        return RA_ERR_INVALID_ARG;
    // 32-bit TMA row coordinates and grid limits
    if ((long long)p.B * p.H * p.S >= (1ll << 31) || (long long)p.B * p.H > 65535)
        return RA_ERR_UNSUPPORTED;
    if (p.dtype == RA_DTYPE_BF16 && p.d != 64 && p.d != 128)
        return RA_ERR_UNSUPPORTED;
    if (p.dtype == RA_DTYPE_F32 && p.d > 256)
        return RA_ERR_UNSUPPORTED;
    if (p.mode != RA_MODE_FUSED && p.d % 4 != 0)
        return RA_ERR_UNSUPPORTED;
    return RA_OK;
}

// Pieces the fused bf16 kernel cuts every unit's walk over its key tiles
// into.  The ring's own decomposition: the key tiles a query tile meets are
// independent partial results that the running softmax combines, so when the
// work units cannot fill half the SMs, each unit's walk (in ring order) is
// split into up to sm / units contiguous pieces, computed by different CTAs
// and combined afterwards.  1 otherwise (and for the fp32 and per-step paths).
int split_count(const Problem &p, int sm)
{
    if (p.mode != RA_MODE_FUSED || p.dtype != RA_DTYPE_BF16)
        return 1;
    const RaUnitSpace sp = ra_unit_space(p.B, p.H, p.Hkv, p.S, p.N, p.layout, p.causal, 0, p.N);
    const long long units = ra_unit_count(sp);
    if (units < 1 || 2 * units > sm)
        return 1;
    const int heaviest = ra_unit_decode(sp, 0).cost;  // the order is heaviest first
    long long n = sm / units;
    if (n > kMaxSplit)
        n = kMaxSplit;
    if (n > heaviest)
        n = heaviest;
    return n > 1 ? (int)n : 1;
}

// Workspace layout (each region 256-byte aligned):
//   striped:            q', k', v' in striped order
//   striped and fused:  out', lse' in striped order (unless split)
//   fused, split:       nsplit fp32 partials of out and lse (kernel order)
//   per-step and ring:  running out/lse (fp32) and step partial out/lse (fp32)
//   ring:               two rotating copies of k and v (rank-major order)
struct WsLayout {
    size_t q = 0, k = 0, v = 0, out = 0, lse = 0, run = 0, run_lse = 0, part = 0, part_lse = 0;
    size_t ring_k[2] = {0, 0}, ring_v[2] = {0, 0};
    size_t split = 0, split_lse = 0;
    int nsplit = 1;
    size_t total = 0;
};

WsLayout ws_layout(const Problem &p, int sm)
{
    WsLayout w;
    w.nsplit = split_count(p, sm);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += align256(bytes);
        return at;
    };
    if (p.layout == RA_LAYOUT_STRIPED && !p.rank_major) {
        w.q = take(p.q_elems() * p.esz());
        w.k = take(p.kv_elems() * p.esz());
        w.v = take(p.kv_elems() * p.esz());
        if (p.mode == RA_MODE_FUSED && w.nsplit == 1) {
            w.out = take(p.q_elems() * p.esz());
            w.lse = take(p.rows() * 4);
        }
    }
    if (w.nsplit > 1) {
        w.split = take((size_t)w.nsplit * p.q_elems() * 4);
        w.split_lse = take((size_t)w.nsplit * p.rows() * 4);
    }
    if (p.mode != RA_MODE_FUSED) {
        w.run = take(p.q_elems() * 4);
        w.run_lse = take(p.rows() * 4);
        w.part = take(p.q_elems() * 4);
        w.part_lse = take(p.rows() * 4);
    }
    if (p.mode == RA_MODE_RING && p.N > 1) {
        for (int b = 0; b < 2; ++b) {
            w.ring_k[b] = take(p.kv_elems() * p.esz());
            w.ring_v[b] = take(p.kv_elems() * p.esz());
        }
    }
    w.total = off;
    return w;
}

// ------------------------------------------------------------------ forward
ra_status attention_pass(const Problem &p, const void *q, const void *k, const void *v, void *out,
                         float *lse, int s_begin, int s_end, bool out_f32, int sm, cudaStream_t st,
                         int rank_lo = 0, int rank_hi = -1, int nsplit = 1)
{
    if (rank_hi < 0)
        rank_hi = p.N;
    if (p.dtype == RA_DTYPE_F32) {
        ra::launch_attn_f32((const float *)q, (const float *)k, (const float *)v, (float *)out, lse,
                            p.B, p.H, p.Hkv, p.S, p.d, p.N, p.layout, p.causal, s_begin, s_end, rank_lo,
                            rank_hi, st);
        count_launch();
        return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_CUDA;
    }
    ra::TcLaunch a{};
    a.q = q, a.k = k, a.v = v, a.out = out, a.lse = lse;
    a.B = p.B, a.H = p.H, a.Hkv = p.Hkv, a.S = p.S, a.d = p.d, a.N = p.N;
    a.layout = p.layout, a.causal = p.causal, a.s_begin = s_begin, a.s_end = s_end;
    a.rank_lo = rank_lo, a.rank_hi = rank_hi;
    a.out_f32 = out_f32 ? 1 : 0;
    a.timeout_ns = g_timeout_ns;
    a.sm_count = sm;
    a.nsplit = nsplit;
    a.split_out_bytes = (long long)p.q_elems() * 4;
    a.split_lse_stride = (long long)p.rows();
    const RaUnitSpace sp = ra_unit_space_ranks(ra_unit_space(p.B, p.H, p.Hkv, p.S, p.N, p.layout, p.causal,
                                                             s_begin, s_end),
                                               rank_lo, rank_hi);
    const int variant = g_kernel_variant.load(std::memory_order_relaxed);
    a.cluster = variant == 1 ? 1 : 2;
    if (ra_unit_count(sp) == 0)
        return ra::launch_attn_tc(a, st) == cudaSuccess ? RA_OK : RA_ERR_CUDA;
    // Large problems (the order grouped by kv head, from 2^19 key/value rows)
    // go kv head by kv head, one launch per (batch, kv head) on contiguous
    // slices: the heads are independent and each alone still fills the GPU,
    // and dealing each head's heaviest-first units from round 0 balances the
    // CTAs better than one snake over all heads, whose heavy-to-light runs
    // fall out of phase with the rounds (host simulation of the dealing at
    // 256K tokens: 2.3 % of idle tail against 0.1 %; measured +2 % at 256K,
    // +1 % at 1M tokens).  Every unit is computed as in the single launch.
    if (nsplit == 1 && sp.kv_outer && (long long)p.B * p.Hkv > 1) {
        const int g = p.H / p.Hkv;
        const long long q_head = (long long)g * p.S * p.d, kv_head = (long long)p.S * p.d;
        const int out_esz = out_f32 ? 4 : 2;
        for (long long bh = 0; bh < (long long)p.B * p.Hkv; ++bh) {
            ra::TcLaunch b = a;
            b.B = 1, b.H = g, b.Hkv = 1;
            b.q = static_cast<const char *>(q) + bh * q_head * 2;
            b.k = static_cast<const char *>(k) + bh * kv_head * 2;
            b.v = static_cast<const char *>(v) + bh * kv_head * 2;
            b.out = static_cast<char *>(out) + bh * q_head * out_esz;
            b.lse = lse + bh * g * p.S;
            count_launch();
            if (ra::launch_attn_tc(b, st) != cudaSuccess)
                return RA_ERR_CUDA;
        }
        return RA_OK;
    }
    count_launch();
    return ra::launch_attn_tc(a, st) == cudaSuccess ? RA_OK : RA_ERR_CUDA;
}

// ------------------------------------------------------------------ ring copies
// The copy stream of each device: created once, non-blocking, lives as long
// as the process.
cudaStream_t copy_stream()
{
    static std::mutex mu;
    static std::vector<cudaStream_t> streams;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if ((int)streams.size() <= dev)
        streams.resize(dev + 1, nullptr);
    if (!streams[dev] && cudaStreamCreateWithFlags(&streams[dev], cudaStreamNonBlocking) != cudaSuccess) {
        cudaGetLastError();
        streams[dev] = nullptr;
    }
    return streams[dev];
}

// Key/value rotation of RA_MODE_RING.  Buffers R[0], R[1] hold the blocks in
// natural block positions: at step t >= 1 every rank i reads block
// j = (i - t) mod N, which the copy for step t moved there from the buffer of
// step t - 1 (where rank i - 1 held it).  Step 0 reads the inputs.  Copy t
// writes R[(t - 1) % 2], last read by step t - 2, so it waits for that step;
// it runs on the copy stream while step t - 1 computes.
struct RingCopies {
    const Problem *p = nullptr;
    cudaStream_t cs = nullptr;
    const char *k0 = nullptr, *v0 = nullptr;
    char *rk[2] = {nullptr, nullptr}, *rv[2] = {nullptr, nullptr};
    std::vector<cudaEvent_t> copied, computed;
    cudaEvent_t fork = nullptr, join = nullptr;

    ~RingCopies()
    {
        for (cudaEvent_t e : copied)
            if (e)
                cudaEventDestroy(e);
        for (cudaEvent_t e : computed)
            if (e)
                cudaEventDestroy(e);
        if (fork)
            cudaEventDestroy(fork);
        if (join)
            cudaEventDestroy(join);
    }

    bool make(cudaEvent_t &e) { return cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess; }

    // copy t: every rank's block for step t into R[(t - 1) % 2].  Rank i
    // receives block (i - t) mod N from rank i - 1; over all ranks that is
    // every block once, at the same offset in source and destination, so the
    // N sends of a step are one copy of K and one of V (one call each keeps
    // the host's enqueue cost off small steps).
    bool copy(int t)
    {
        const Problem &P = *p;
        const size_t bytes = P.kv_elems() * P.esz();
        const char *sk = t == 1 ? k0 : rk[t % 2], *sv = t == 1 ? v0 : rv[t % 2];
        char *dk = rk[(t - 1) % 2], *dv = rv[(t - 1) % 2];
        if (t >= 3 && cudaStreamWaitEvent(cs, computed[t - 2], 0) != cudaSuccess)
            return false;
        if (cudaMemcpyAsync(dk, sk, bytes, cudaMemcpyDeviceToDevice, cs) != cudaSuccess ||
            cudaMemcpyAsync(dv, sv, bytes, cudaMemcpyDeviceToDevice, cs) != cudaSuccess)
            return false;
        return cudaEventRecord(copied[t], cs) == cudaSuccess;
    }

    ra_status begin(const Problem &P, const void *k, const void *v, char *base, const WsLayout &w,
                    cudaStream_t st)
    {
        p = &P;
        k0 = static_cast<const char *>(k), v0 = static_cast<const char *>(v);
        if (P.N == 1)
            return RA_OK;
        for (int b = 0; b < 2; ++b)
            rk[b] = base + w.ring_k[b], rv[b] = base + w.ring_v[b];
        cs = copy_stream();
        if (!cs)
            return RA_ERR_CUDA;
        copied.assign(P.N, nullptr), computed.assign(P.N, nullptr);
        for (int s = 0; s < P.N; ++s)
            if (!make(copied[s]) || !make(computed[s]))
                return RA_ERR_CUDA;
        if (!make(fork) || !make(join))
            return RA_ERR_CUDA;
        // the copy stream starts after everything already on st (the inputs)
        if (cudaEventRecord(fork, st) != cudaSuccess || cudaStreamWaitEvent(cs, fork, 0) != cudaSuccess)
            return RA_ERR_CUDA;
        return copy(1) ? RA_OK : RA_ERR_CUDA;
    }

    // K and V that step s reads; waits on st for their copy
    ra_status before_step(int s, const void **k, const void **v, cudaStream_t st)
    {
        if (s == 0 || p->N == 1) {
            *k = k0, *v = v0;
            return RA_OK;
        }
        if (cudaStreamWaitEvent(st, copied[s], 0) != cudaSuccess)
            return RA_ERR_CUDA;
        *k = rk[(s - 1) % 2], *v = rv[(s - 1) % 2];
        return RA_OK;
    }

    // after step s's launches: record it, start the copy for step s + 2
    ra_status after_step(int s, cudaStream_t st)
    {
        if (p->N == 1)
            return RA_OK;
        if (cudaEventRecord(computed[s], st) != cudaSuccess)
            return RA_ERR_CUDA;
        if (s + 2 < p->N && !copy(s + 2))
            return RA_ERR_CUDA;
        return RA_OK;
    }

    // st waits for the copy stream (no copy outlives the call's stream order)
    ra_status end(cudaStream_t st)
    {
        if (p->N == 1)
            return RA_OK;
        if (cudaEventRecord(join, cs) != cudaSuccess || cudaStreamWaitEvent(st, join, 0) != cudaSuccess)
            return RA_ERR_CUDA;
        return RA_OK;
    }
};

// Pointer checks shared by the forward entry points that take q, k, v, out
// and lse in natural or rank-major order: non-null, 16-byte aligned, outputs
// disjoint from the inputs and from each other.
ra_status check_forward_ptrs(const Problem &p, const void *q, const void *k, const void *v, const void *out,
                             const float *lse)
{
    if (!q || !k || !v || !out || !lse)
        return RA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
        return RA_ERR_INVALID_ARG;
    const size_t qb = p.q_elems() * p.esz(), kvb = p.kv_elems() * p.esz(), lb = p.rows() * 4;
    for (const void *in : {q, k, v})
        if (overlaps(out, qb, in, in == q ? qb : kvb) || overlaps(lse, lb, in, in == q ? qb : kvb))
            return RA_ERR_INVALID_ARG;
    if (overlaps(out, qb, lse, lb))
        return RA_ERR_INVALID_ARG;
    return RA_OK;
}

bool forward_resident(const Problem &p, const void *q, const void *k, const void *v, const void *out,
                      const float *lse)
{
    const size_t qb = p.q_elems() * p.esz(), kvb = p.kv_elems() * p.esz(), lb = p.rows() * 4;
    return resident_here({{q, qb}, {k, kvb}, {v, kvb}, {out, qb}, {lse, lb}});
}

// resident_checked: the caller has checked that q, k, v, out and lse are
// device memory of the current device; ws_internal: ws is the library's own
// scratch array (no residency check needed).
ra_status forward_impl(const Problem &p, const void *q, const void *k, const void *v, void *out,
                       float *lse, void *ws, size_t ws_bytes, cudaStream_t st, bool resident_checked = false,
                       bool ws_internal = false)
{
    ra_status rs = check_problem(p);
    if (rs != RA_OK)
        return rs;
    if ((rs = check_forward_ptrs(p, q, k, v, out, lse)) != RA_OK)
        return rs;
    const int sm = sm_count_current();
    const WsLayout w = ws_layout(p, sm);
    if (w.total > 0 && (!ws || ws_bytes < w.total || (reinterpret_cast<uintptr_t>(ws) & 255u)))
        return RA_ERR_WORKSPACE;
    if (!resident_checked && !forward_resident(p, q, k, v, out, lse))
        return RA_ERR_INVALID_ARG;
    if (w.total > 0 && !ws_internal && !resident_here({{ws, w.total}}))
        return RA_ERR_WORKSPACE;

    char *base = static_cast<char *>(ws);
    const bool striped = p.layout == RA_LAYOUT_STRIPED && !p.rank_major;
    const long long row_bytes = (long long)p.d * (long long)p.esz();
    NvtxRange r_call(p.mode == RA_MODE_FUSED ? "ra_forward (fused)"
                     : p.mode == RA_MODE_RING ? "ra_forward (ring)" : "ra_forward (per step)");
    const void *qk = q, *kk = k, *vk = v;
    if (striped) {
        NvtxRange r_perm("ra: permute q, k, v to rank-major");
        ra::launch_permute(q, base + w.q, (long long)p.B * p.H * p.S, p.S, p.N, row_bytes, 0, sm, st);
        ra::launch_permute(k, base + w.k, (long long)p.B * p.Hkv * p.S, p.S, p.N, row_bytes, 0, sm, st);
        ra::launch_permute(v, base + w.v, (long long)p.B * p.Hkv * p.S, p.S, p.N, row_bytes, 0, sm, st);
        count_launch(3);
        if (cudaGetLastError() != cudaSuccess)
            return RA_ERR_CUDA;
        qk = base + w.q, kk = base + w.k, vk = base + w.v;
    }

    if (p.mode == RA_MODE_FUSED && w.nsplit > 1) {
        {
            NvtxRange r_att("ra: attention, all ring steps, walks split into pieces");
            rs = attention_pass(p, qk, kk, vk, base + w.split, (float *)(base + w.split_lse), 0, p.N, true, sm,
                                st, 0, -1, w.nsplit);
        }
        if (rs != RA_OK)
            return rs;
        NvtxRange r_comb("ra: combine the pieces (natural order)");
        ra::launch_combine((const float *)(base + w.split), (const float *)(base + w.split_lse), w.nsplit,
                           (long long)p.rows(), out, lse, 1, (long long)p.rows(), p.S, p.N, striped ? 1 : 0,
                           p.d, sm, st);
        count_launch();
        return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_CUDA;
    }
    if (p.mode == RA_MODE_FUSED) {
        void *ok_out = striped ? (void *)(base + w.out) : out;
        float *ok_lse = striped ? (float *)(base + w.lse) : lse;
        {
            NvtxRange r_att("ra: attention, all ring steps");
            rs = attention_pass(p, qk, kk, vk, ok_out, ok_lse, 0, p.N, p.dtype == RA_DTYPE_F32, sm, st);
        }
        if (rs != RA_OK)
            return rs;
        if (striped) {
            NvtxRange r_unperm("ra: out, lse back to natural order");
            ra::launch_permute(ok_out, out, (long long)p.rows(), p.S, p.N, row_bytes, 1, sm, st);
            ra::launch_permute(ok_lse, lse, (long long)p.rows(), p.S, p.N, 4, 1, sm, st);
            count_launch(2);
            if (cudaGetLastError() != cudaSuccess)
                return RA_ERR_CUDA;
        }
        return RA_OK;
    }

    // per-step and ring: step 0 initialises the running state, later steps
    // are merged
    float *run = (float *)(base + w.run), *run_lse = (float *)(base + w.run_lse);
    float *part = (float *)(base + w.part), *part_lse = (float *)(base + w.part_lse);
    const long long L = p.L();
    const bool ring = p.mode == RA_MODE_RING;
    RingCopies rc;
    if (ring && (rs = rc.begin(p, kk, vk, base, w, st)) != RA_OK)
        return rs;
    for (int s = 0; s < p.N; ++s) {
        char step_name[48];
        snprintf(step_name, sizeof(step_name), "ra: ring step %d", s);
        NvtxRange r_step(step_name);
        const void *ks = kk, *vs = vk;
        if (ring && (rs = rc.before_step(s, &ks, &vs, st)) != RA_OK)
            return rs;
        rs = attention_pass(p, qk, ks, vs, s == 0 ? run : part, s == 0 ? run_lse : part_lse, s, s + 1, true,
                            sm, st);
        if (rs != RA_OK)
            return rs;
        if (s > 0) {
            // contiguous causal: at step s only ranks i >= s hold a visible block
            const long long begin = (p.causal && p.layout == RA_LAYOUT_CONTIGUOUS) ? s * L : 0;
            ra::launch_merge(run, run_lse, part, part_lse, (long long)p.B * p.H, p.S, begin, p.S - begin,
                             p.d, sm, st);
            count_launch();
            if (cudaGetLastError() != cudaSuccess)
                return RA_ERR_CUDA;
        }
        if (ring && (rs = rc.after_step(s, st)) != RA_OK)
            return rs;
    }
    if (ring && (rs = rc.end(st)) != RA_OK)
        return rs;
    NvtxRange r_fin("ra: finalise (divide, natural order)");
    ra::launch_finalize(run, run_lse, out, lse, p.dtype == RA_DTYPE_BF16, (long long)p.rows(), p.S,
                        p.N, striped ? 1 : 0, p.d, sm, st);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_CUDA;
}

ra_status forward_alloc(const Problem &p, const void *q, const void *k, const void *v, void *out,
                        float *lse, cudaStream_t st)
{
    ra_status rs = check_problem(p);
    if (rs != RA_OK)
        return rs;
    if ((rs = check_forward_ptrs(p, q, k, v, out, lse)) != RA_OK)
        return rs;
    if (!forward_resident(p, q, k, v, out, lse))
        return RA_ERR_INVALID_ARG;
    const size_t bytes = ws_layout(p, sm_count_current()).total;
    void *ws = nullptr;
    if (bytes > 0 && cudaMallocAsync(&ws, bytes, st) != cudaSuccess) {
        cudaGetLastError();
        return RA_ERR_NO_MEMORY;
    }
    rs = forward_impl(p, q, k, v, out, lse, ws, bytes, st, true);
    if (ws && cudaFreeAsync(ws, st) != cudaSuccess && rs == RA_OK)
        rs = RA_ERR_CUDA;
    return rs;
}

// Workspace of ra_forward_ulysses: head-sharded q, k, v, out (input dtype)
// and lse (fp32), each 256-byte aligned.
struct UlyssesWs {
    size_t q = 0, k = 0, v = 0, out = 0, lse = 0, total = 0;
};

// Validates the request; on success fills the per-device attention problem
// (all devices' head groups as one batch of n_dev * B) and the workspace.
ra_status ulysses_plan(int B, int H, int Hkv, int S, int d, int n_dev, int causal, int dtype, Problem *pa,
                       UlyssesWs *w)
{
    if (n_dev < 1 || B < 1 || H < 1 || Hkv < 1 || S < 1)
        return RA_ERR_INVALID_ARG;
    if (S % n_dev != 0 || H % Hkv != 0)
        return RA_ERR_INVALID_ARG;
    // every device needs whole kv heads: the head count limits the devices
    if (H % n_dev != 0 || Hkv % n_dev != 0)
        return RA_ERR_UNSUPPORTED;
    *pa = Problem{B * n_dev, H / n_dev, Hkv / n_dev, S, d, 1, RA_LAYOUT_CONTIGUOUS, causal, dtype,
                  RA_MODE_FUSED};
    ra_status rs = check_problem(*pa);
    if (rs != RA_OK)
        return rs;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += align256(bytes);
        return at;
    };
    w->q = take(pa->q_elems() * pa->esz());
    w->k = take(pa->kv_elems() * pa->esz());
    w->v = take(pa->kv_elems() * pa->esz());
    w->out = take(pa->q_elems() * pa->esz());
    w->lse = take(pa->rows() * 4);
    w->total = off;
    return RA_OK;
}

// ------------------------------------------------------------------ backward
// Workspace of the backward pass: delta (fp32 per row); for the striped
// layout also rank-major copies of q, k, v, out, dout, lse and of the
// gradients before they are put back in natural order.
struct BwdWs {
    size_t delta = 0, q = 0, k = 0, v = 0, out = 0, dout = 0, lse = 0, dq = 0, dk = 0, dv = 0, total = 0;
};

BwdWs bwd_ws_layout(const Problem &p)
{
    BwdWs w;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += align256(bytes);
        return at;
    };
    w.delta = take(p.rows() * 4);
    if (p.layout == RA_LAYOUT_STRIPED) {
        const size_t qb = p.q_elems() * p.esz(), kvb = p.kv_elems() * p.esz();
        w.q = take(qb), w.k = take(kvb), w.v = take(kvb), w.out = take(qb), w.dout = take(qb);
        w.lse = take(p.rows() * 4);
        w.dq = take(qb), w.dk = take(kvb), w.dv = take(kvb);
    }
    w.total = off;
    return w;
}

ra_status backward_impl(const Problem &p, const void *q, const void *k, const void *v, const void *out,
                        const float *lse, const void *dout, void *dq, void *dk, void *dv, void *ws,
                        size_t ws_bytes, cudaStream_t st)
{
    ra_status rs = check_problem(p);
    if (rs != RA_OK)
        return rs;
    if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv)
        return RA_ERR_INVALID_ARG;
    const void *all[] = {q, k, v, out, lse, dout, dq, dk, dv};
    for (const void *x : all)
        if (!aligned16(x))
            return RA_ERR_INVALID_ARG;
    const size_t qb = p.q_elems() * p.esz(), kvb = p.kv_elems() * p.esz(), lb = p.rows() * 4;
    const size_t sizes[] = {qb, kvb, kvb, qb, lb, qb, qb, kvb, kvb};
    // the three gradients must not overlap any input or each other
    for (int o = 6; o < 9; ++o)
        for (int x = 0; x < 9; ++x)
            if (x != o && overlaps(all[o], sizes[o], all[x], sizes[x]))
                return RA_ERR_INVALID_ARG;
    const BwdWs w = bwd_ws_layout(p);
    if (!ws || ws_bytes < w.total || (reinterpret_cast<uintptr_t>(ws) & 255u))
        return RA_ERR_WORKSPACE;
    if (!resident_here({{q, qb}, {k, kvb}, {v, kvb}, {out, qb}, {lse, lb}, {dout, qb}, {dq, qb}, {dk, kvb},
                        {dv, kvb}}))
        return RA_ERR_INVALID_ARG;
    if (!resident_here({{ws, w.total}}))
        return RA_ERR_WORKSPACE;
    const int sm = sm_count_current();
    char *base = static_cast<char *>(ws);
    const bool striped = p.layout == RA_LAYOUT_STRIPED;
    const long long row = (long long)p.d * (long long)p.esz();
    const long long qrows = (long long)p.B * p.H * p.S, kvrows = (long long)p.B * p.Hkv * p.S;
    NvtxRange r_call("ra_backward");
    ra::BwdLaunch a{};
    a.q = q, a.k = k, a.v = v, a.out = out, a.dout = dout, a.lse = lse;
    a.dq = dq, a.dk = dk, a.dv = dv;
    if (striped) {
        ra::launch_permute(q, base + w.q, qrows, p.S, p.N, row, 0, sm, st);
        ra::launch_permute(k, base + w.k, kvrows, p.S, p.N, row, 0, sm, st);
        ra::launch_permute(v, base + w.v, kvrows, p.S, p.N, row, 0, sm, st);
        ra::launch_permute(out, base + w.out, qrows, p.S, p.N, row, 0, sm, st);
        ra::launch_permute(dout, base + w.dout, qrows, p.S, p.N, row, 0, sm, st);
        ra::launch_permute(lse, base + w.lse, qrows, p.S, p.N, 4, 0, sm, st);
        count_launch(6);
        if (cudaGetLastError() != cudaSuccess)
            return RA_ERR_CUDA;
        a.q = base + w.q, a.k = base + w.k, a.v = base + w.v, a.out = base + w.out, a.dout = base + w.dout;
        a.lse = (const float *)(base + w.lse);
        a.dq = base + w.dq, a.dk = base + w.dk, a.dv = base + w.dv;
    }
    a.delta = (float *)(base + w.delta);
    a.B = p.B, a.H = p.H, a.Hkv = p.Hkv, a.S = p.S, a.d = p.d, a.N = p.N;
    a.layout = p.layout, a.causal = p.causal;
    a.timeout_ns = g_timeout_ns;
    count_launch(3);
    if (p.dtype == RA_DTYPE_F32)
        ra::launch_bwd_f32(a, st);
    else if (ra::launch_bwd(a, st) != cudaSuccess)
        return RA_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess)
        return RA_ERR_CUDA;
    if (striped) {
        ra::launch_permute(base + w.dq, dq, qrows, p.S, p.N, row, 1, sm, st);
        ra::launch_permute(base + w.dk, dk, kvrows, p.S, p.N, row, 1, sm, st);
        ra::launch_permute(base + w.dv, dv, kvrows, p.S, p.N, row, 1, sm, st);
        count_launch(3);
    }
    return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_CUDA;
}

}  // namespace

extern "C" {

ra_status ra_forward(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H,
                     int Hkv, int S, int d, int n_blocks, int layout, int causal, ra_stream_t stream)
{
    const Problem p{B, H, Hkv, S, d, n_blocks, layout, causal, RA_DTYPE_BF16, RA_MODE_FUSED};
    return forward_alloc(p, q, k, v, out, lse, (cudaStream_t)stream);
}

ra_status ra_forward_f32(const float *q, const float *k, const float *v, float *out, float *lse, int B,
                         int H, int Hkv, int S, int d, int n_blocks, int layout, int causal,
                         ra_stream_t stream)
{
    const Problem p{B, H, Hkv, S, d, n_blocks, layout, causal, RA_DTYPE_F32, RA_MODE_FUSED};
    return forward_alloc(p, q, k, v, out, lse, (cudaStream_t)stream);
}

size_t ra_workspace_bytes(int B, int H, int Hkv, int S, int d, int n_blocks, int layout, int causal,
                          int mode, int dtype)
{
    const Problem p{B, H, Hkv, S, d, n_blocks, layout, causal, dtype, mode};
    if (check_problem(p) != RA_OK)
        return 0;
    return ws_layout(p, sm_count_current()).total;
}

ra_status ra_forward_ws(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H,
                        int Hkv, int S, int d, int n_blocks, int layout, int causal, int dtype, int mode,
                        void *ws, size_t ws_bytes, ra_stream_t stream)
{
    const Problem p{B, H, Hkv, S, d, n_blocks, layout, causal, dtype, mode};
    return forward_impl(p, q, k, v, out, lse, ws, ws_bytes, (cudaStream_t)stream);
}

ra_status ra_forward_rank_major(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                                int H, int Hkv, int S, int d, int n_blocks, int layout, int causal, int dtype,
                                int mode, void *ws, size_t ws_bytes, ra_stream_t stream)
{
    Problem p{B, H, Hkv, S, d, n_blocks, layout, causal, dtype, mode};
    p.rank_major = true;
    return forward_impl(p, q, k, v, out, lse, ws, ws_bytes, (cudaStream_t)stream);
}

ra_status ra_forward_block(const void *q, const void *k, const void *v, float *out_s, float *lse_s, int B,
                           int H, int Hkv, int S, int d, int n_blocks, int layout, int causal, int dtype,
                           int rank, int step, ra_stream_t stream)
{
    const Problem p{B, H, Hkv, S, d, n_blocks, layout, causal, dtype, RA_MODE_PER_STEP};
    ra_status rs = check_problem(p);
    if (rs != RA_OK)
        return rs;
    if (rank < 0 || rank >= n_blocks || step < 0 || step >= n_blocks)
        return RA_ERR_INVALID_ARG;
    if (!q || !k || !v || !out_s || !lse_s)
        return RA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out_s) || !aligned16(lse_s))
        return RA_ERR_INVALID_ARG;
    const size_t qb = p.q_elems() * p.esz(), kvb = p.kv_elems() * p.esz();
    const size_t ob = p.q_elems() * 4, lb = p.rows() * 4;
    for (const void *in : {q, k, v})
        if (overlaps(out_s, ob, in, in == q ? qb : kvb) || overlaps(lse_s, lb, in, in == q ? qb : kvb))
            return RA_ERR_INVALID_ARG;
    if (overlaps(out_s, ob, lse_s, lb))
        return RA_ERR_INVALID_ARG;
    if (!resident_here({{q, qb}, {k, kvb}, {v, kvb}, {out_s, ob}, {lse_s, lb}}))
        return RA_ERR_INVALID_ARG;
    const int sm = sm_count_current();
    cudaStream_t st = (cudaStream_t)stream;
    const int j = ra_ring_block(rank, step, n_blocks);
    if (ra_block_class(layout, causal, rank, j) == RA_CLS_SKIP) {
        ra::launch_fill_empty(out_s, lse_s, (long long)B * H, S, (long long)rank * p.L(), p.L(), d, sm, st);
        count_launch();
        return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_CUDA;
    }
    return attention_pass(p, q, k, v, out_s, lse_s, step, step + 1, true, sm, st, rank, rank + 1);
}

ra_status ra_all_to_all(const void *src, void *dst, int B, int Hn, int S, int d, int elem_bytes, int n_dev,
                        int inverse, ra_stream_t stream)
{
    if (!src || !dst || B < 1 || Hn < 1 || S < 1 || d < 1 || n_dev < 1 || S % n_dev != 0 || Hn % n_dev != 0)
        return RA_ERR_INVALID_ARG;
    if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8)
        return RA_ERR_INVALID_ARG;
    if (inverse != 0 && inverse != 1)
        return RA_ERR_INVALID_ARG;
    if ((long long)B * Hn * S >= (1ll << 40))
        return RA_ERR_UNSUPPORTED;
    const long long row_bytes = (long long)d * elem_bytes;
    const size_t total = (size_t)B * Hn * S * row_bytes;
    if (overlaps(src, total, dst, total))
        return RA_ERR_INVALID_ARG;
    const uintptr_t mis = (reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst));
    if ((row_bytes % 16 == 0 && (mis & 15u)) || (row_bytes % 4 == 0 && (mis & 3u)))
        return RA_ERR_INVALID_ARG;
    if (!resident_here({{src, total}, {dst, total}}))
        return RA_ERR_INVALID_ARG;
    ra::launch_all_to_all(src, dst, B, Hn, S, n_dev, row_bytes, inverse, sm_count_current(),
                          (cudaStream_t)stream);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_CUDA;
}


size_t ra_ulysses_workspace_bytes(int B, int H, int Hkv, int S, int d, int n_dev, int causal, int dtype)
{
    Problem pa{};
    UlyssesWs w;
    return ulysses_plan(B, H, Hkv, S, d, n_dev, causal, dtype, &pa, &w) == RA_OK ? w.total : 0;
}

ra_status ra_forward_ulysses(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H,
                             int Hkv, int S, int d, int n_dev, int causal, int dtype, void *ws, size_t ws_bytes,
                             ra_stream_t stream)
{
    Problem pa{};
    UlyssesWs w;
    ra_status rs = ulysses_plan(B, H, Hkv, S, d, n_dev, causal, dtype, &pa, &w);
    if (rs != RA_OK)
        return rs;
    if (!q || !k || !v || !out || !lse)
        return RA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
        return RA_ERR_INVALID_ARG;
    const size_t qb = pa.q_elems() * pa.esz(), kvb = pa.kv_elems() * pa.esz(), lb = pa.rows() * 4;
    for (const void *in : {q, k, v})
        if (overlaps(out, qb, in, in == q ? qb : kvb) || overlaps(lse, lb, in, in == q ? qb : kvb))
            return RA_ERR_INVALID_ARG;
    if (overlaps(out, qb, lse, lb))
        return RA_ERR_INVALID_ARG;
    if (!ws || ws_bytes < w.total || (reinterpret_cast<uintptr_t>(ws) & 255u))
        return RA_ERR_WORKSPACE;
    if (!resident_here({{q, qb}, {k, kvb}, {v, kvb}, {out, qb}, {lse, lb}}))
        return RA_ERR_INVALID_ARG;
    if (!resident_here({{ws, w.total}}))
        return RA_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    const int sm = sm_count_current();
    char *base = static_cast<char *>(ws);
    const long long row = (long long)d * pa.esz();
    NvtxRange r_call("ra_forward_ulysses");
    // all-to-all in: every device gets all tokens of its heads
    ra::launch_all_to_all(q, base + w.q, B, H, S, n_dev, row, 0, sm, st);
    ra::launch_all_to_all(k, base + w.k, B, Hkv, S, n_dev, row, 0, sm, st);
    ra::launch_all_to_all(v, base + w.v, B, Hkv, S, n_dev, row, 0, sm, st);
    count_launch(3);
    if (cudaGetLastError() != cudaSuccess)
        return RA_ERR_CUDA;
    // each device: exact attention over the whole sequence for its heads
    rs = attention_pass(pa, base + w.q, base + w.k, base + w.v, base + w.out, (float *)(base + w.lse), 0, 1,
                        dtype == RA_DTYPE_F32, sm, st);
    if (rs != RA_OK)
        return rs;
    // all-to-all out: back to the sequence shards
    ra::launch_all_to_all(base + w.out, out, B, H, S, n_dev, row, 1, sm, st);
    ra::launch_all_to_all(base + w.lse, lse, B, H, S, n_dev, 4, 1, sm, st);
    count_launch(2);
    return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_CUDA;
}

long long ra_backward_tile_pairs(int B, int H, int Hkv, int S, int n_blocks, int layout, int causal, int which,
                                 int *pairs, long long capacity)
{
    const Problem p{B, H, Hkv, S, 64, n_blocks, layout, causal, RA_DTYPE_BF16, RA_MODE_FUSED};
    if (check_problem(p) != RA_OK || (which != 0 && which != 1))
        return -1;
    const int L = S / n_blocks, ntiles = (L + RA_TILE - 1) / RA_TILE, grp = H / Hkv;
    const long long units = (long long)(which == 0 ? B * Hkv : B * H) * n_blocks * ntiles;
    long long n = 0;
    auto put = [&](long long u, int bh, int i, int ta, int j, int tb, long long k) {
        if (pairs && n < capacity) {
            int *o = pairs + 8 * n;
            o[0] = (int)u, o[1] = bh, o[2] = i, o[3] = ta, o[4] = j, o[5] = tb, o[6] = (int)k, o[7] = 0;
        }
        ++n;
    };
    for (long long u = 0; u < units; ++u) {
        long long k = 0;
        if (which == 0) {
            int bhkv, j, tb;
            ra_bwd_dkdv_unit((int)u, B, Hkv, n_blocks, ntiles, layout, ra_bwd_kv_outer(B, Hkv, S), bhkv, j, tb);
            const int b = bhkv / Hkv, g = bhkv % Hkv;
            RaQWalk w;
            for (w.start(j, tb, n_blocks, layout, causal, ntiles, grp); w.valid(); w.advance())
                put(u, b * H + g * grp + w.hh, w.i, w.ta, j, tb, k++);
        } else {
            int bh, i, ta;
            ra_bwd_dq_unit((int)u, B, H, Hkv, n_blocks, ntiles, layout, ra_bwd_kv_outer(B, Hkv, S), bh, i, ta);
            RaKWalk w;
            for (w.start(i, ta, n_blocks, layout, causal, ntiles); w.valid(); w.advance())
                put(u, bh, i, ta, w.j, w.tb, k++);
        }
    }
    return n;
}

size_t ra_backward_workspace_bytes(int B, int H, int Hkv, int S, int d, int n_blocks, int layout, int causal)
{
    const Problem p{B, H, Hkv, S, d, n_blocks, layout, causal, RA_DTYPE_BF16, RA_MODE_FUSED};
    if (check_problem(p) != RA_OK)
        return 0;
    return bwd_ws_layout(p).total;
}

ra_status ra_backward_ws(const void *q, const void *k, const void *v, const void *out, const float *lse,
                         const void *dout, void *dq, void *dk, void *dv, int B, int H, int Hkv, int S, int d,
                         int n_blocks, int layout, int causal, void *ws, size_t ws_bytes, ra_stream_t stream)
{
    const Problem p{B, H, Hkv, S, d, n_blocks, layout, causal, RA_DTYPE_BF16, RA_MODE_FUSED};
    return backward_impl(p, q, k, v, out, lse, dout, dq, dk, dv, ws, ws_bytes, (cudaStream_t)stream);
}

namespace {
ra_status backward_alloc(const Problem &p, const void *q, const void *k, const void *v, const void *out,
                         const float *lse, const void *dout, void *dq, void *dk, void *dv, cudaStream_t st)
{
    ra_status rs = check_problem(p);
    if (rs != RA_OK)
        return rs;
    const size_t bytes = bwd_ws_layout(p).total;
    void *ws = nullptr;
    if (cudaMallocAsync(&ws, bytes, st) != cudaSuccess) {
        cudaGetLastError();
        return RA_ERR_NO_MEMORY;
    }
    rs = backward_impl(p, q, k, v, out, lse, dout, dq, dk, dv, ws, bytes, st);
    if (cudaFreeAsync(ws, st) != cudaSuccess && rs == RA_OK)
        rs = RA_ERR_CUDA;
    return rs;
}
}  // namespace

ra_status ra_backward_f32(const float *q, const float *k, const float *v, const float *out, const float *lse,
                          const float *dout, float *dq, float *dk, float *dv, int B, int H, int Hkv, int S, int d,
                          int n_blocks, int layout, int causal, ra_stream_t stream)
{
    const Problem p{B, H, Hkv, S, d, n_blocks, layout, causal, RA_DTYPE_F32, RA_MODE_FUSED};
    return backward_alloc(p, q, k, v, out, lse, dout, dq, dk, dv, (cudaStream_t)stream);
}

ra_status ra_backward(const void *q, const void *k, const void *v, const void *out, const float *lse,
                      const void *dout, void *dq, void *dk, void *dv, int B, int H, int Hkv, int S, int d,
                      int n_blocks, int layout, int causal, ra_stream_t stream)
{
    const Problem p{B, H, Hkv, S, d, n_blocks, layout, causal, RA_DTYPE_BF16, RA_MODE_FUSED};
    ra_status rs = check_problem(p);
    if (rs != RA_OK)
        return rs;
    cudaStream_t st = (cudaStream_t)stream;
    const size_t bytes = bwd_ws_layout(p).total;
    void *ws = nullptr;
    if (cudaMallocAsync(&ws, bytes, st) != cudaSuccess) {
        cudaGetLastError();
        return RA_ERR_NO_MEMORY;
    }
    rs = backward_impl(p, q, k, v, out, lse, dout, dq, dk, dv, ws, bytes, st);
    if (cudaFreeAsync(ws, st) != cudaSuccess && rs == RA_OK)
        rs = RA_ERR_CUDA;
    return rs;
}

unsigned long long ra_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int ra_set_kernel_variant(int variant)
{
    if (variant < 0 || variant > 3 || variant == 2)
        return -1;
    return g_kernel_variant.exchange(variant);
}

void ra_set_wait_timeout_ns(unsigned long long timeout_ns)
{
    g_timeout_ns = timeout_ns ? timeout_ns : kDefaultTimeoutNs;
}

ra_status ra_wait_probe(unsigned long long timeout_ns, ra_stream_t stream)
{
    if (timeout_ns < 1000000ull || timeout_ns > 10000000000ull)
        return RA_ERR_INVALID_ARG;
    count_launch();
    return ra::launch_wait_probe(timeout_ns, (cudaStream_t)stream) == cudaSuccess ? RA_OK : RA_ERR_CUDA;
}

ra_status ra_permute(const void *src, void *dst, int B, int Hn, int S, int d, int elem_bytes, int n_blocks,
                     int inverse, ra_stream_t stream)
{
    if (!src || !dst || B < 1 || Hn < 1 || S < 1 || d < 1 || n_blocks < 1 || S % n_blocks != 0)
        return RA_ERR_INVALID_ARG;
    if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8)
        return RA_ERR_INVALID_ARG;
    if (inverse != 0 && inverse != 1)
        return RA_ERR_INVALID_ARG;
    const long long row_bytes = (long long)d * elem_bytes;
    const size_t total = (size_t)B * Hn * S * row_bytes;
    if (overlaps(src, total, dst, total))
        return RA_ERR_INVALID_ARG;
    const uintptr_t mis = (reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst));
    // vector width is chosen from the row size; pointers must match it
    if ((row_bytes % 16 == 0 && (mis & 15u)) || (row_bytes % 4 == 0 && (mis & 3u)))
        return RA_ERR_INVALID_ARG;
    if (!resident_here({{src, total}, {dst, total}}))
        return RA_ERR_INVALID_ARG;
    ra::launch_permute(src, dst, (long long)B * Hn * S, S, n_blocks, row_bytes, inverse,
                       sm_count_current(), (cudaStream_t)stream);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_CUDA;
}

ra_status ra_merge(float *out_run, float *lse_run, const float *out_s, const float *lse_s, long long rows,
                   int d, ra_stream_t stream)
{
    if (!out_run || !lse_run || !out_s || !lse_s || rows < 1 || d < 4 || d > 256 || d % 4 != 0)
        return RA_ERR_INVALID_ARG;
    if (!aligned16(out_run) || !aligned16(out_s) || ((reinterpret_cast<uintptr_t>(lse_run) |
                                                      reinterpret_cast<uintptr_t>(lse_s)) & 3u))
        return RA_ERR_INVALID_ARG;
    const size_t ob = (size_t)rows * d * 4, lb = (size_t)rows * 4;
    if (overlaps(out_run, ob, out_s, ob) || overlaps(lse_run, lb, lse_s, lb) ||
        overlaps(out_run, ob, lse_run, lb) || overlaps(out_run, ob, lse_s, lb) ||
        overlaps(lse_run, lb, out_s, ob))
        return RA_ERR_INVALID_ARG;
    if (!resident_here({{out_run, ob}, {lse_run, lb}, {out_s, ob}, {lse_s, lb}}))
        return RA_ERR_INVALID_ARG;
    ra::launch_merge(out_run, lse_run, out_s, lse_s, 1, rows, 0, rows, d, sm_count_current(),
                     (cudaStream_t)stream);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_CUDA;
}

ra_status ra_check(ra_stream_t stream)
{
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess)
        return RA_ERR_CUDA;
    unsigned int st = 0;
    if (ra::read_and_clear_device_status(&st) != cudaSuccess)
        return RA_ERR_CUDA;
    if (st == 0)
        return RA_OK;
    return (st & 0xffu) == ra::RA_DEV_TIMEOUT_CODE ? RA_ERR_TIMEOUT : RA_ERR_CUDA;
}

const char *ra_status_string(int status)
{
    switch (status) {
    case RA_OK: return "RA_OK";
    case RA_ERR_INVALID_ARG: return "RA_ERR_INVALID_ARG";
    case RA_ERR_UNSUPPORTED: return "RA_ERR_UNSUPPORTED";
    case RA_ERR_CUDA: return "RA_ERR_CUDA";
    case RA_ERR_NO_MEMORY: return "RA_ERR_NO_MEMORY";
    case RA_ERR_TIMEOUT: return "RA_ERR_TIMEOUT";
    case RA_ERR_WORKSPACE: return "RA_ERR_WORKSPACE";
    case RA_ERR_SCRATCH_LIMIT: return "RA_ERR_SCRATCH_LIMIT";
    default: return "RA_ERR_UNKNOWN";
    }
}

const char *ra_version(void) { return "ra 0.1.0 sm_103a"; }

long long ra_schedule_units(int B, int H, int Hkv, int S, int n_blocks, int layout, int causal,
                            int s_begin, int s_end, int *units, long long capacity)
{
    const Problem p{B, H, Hkv, S, 64, n_blocks, layout, causal, RA_DTYPE_BF16, RA_MODE_FUSED};
    if (check_problem(p) != RA_OK || s_begin < 0 || s_end > n_blocks || s_begin >= s_end ||
        (!(s_begin == 0 && s_end == n_blocks) && s_end != s_begin + 1))
        return -1;
    const RaUnitSpace sp = ra_unit_space(B, H, Hkv, S, n_blocks, layout, causal, s_begin, s_end);
    const long long n = ra_unit_count(sp);
    for (long long u = 0; units && u < n && u < capacity; ++u) {
        const RaUnit U = ra_unit_decode(sp, u);
        int *o = units + 8 * u;
        o[0] = U.bh0, o[1] = U.ta0, o[2] = U.bh1, o[3] = U.ta1;
        o[4] = U.rank, o[5] = U.cost, o[6] = U.tile1_valid, o[7] = 0;
    }
    return n;
}

long long ra_schedule_block_units(int B, int H, int Hkv, int S, int n_blocks, int layout, int causal, int rank,
                                  int step, int *units, long long capacity)
{
    const Problem p{B, H, Hkv, S, 64, n_blocks, layout, causal, RA_DTYPE_BF16, RA_MODE_PER_STEP};
    if (check_problem(p) != RA_OK || rank < 0 || rank >= n_blocks || step < 0 || step >= n_blocks)
        return -1;
    const RaUnitSpace sp = ra_unit_space_ranks(
        ra_unit_space(B, H, Hkv, S, n_blocks, layout, causal, step, step + 1), rank, rank + 1);
    const long long n = ra_unit_count(sp);
    for (long long u = 0; units && u < n && u < capacity; ++u) {
        const RaUnit U = ra_unit_decode(sp, u);
        int *o = units + 8 * u;
        o[0] = U.bh0, o[1] = U.ta0, o[2] = U.bh1, o[3] = U.ta1;
        o[4] = U.rank, o[5] = U.cost, o[6] = U.tile1_valid, o[7] = 0;
    }
    return n;
}

long long ra_schedule_stats(int layout, int causal, int n_blocks, int L, long long *pairs, long long *tiles)
{
    if (n_blocks < 1 || L < 1 || (layout != 0 && layout != 1) || (causal != 0 && causal != 1))
        return -1;
    const int ntiles = (L + RA_TILE - 1) / RA_TILE;
    long long total = 0;
    for (int i = 0; i < n_blocks; ++i)
        for (int s = 0; s < n_blocks; ++s) {
            const int cls = ra_block_class(layout, causal, i, ra_ring_block(i, s, n_blocks));
            long long np = 0, nt = 0;
            for (int a = 0; a < L; ++a)
                np += ra_key_limit(cls, a, L);
            for (int ta = 0; ta < ntiles; ++ta)
                nt += ra_kv_tiles(cls, ta, ntiles);
            if (pairs)
                pairs[i * n_blocks + s] = np;
            if (tiles)
                tiles[i * n_blocks + s] = nt;
            total += np;
        }
    return total;
}

}  // extern "C"

// ------------------------------------------------------------------ no-alloc variant
// ra_forward for callers that cannot allocate device memory (see include/ra.h):
// all scratch lives in one fixed device array that is part of the library's
// image, so nothing is allocated per call or per shape.
static __device__ __align__(256) unsigned char g_noalloc_scratch[RA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device with that device current.  In host code the array's name is only
// a host-side stand-in, never a device address.
ra_status noalloc_scratch(void **ptr)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return RA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return RA_ERR_CUDA;
        }
        g_noalloc_ptr[dev] = p;
    }
    *ptr = g_noalloc_ptr[dev];
    return RA_OK;
}

}  // namespace

extern "C" ra_status ra_forward_noalloc(const void *q, const void *k, const void *v, void *out, float *lse,
                                        int B, int H, int Hkv, int S, int d, int n_blocks, int layout,
                                        int causal, ra_stream_t stream)
{
    const Problem p{B, H, Hkv, S, d, n_blocks, layout, causal, RA_DTYPE_BF16, RA_MODE_FUSED};
    ra_status rs = check_problem(p);
    if (rs != RA_OK)
        return rs;
    if ((rs = check_forward_ptrs(p, q, k, v, out, lse)) != RA_OK)
        return rs;
    // the workspace ra_forward would allocate, taken from the fixed array
    const size_t need = ws_layout(p, sm_count_current()).total;
    if (need > RA_NOALLOC_SCRATCH_BYTES)
        return RA_ERR_SCRATCH_LIMIT;
    if (!forward_resident(p, q, k, v, out, lse))
        return RA_ERR_INVALID_ARG;
    void *scratch = nullptr;
    if (need > 0 && (rs = noalloc_scratch(&scratch)) != RA_OK)
        return rs;
    // the same enqueue as ra_forward, on the library's array
    return forward_impl(p, q, k, v, out, lse, scratch, need, (cudaStream_t)stream, true, true);
}
