// SIMT kernels of the ring-attention library:
//   * ra_attn_f32_kernel  exact fp32 ring-ordered attention (no tensor cores)
//   * ra_permute_kernel   natural <-> striped token order, bit-exact copy (and a
//                         32-bit-index variant with division by invariant integers)
//   * ra_all_to_all_kernel sequence-sharded <-> head-sharded relayout (Ulysses)
//   * ra_merge_kernel     running-softmax merge of one ring step's partials
//   * ra_finalize_kernel  fp32 running result -> output dtype, natural order
//   * ra_combine_kernel   the pieces of a split ring walk -> output, natural order
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ra_internal.h"
#include "ra_schedule.h"

namespace ra {

// ---------------------------------------------------------------- fp32 path
// One warp per query row.  The warp walks the ring steps s in [s_begin,
// s_end): key block j = (i - s) mod N, visible keys b < ra_key_limit(...),
// and keeps the running max m, the running sum l of exp(score - m) and the
// running weighted values, rescaled whenever m grows ("Ring Attention" page,
// section "Halka Dikkati Nasil Calisir": running softmax of flash attention,
// divided at the end).  Lane c owns columns c, c + 32, ...
constexpr int F32_WARPS = 8;
constexpr int F32_MAXW = 8;  // d <= 256

__global__ void __launch_bounds__(F32_WARPS * 32)
ra_attn_f32_kernel(const float *__restrict__ q, const float *__restrict__ k,
                   const float *__restrict__ v, float *__restrict__ out,
                   float *__restrict__ lse, int H, int Hkv, int S, int d, int L, int N,
                   int layout, int causal, int s_begin, int s_end, int rank_lo, float scale)
{
    const int lane = threadIdx.x & 31;
    const int a = blockIdx.x * F32_WARPS + (threadIdx.x >> 5);
    const int i = rank_lo + (int)blockIdx.y;
    const long long bh = blockIdx.z;
    if (a >= L)
        return;
    const long long b = bh / H;
    const int h = (int)(bh % H);
    const long long bhkv = b * Hkv + h / (H / Hkv);
    const long long qrow = bh * S + (long long)i * L + a;
    const int nw = (d + 31) / 32;

    float qv[F32_MAXW], acc[F32_MAXW];
#pragma unroll
    for (int w = 0; w < F32_MAXW; ++w) {
        const int c = lane + 32 * w;
        qv[w] = (w < nw && c < d) ? q[qrow * d + c] * scale : 0.f;
        acc[w] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    for (int s = s_begin; s < s_end; ++s) {
        const int j = ra_ring_block(i, s, N);
        const int cls = ra_block_class(layout, causal, i, j);
        if (cls == RA_CLS_SKIP)
            continue;
        const int lim = ra_key_limit(cls, a, L);
        const float *kb = k + (bhkv * S + (long long)j * L) * d;
        const float *vb = v + (bhkv * S + (long long)j * L) * d;
        for (int u = 0; u < lim; ++u) {
            float part = 0.f;
#pragma unroll
            for (int w = 0; w < F32_MAXW; ++w) {
                const int c = lane + 32 * w;
                if (w < nw && c < d)
                    part = fmaf(qv[w], kb[(long long)u * d + c], part);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                part += __shfl_xor_sync(0xffffffffu, part, off);
            const float sc = __shfl_sync(0xffffffffu, part, 0);
            const float m_new = fmaxf(m, sc);
            const float corr = expf(m - m_new);  // m = -inf -> 0
            const float p = expf(sc - m_new);
            l = fmaf(l, corr, p);
#pragma unroll
            for (int w = 0; w < F32_MAXW; ++w) {
                const int c = lane + 32 * w;
                if (w < nw && c < d)
                    acc[w] = fmaf(acc[w], corr, p * vb[(long long)u * d + c]);
            }
            m = m_new;
        }
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int w = 0; w < F32_MAXW; ++w) {
        const int c = lane + 32 * w;
        if (w < nw && c < d)
            out[qrow * d + c] = acc[w] * inv;
    }
    if (lane == 0)
        lse[qrow] = l > 0.f ? m + logf(l) : -INFINITY;
}

void launch_attn_f32(const float *q, const float *k, const float *v, float *out, float *lse,
                     int B, int H, int Hkv, int S, int d, int N, int layout, int causal,
                     int s_begin, int s_end, int rank_lo, int rank_hi, cudaStream_t st)
{
    const int L = S / N;
    if (rank_hi <= rank_lo)
        return;
    dim3 grid((L + F32_WARPS - 1) / F32_WARPS, rank_hi - rank_lo, B * H);
    ra_attn_f32_kernel<<<grid, F32_WARPS * 32, 0, st>>>(
        q, k, v, out, lse, H, Hkv, S, d, L, N, layout, causal, s_begin, s_end, rank_lo,
        1.0f / sqrtf((float)d));
}

// ---------------------------------------------------------------- empty rows
// A partial over no visible key: O = 0 and lse = -inf, the neutral element of
// the merge.  One thread per 16-byte word of out (d % 4 == 0) or per float.
__global__ void ra_fill_empty_kernel(float *__restrict__ out, float *__restrict__ lse, long long BH,
                                     int S, long long row0, long long nrows, int d)
{
    const long long words = (long long)d / 4;
    const long long total = BH * nrows * words;
    for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < total;
         x += (long long)gridDim.x * blockDim.x) {
        const long long w = x % words, rr = x / words;
        const long long row = (rr / nrows) * S + row0 + rr % nrows;
        reinterpret_cast<float4 *>(out + row * d)[w] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (w == 0)
            lse[row] = -INFINITY;
    }
}

void launch_fill_empty(float *out, float *lse, long long BH, int S, long long row0, long long nrows,
                       int d, int sm_count, cudaStream_t st)
{
    const long long total = BH * nrows * (d / 4);
    if (total <= 0)
        return;
    const long long want = (total + 255) / 256;
    const int grid = (int)(want < 8ll * sm_count ? want : 8ll * sm_count);
    ra_fill_empty_kernel<<<grid, 256, 0, st>>>(out, lse, BH, S, row0, nrows, d);
}

// ---------------------------------------------------------------- index helpers
// Division of n < 2^31 by an invariant d as a multiply-high and shift
// (Granlund and Montgomery, "Division by Invariant Integers using
// Multiplication", PLDI 1994, Theorem 4.2 with N = 31): with l = ceil(log2 d)
// and m = ceil(2^(31 + l) / d), which fits in 32 bits, n / d = (n m) >> (31 + l).
struct FastDiv {
    uint32_t d, m, s;
};

FastDiv make_fastdiv(uint32_t d)
{
    uint32_t l = 0;
    while ((1ull << l) < d)
        ++l;
    const uint32_t s = 31 + l;
    const uint64_t m = ((1ull << s) + d - 1) / d;
    return FastDiv{d, (uint32_t)m, s};
}

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv &f)
{
    return (uint32_t)(((uint64_t)n * f.m) >> f.s);
}

// ---------------------------------------------------------------- permute
// Striped row p = r L + a holds natural token t = a N + r.  Each thread moves
// VEC-byte words; the grid walks destination rows, so writes are contiguous
// and each source row is read whole.  Every thread keeps UNROLL independent
// loads in flight before it stores, which HBM needs to reach its bandwidth.
template <typename VEC, int UNROLL>
__global__ void ra_permute_kernel(const VEC *__restrict__ src, VEC *__restrict__ dst,
                                  long long n_rows_total, int S, int L, int N,
                                  int words_per_row, int inverse)
{
    const long long n = n_rows_total * words_per_row;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long base = blockIdx.x * (long long)blockDim.x + threadIdx.x; base < n;
         base += stride * UNROLL) {
        VEC v[UNROLL];
        long long at[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const long long idx = base + u * stride;
            at[u] = idx;
            if (idx < n) {
                const long long row = idx / words_per_row;
                const int w = (int)(idx - row * words_per_row);
                const long long bh = row / S;
                const int x = (int)(row - bh * S);
                // forward: x is the striped row p, read natural t(p)
                // inverse: x is the natural token t, read striped p(t)
                const int other = !inverse ? (x % L) * N + x / L : (x % N) * L + x / N;
                v[u] = src[(bh * S + other) * words_per_row + w];
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u)
            if (at[u] < n)
                dst[at[u]] = v[u];
    }
}

// The permutation with 32-bit index arithmetic (every word index < 2^31).
template <typename VEC, int UNROLL>
__global__ void ra_permute32_kernel(const VEC *__restrict__ src, VEC *__restrict__ dst, uint32_t n_words,
                                    FastDiv wpr, FastDiv S, FastDiv L, FastDiv N, int inverse)
{
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t base = blockIdx.x * blockDim.x + threadIdx.x; base < n_words; base += stride * UNROLL) {
        VEC v[UNROLL];
        uint32_t at[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const uint32_t idx = base + u * stride;
            at[u] = idx;
            if (idx < n_words) {
                const uint32_t row = fdiv(idx, wpr);
                const uint32_t w = idx - row * wpr.d;
                const uint32_t bh = fdiv(row, S);
                const uint32_t x = row - bh * S.d;
                // forward: x is the striped row p, read natural t(p)
                // inverse: x is the natural token t, read striped p(t)
                uint32_t other;
                if (!inverse) {
                    const uint32_t r = fdiv(x, L);
                    other = (x - r * L.d) * N.d + r;
                } else {
                    const uint32_t a = fdiv(x, N);
                    other = (x - a * N.d) * L.d + a;
                }
                v[u] = src[(size_t)(bh * S.d + other) * wpr.d + w];
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u)
            if (at[u] < n_words)
                dst[at[u]] = v[u];
    }
}

void launch_permute(const void *src, void *dst, long long rows_total, int S, int N,
                    long long row_bytes, int inverse, int sm_count, cudaStream_t st)
{
    const int L = S / N;
    const int threads = 256;
    auto grid_for = [&](long long n) {
        long long g = (n + threads - 1) / threads;
        const long long cap = (long long)sm_count * 8;
        return (int)(g < cap ? (g > 0 ? g : 1) : cap);
    };
    const long long vec = row_bytes % 16 == 0 ? 16 : (row_bytes % 4 == 0 ? 4 : 1);
    const long long words = rows_total * (row_bytes / vec);
    // 32-bit path: every word index (and the grid-stride sum) below 2^31
    if (words + 4ll * 8 * sm_count * threads < (1ll << 31)) {
        const FastDiv fw = make_fastdiv((uint32_t)(row_bytes / vec)), fS = make_fastdiv((uint32_t)S),
                      fL = make_fastdiv((uint32_t)L), fN = make_fastdiv((uint32_t)N);
        if (vec == 16)
            ra_permute32_kernel<uint4, 4><<<grid_for(words), threads, 0, st>>>(
                (const uint4 *)src, (uint4 *)dst, (uint32_t)words, fw, fS, fL, fN, inverse);
        else if (vec == 4)
            ra_permute32_kernel<uint32_t, 4><<<grid_for(words), threads, 0, st>>>(
                (const uint32_t *)src, (uint32_t *)dst, (uint32_t)words, fw, fS, fL, fN, inverse);
        else
            ra_permute32_kernel<uint8_t, 4><<<grid_for(words), threads, 0, st>>>(
                (const uint8_t *)src, (uint8_t *)dst, (uint32_t)words, fw, fS, fL, fN, inverse);
        return;
    }
    if (row_bytes % 16 == 0) {
        const int wpr = (int)(row_bytes / 16);
        ra_permute_kernel<uint4, 4><<<grid_for(rows_total * wpr), threads, 0, st>>>(
            (const uint4 *)src, (uint4 *)dst, rows_total, S, L, N, wpr, inverse);
    } else if (row_bytes % 4 == 0) {
        const int wpr = (int)(row_bytes / 4);
        ra_permute_kernel<uint32_t, 4><<<grid_for(rows_total * wpr), threads, 0, st>>>(
            (const uint32_t *)src, (uint32_t *)dst, rows_total, S, L, N, wpr, inverse);
    } else {
        const int wpr = (int)row_bytes;
        ra_permute_kernel<uint8_t, 4><<<grid_for(rows_total * wpr), threads, 0, st>>>(
            (const uint8_t *)src, (uint8_t *)dst, rows_total, S, L, N, wpr, inverse);
    }
}

// ---------------------------------------------------------------- all-to-all
// Sequence-sharded <-> head-sharded relayout of DeepSpeed Ulysses, the
// alternative to the ring that the "Ring Attention" page names (section on
// other kinds of parallelism: an all-to-all exchange gives every device all
// tokens of a subset of the heads).  n devices, Hn heads, Hg = Hn / n per
// device, L = S / n tokens per device:
//   sequence-sharded  [n][B][Hn][L][d]  device i holds tokens [i L, i L + L)
//   head-sharded      [n][B][Hg][S][d]  device g holds heads [g Hg, g Hg + Hg)
// The grid walks destination rows (coalesced writes); each source row is read
// whole, UNROLL loads in flight per thread as in the permutation.
template <typename VEC, int UNROLL>
__global__ void ra_all_to_all_kernel(const VEC *__restrict__ src, VEC *__restrict__ dst, long long n_rows_total,
                                     int B, int Hn, int Hg, int S, int L, int words_per_row, int inverse)
{
    const long long n = n_rows_total * words_per_row;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long base = blockIdx.x * (long long)blockDim.x + threadIdx.x; base < n;
         base += stride * UNROLL) {
        VEC v[UNROLL];
        long long at[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const long long idx = base + u * stride;
            at[u] = idx;
            if (idx < n) {
                const long long row = idx / words_per_row;
                const int w = (int)(idx - row * words_per_row);
                long long from;
                if (!inverse) {
                    // dst row ((g B + b) Hg + h') S + t  <-  src ((i B + b) Hn + g Hg + h') L + a
                    const int t = (int)(row % S);
                    const long long r1 = row / S;
                    const int hl = (int)(r1 % Hg);
                    const long long r2 = r1 / Hg;
                    const int b = (int)(r2 % B);
                    const int g = (int)(r2 / B);
                    const int i = t / L, a = t - i * L;
                    from = (((long long)i * B + b) * Hn + (long long)g * Hg + hl) * L + a;
                } else {
                    // dst row ((i B + b) Hn + h) L + a  <-  src ((g B + b) Hg + h') S + i L + a
                    const int a = (int)(row % L);
                    const long long r1 = row / L;
                    const int h = (int)(r1 % Hn);
                    const long long r2 = r1 / Hn;
                    const int b = (int)(r2 % B);
                    const int i = (int)(r2 / B);
                    const int g = h / Hg, hl = h - g * Hg;
                    from = (((long long)g * B + b) * Hg + hl) * S + (long long)i * L + a;
                }
                v[u] = src[from * words_per_row + w];
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u)
            if (at[u] < n)
                dst[at[u]] = v[u];
    }
}

// The relayout of ra_all_to_all_kernel with 32-bit index arithmetic and the
// divisions above (every word index < 2^31).
template <typename VEC, int UNROLL>
__global__ void ra_all_to_all32_kernel(const VEC *__restrict__ src, VEC *__restrict__ dst, uint32_t n_words,
                                       FastDiv wpr, FastDiv S, FastDiv Hg, FastDiv B, FastDiv L, FastDiv Hn,
                                       int inverse)
{
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t base = blockIdx.x * blockDim.x + threadIdx.x; base < n_words; base += stride * UNROLL) {
        VEC v[UNROLL];
        uint32_t at[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const uint32_t idx = base + u * stride;
            at[u] = idx;
            if (idx < n_words) {
                const uint32_t row = fdiv(idx, wpr);
                const uint32_t w = idx - row * wpr.d;
                uint32_t from;
                if (!inverse) {
                    const uint32_t r1 = fdiv(row, S), t = row - r1 * S.d;
                    const uint32_t r2 = fdiv(r1, Hg), hl = r1 - r2 * Hg.d;
                    const uint32_t g = fdiv(r2, B), b = r2 - g * B.d;
                    const uint32_t i = fdiv(t, L), a = t - i * L.d;
                    from = ((i * B.d + b) * Hn.d + g * Hg.d + hl) * L.d + a;
                } else {
                    const uint32_t r1 = fdiv(row, L), a = row - r1 * L.d;
                    const uint32_t r2 = fdiv(r1, Hn), h = r1 - r2 * Hn.d;
                    const uint32_t i = fdiv(r2, B), b = r2 - i * B.d;
                    const uint32_t g = fdiv(h, Hg), hl = h - g * Hg.d;
                    from = ((g * B.d + b) * Hg.d + hl) * S.d + i * L.d + a;
                }
                v[u] = src[(size_t)from * wpr.d + w];
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u)
            if (at[u] < n_words)
                dst[at[u]] = v[u];
    }
}

void launch_all_to_all(const void *src, void *dst, int B, int Hn, int S, int n_dev, long long row_bytes,
                       int inverse, int sm_count, cudaStream_t st)
{
    const long long rows_total = (long long)B * Hn * S;
    const int L = S / n_dev, Hg = Hn / n_dev;
    const int threads = 256;
    auto grid_for = [&](long long n) {
        long long g = (n + threads - 1) / threads;
        const long long cap = (long long)sm_count * 8;
        return (int)(g < cap ? (g > 0 ? g : 1) : cap);
    };
    const long long vec = row_bytes % 16 == 0 ? 16 : (row_bytes % 4 == 0 ? 4 : 1);
    const long long words = rows_total * (row_bytes / vec);
    // 32-bit path: every word index (and the grid-stride sum) below 2^31
    if (words + 4ll * 8 * sm_count * threads < (1ll << 31)) {
        const FastDiv fw = make_fastdiv((uint32_t)(row_bytes / vec)), fS = make_fastdiv((uint32_t)S),
                      fHg = make_fastdiv((uint32_t)Hg), fB = make_fastdiv((uint32_t)B),
                      fL = make_fastdiv((uint32_t)L), fHn = make_fastdiv((uint32_t)Hn);
        if (vec == 16)
            ra_all_to_all32_kernel<uint4, 4><<<grid_for(words), threads, 0, st>>>(
                (const uint4 *)src, (uint4 *)dst, (uint32_t)words, fw, fS, fHg, fB, fL, fHn, inverse);
        else if (vec == 4)
            ra_all_to_all32_kernel<uint32_t, 4><<<grid_for(words), threads, 0, st>>>(
                (const uint32_t *)src, (uint32_t *)dst, (uint32_t)words, fw, fS, fHg, fB, fL, fHn, inverse);
        else
            ra_all_to_all32_kernel<uint8_t, 4><<<grid_for(words), threads, 0, st>>>(
                (const uint8_t *)src, (uint8_t *)dst, (uint32_t)words, fw, fS, fHg, fB, fL, fHn, inverse);
        return;
    }
    if (row_bytes % 16 == 0) {
        const int wpr = (int)(row_bytes / 16);
        ra_all_to_all_kernel<uint4, 4><<<grid_for(rows_total * wpr), threads, 0, st>>>(
            (const uint4 *)src, (uint4 *)dst, rows_total, B, Hn, Hg, S, L, wpr, inverse);
    } else if (row_bytes % 4 == 0) {
        const int wpr = (int)(row_bytes / 4);
        ra_all_to_all_kernel<uint32_t, 4><<<grid_for(rows_total * wpr), threads, 0, st>>>(
            (const uint32_t *)src, (uint32_t *)dst, rows_total, B, Hn, Hg, S, L, wpr, inverse);
    } else {
        const int wpr = (int)row_bytes;
        ra_all_to_all_kernel<uint8_t, 4><<<grid_for(rows_total * wpr), threads, 0, st>>>(
            (const uint8_t *)src, (uint8_t *)dst, rows_total, B, Hn, Hg, S, L, wpr, inverse);
    }
}

// ---------------------------------------------------------------- merge
// Rows are grouped: `outer` groups of `count` rows starting at row `begin`
// of every group of `stride` rows (for the flat API: outer = 1).  A row is
// handled by d/4 lanes (16-byte vectors); every lane reads both lse values
// before the warp synchronises and one lane writes the merged lse.
__device__ __forceinline__ void merge_weights(float la, float lb, float &wa, float &wb, float &l)
{
    const float mx = fmaxf(la, lb);
    if (mx == -INFINITY) {
        wa = 0.f, wb = 0.f, l = -INFINITY;
        return;
    }
    const float ea = expf(la - mx), eb = expf(lb - mx);  // -inf -> 0
    const float sum = ea + eb;
    l = mx + logf(sum);
    wa = ea / sum;
    wb = eb / sum;
}

__global__ void ra_merge_kernel(float *__restrict__ out_run, float *__restrict__ lse_run,
                                const float *__restrict__ out_s, const float *__restrict__ lse_s,
                                long long outer, long long stride, long long begin,
                                long long count, int d)
{
    const int lane = threadIdx.x & 31;
    const int vpr = d / 4;  // 16-byte vectors per row
    const int rows_per_warp = vpr >= 32 ? 1 : 32 / vpr;
    const int vec_per_lane = vpr >= 32 ? (vpr + 31) / 32 : 1;
    const int sub = vpr >= 32 ? 0 : lane / vpr;  // row within the warp
    const int lv = vpr >= 32 ? lane : lane % vpr;
    const long long n_rows = outer * count;
    const long long warp0 = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
    const long long n_warps = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long wr = warp0 * rows_per_warp; wr < n_rows; wr += n_warps * rows_per_warp) {
        const long long rr = wr + sub;
        const bool active = sub < rows_per_warp && rr < n_rows;
        long long row = 0;
        float la = -INFINITY, lb = -INFINITY;
        if (active) {
            const long long o = rr / count;
            row = o * stride + begin + (rr - o * count);
            la = lse_run[row];
            lb = lse_s[row];
        }
        float wa, wb, l;
        merge_weights(la, lb, wa, wb, l);
        if (active) {
            float4 *orun = reinterpret_cast<float4 *>(out_run + row * d);
            const float4 *os = reinterpret_cast<const float4 *>(out_s + row * d);
            for (int t = 0; t < vec_per_lane; ++t) {
                const int c = lv + 32 * t;
                if (c >= vpr)
                    break;
                const float4 x = orun[c], y = os[c];
                float4 r;
                r.x = wa * x.x + wb * y.x;
                r.y = wa * x.y + wb * y.y;
                r.z = wa * x.z + wb * y.z;
                r.w = wa * x.w + wb * y.w;
                orun[c] = r;
            }
        }
        __syncwarp();
        if (active && lv == 0)
            lse_run[row] = l;
    }
}

void launch_merge(float *out_run, float *lse_run, const float *out_s, const float *lse_s,
                  long long outer, long long stride, long long begin, long long count, int d,
                  int sm_count, cudaStream_t st)
{
    const int threads = 256;
    const int vpr = d / 4;
    const int rows_per_warp = vpr >= 32 ? 1 : 32 / vpr;
    const long long warps = (outer * count + rows_per_warp - 1) / rows_per_warp;
    long long blocks = (warps + 7) / 8;
    const long long cap = (long long)sm_count * 8;
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    ra_merge_kernel<<<(int)blocks, threads, 0, st>>>(out_run, lse_run, out_s, lse_s, outer,
                                                     stride, begin, count, d);
}

// ---------------------------------------------------------------- finalize
// fp32 running result (kernel order) -> output in natural order; bf16 output
// is rounded to nearest even.  Striped rows are scattered back to t(p).
template <typename OUT>
__global__ void ra_finalize_kernel(const float *__restrict__ run, const float *__restrict__ run_lse,
                                   OUT *__restrict__ out, float *__restrict__ lse,
                                   long long rows_total, int S, int L, int N, int striped, int d)
{
    const long long n = rows_total * (d / 4);
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long row = idx / (d / 4);
        const int c4 = (int)(idx - row * (d / 4));
        const long long bh = row / S;
        const int p = (int)(row - bh * S);
        const int t = striped ? (p % L) * N + p / L : p;
        const long long drow = bh * S + t;
        const float4 x = reinterpret_cast<const float4 *>(run + row * d)[c4];
        if constexpr (sizeof(OUT) == 4) {
            reinterpret_cast<float4 *>(out + drow * d)[c4] = x;
        } else {
            __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y);
            __nv_bfloat162 hi = __floats2bfloat162_rn(x.z, x.w);
            uint2 w;
            w.x = *reinterpret_cast<uint32_t *>(&lo);
            w.y = *reinterpret_cast<uint32_t *>(&hi);
            reinterpret_cast<uint2 *>(out + drow * d)[c4] = w;
        }
        if (c4 == 0)
            lse[drow] = run_lse[row];
    }
}

void launch_finalize(const float *run, const float *run_lse, void *out, float *lse, int out_bf16,
                     long long rows_total, int S, int N, int striped, int d, int sm_count,
                     cudaStream_t st)
{
    const int threads = 256;
    long long blocks = (rows_total * (d / 4) + threads - 1) / threads;
    const long long cap = (long long)sm_count * 8;
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    const int L = S / N;
    if (out_bf16)
        ra_finalize_kernel<__nv_bfloat16><<<(int)blocks, threads, 0, st>>>(
            run, run_lse, (__nv_bfloat16 *)out, lse, rows_total, S, L, N, striped, d);
    else
        ra_finalize_kernel<float><<<(int)blocks, threads, 0, st>>>(
            run, run_lse, (float *)out, lse, rows_total, S, L, N, striped, d);
}

// ---------------------------------------------------------------- combine
// The nsplit normalised fp32 partials (out_k, lse_k) of every query row
// (kernel order, partial k at part + k part_stride rows) folded into the
// final row: lse = log sum_k exp(lse_k), out = sum_k exp(lse_k - lse) out_k,
// written in natural order (striped rows scattered back to t(p)); bf16
// output is rounded to nearest even.  A partial with lse_k = -inf holds no
// key and is not read.  The same running-softmax merge as ra_merge_kernel,
// over nsplit partials at once.
template <typename OUT>
__device__ __forceinline__ void combine_row_vector(const float *__restrict__ part, const float *__restrict__ part_lse,
                                                   int nsplit, long long part_stride, OUT *__restrict__ out,
                                                   float *__restrict__ lse, long long row, int c4, long long drow,
                                                   int d)
{
    float m = -INFINITY;
    for (int k = 0; k < nsplit; ++k)
        m = fmaxf(m, __ldg(part_lse + k * part_stride + row));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float sum = 0.f;
    if (m != -INFINITY) {
        for (int k = 0; k < nsplit; ++k) {
            const float lk = __ldg(part_lse + k * part_stride + row);
            if (lk == -INFINITY)
                continue;
            const float wk = expf(lk - m);
            const float4 x = __ldg(reinterpret_cast<const float4 *>(part + (k * part_stride + row) * d) + c4);
            acc.x += wk * x.x;
            acc.y += wk * x.y;
            acc.z += wk * x.z;
            acc.w += wk * x.w;
            sum += wk;
        }
        const float inv = 1.f / sum;
        acc.x *= inv, acc.y *= inv, acc.z *= inv, acc.w *= inv;
    }
    if constexpr (sizeof(OUT) == 4) {
        reinterpret_cast<float4 *>(out + drow * d)[c4] = acc;
    } else {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 w;
        w.x = *reinterpret_cast<uint32_t *>(&lo);
        w.y = *reinterpret_cast<uint32_t *>(&hi);
        reinterpret_cast<uint2 *>(out + drow * d)[c4] = w;
    }
    if (c4 == 0)
        lse[drow] = m == -INFINITY ? -INFINITY : m + logf(sum);
}

// One thread per 16-byte vector of an output row.  NARROW: every vector
// index is below 2^31, and the row, head and position come from 32-bit
// division by invariant integers; otherwise 64-bit arithmetic.
template <typename OUT, bool NARROW>
__global__ void ra_combine_kernel(const float *__restrict__ part, const float *__restrict__ part_lse, int nsplit,
                                  long long part_stride, OUT *__restrict__ out, float *__restrict__ lse,
                                  long long rows_total, int S, int L, int N, int striped, int d, FastDiv fv,
                                  FastDiv fS, FastDiv fL)
{
    const int vpr = d / 4;  // 16-byte vectors per row
    // launched as a programmatic dependent of the attention kernel: the CTAs
    // may start while its last CTAs finish, and wait here until its writes
    // (the partials) are complete and visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (NARROW) {
        const uint32_t n = (uint32_t)(rows_total * vpr);
        for (uint32_t idx = blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += gridDim.x * blockDim.x) {
            const uint32_t row = fdiv(idx, fv);
            const int c4 = (int)(idx - row * (uint32_t)vpr);
            const uint32_t bh = fdiv(row, fS);
            const uint32_t p = row - bh * (uint32_t)S;
            uint32_t t = p;
            if (striped) {
                const uint32_t r = fdiv(p, fL);
                t = (p - r * (uint32_t)L) * (uint32_t)N + r;
            }
            combine_row_vector<OUT>(part, part_lse, nsplit, part_stride, out, lse, row, c4,
                                    (long long)bh * S + t, d);
        }
    } else {
        const long long n = rows_total * vpr;
        for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n;
             idx += (long long)gridDim.x * blockDim.x) {
            const long long row = idx / vpr;
            const int c4 = (int)(idx - row * vpr);
            const long long bh = row / S;
            const int p = (int)(row - bh * S);
            const int t = striped ? (p % L) * N + p / L : p;
            combine_row_vector<OUT>(part, part_lse, nsplit, part_stride, out, lse, row, c4, bh * S + t, d);
        }
    }
}

void launch_combine(const float *part, const float *part_lse, int nsplit, long long part_stride, void *out,
                    float *lse, int out_bf16, long long rows_total, int S, int N, int striped, int d,
                    int sm_count, cudaStream_t st)
{
    const int threads = 256;
    long long blocks = (rows_total * (d / 4) + threads - 1) / threads;
    const long long cap = (long long)sm_count * 8;
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    const int L = S / N;
    const bool narrow = rows_total * (d / 4) < (1ll << 31);
    const FastDiv fv = make_fastdiv((uint32_t)(d / 4)), fS = make_fastdiv((uint32_t)S), fL = make_fastdiv((uint32_t)L);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(threads);
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (out_bf16) {
        auto *o = (__nv_bfloat16 *)out;
        if (narrow)
            cudaLaunchKernelEx(&cfg, ra_combine_kernel<__nv_bfloat16, true>, part, part_lse, nsplit, part_stride, o,
                               lse, rows_total, S, L, N, striped, d, fv, fS, fL);
        else
            cudaLaunchKernelEx(&cfg, ra_combine_kernel<__nv_bfloat16, false>, part, part_lse, nsplit, part_stride, o,
                               lse, rows_total, S, L, N, striped, d, fv, fS, fL);
    } else {
        auto *o = (float *)out;
        if (narrow)
            cudaLaunchKernelEx(&cfg, ra_combine_kernel<float, true>, part, part_lse, nsplit, part_stride, o, lse,
                               rows_total, S, L, N, striped, d, fv, fS, fL);
        else
            cudaLaunchKernelEx(&cfg, ra_combine_kernel<float, false>, part, part_lse, nsplit, part_stride, o, lse,
                               rows_total, S, L, N, striped, d, fv, fS, fL);
    }
}

}  // namespace ra
