// Exact fp32 backward pass (SIMT, no tensor cores): the gradients of exact
// attention written out per row, in the ring's order, for checks at fp32
// precision (the tensor-core kernels in ra_bwd_sm103.cu take bf16).
//
// Same definition as the tensor-core path ("Context Parallelism" glossary
// page, ultralytics.com/tr, section "Pratik Kullanim ve Odunlesimler": the
// example trains through the ring; "Ring Attention" page, section "Halka
// Dikkati Nasil Calisir": the ring is exact), with c = 1/sqrt(d):
//   p = exp(c q.k - lse), dp = dO.v, ds = p (dp - delta),
//   dq = c sum ds k,  dk = c sum ds q,  dv = sum p dO.
// One warp per row; lane l owns columns l, l + 32, ...
#include <cstdint>
#include <cuda_runtime.h>

#include "ra_internal.h"
#include "ra_schedule.h"

namespace ra {

namespace {

constexpr int BF_WARPS = 8;
constexpr int BF_MAXW = 8;  // d <= 256

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// delta[row] = sum_c dout[row, c] out[row, c]
__global__ void ra_bwd_delta_f32_kernel(const float *__restrict__ o, const float *__restrict__ dout,
                                        float *__restrict__ delta, long long rows, int d)
{
    const long long row = (long long)blockIdx.x * BF_WARPS + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows)
        return;
    float acc = 0.f;
    for (int c = lane; c < d; c += 32)
        acc = fmaf(o[row * d + c], dout[row * d + c], acc);
    acc = warp_sum(acc);
    if (lane == 0)
        delta[row] = acc;
}

// dq of query row a of block i (head bh): key blocks j = (i - s) mod N.
__global__ void __launch_bounds__(BF_WARPS * 32)
ra_bwd_dq_f32_kernel(const float *__restrict__ q, const float *__restrict__ k, const float *__restrict__ v,
                     const float *__restrict__ dout, const float *__restrict__ lse,
                     const float *__restrict__ delta, float *__restrict__ dq, int H, int Hkv, int S, int d, int L,
                     int N, int layout, int causal, float scale)
{
    const int lane = threadIdx.x & 31;
    const int a = blockIdx.x * BF_WARPS + (threadIdx.x >> 5);
    const int i = blockIdx.y;
    const long long bh = blockIdx.z;
    if (a >= L)
        return;
    const long long b = bh / H;
    const int h = (int)(bh % H);
    const long long bhkv = b * Hkv + h / (H / Hkv);
    const long long row = bh * S + (long long)i * L + a;
    const int nw = (d + 31) / 32;
    float qv[BF_MAXW], dov[BF_MAXW], acc[BF_MAXW];
#pragma unroll
    for (int w = 0; w < BF_MAXW; ++w) {
        const int c = lane + 32 * w;
        const bool in = w < nw && c < d;
        qv[w] = in ? q[row * d + c] * scale : 0.f;
        dov[w] = in ? dout[row * d + c] : 0.f;
        acc[w] = 0.f;
    }
    const float lr = lse[row], dr = delta[row];
    for (int s = 0; s < N; ++s) {
        const int j = ra_ring_block(i, s, N);
        const int cls = ra_block_class(layout, causal, i, j);
        if (cls == RA_CLS_SKIP)
            continue;
        const int lim = ra_key_limit(cls, a, L);
        const float *kb = k + (bhkv * S + (long long)j * L) * d;
        const float *vb = v + (bhkv * S + (long long)j * L) * d;
        for (int u = 0; u < lim; ++u) {
            float sc = 0.f, dp = 0.f;
#pragma unroll
            for (int w = 0; w < BF_MAXW; ++w) {
                const int c = lane + 32 * w;
                if (w < nw && c < d) {
                    sc = fmaf(qv[w], kb[(long long)u * d + c], sc);
                    dp = fmaf(dov[w], vb[(long long)u * d + c], dp);
                }
            }
            sc = warp_sum(sc);
            dp = warp_sum(dp);
            const float ds = expf(sc - lr) * (dp - dr);
#pragma unroll
            for (int w = 0; w < BF_MAXW; ++w) {
                const int c = lane + 32 * w;
                if (w < nw && c < d)
                    acc[w] = fmaf(ds, kb[(long long)u * d + c], acc[w]);
            }
        }
    }
#pragma unroll
    for (int w = 0; w < BF_MAXW; ++w) {
        const int c = lane + 32 * w;
        if (w < nw && c < d)
            dq[row * d + c] = acc[w] * scale;
    }
}

// dk, dv of key row bl of block j (kv head bhkv): query blocks i = (j + s)
// mod N, the group's query heads, the query rows a that see the key.
__global__ void __launch_bounds__(BF_WARPS * 32)
ra_bwd_dkdv_f32_kernel(const float *__restrict__ q, const float *__restrict__ k, const float *__restrict__ v,
                       const float *__restrict__ dout, const float *__restrict__ lse,
                       const float *__restrict__ delta, float *__restrict__ dk, float *__restrict__ dv, int H,
                       int Hkv, int S, int d, int L, int N, int layout, int causal, float scale)
{
    const int lane = threadIdx.x & 31;
    const int bl = blockIdx.x * BF_WARPS + (threadIdx.x >> 5);
    const int j = blockIdx.y;
    const long long bhkv = blockIdx.z;
    if (bl >= L)
        return;
    const long long b = bhkv / Hkv;
    const int g = (int)(bhkv % Hkv), grp = H / Hkv;
    const long long row = bhkv * S + (long long)j * L + bl;
    const int nw = (d + 31) / 32;
    float kv[BF_MAXW], vv[BF_MAXW], ak[BF_MAXW], av[BF_MAXW];
#pragma unroll
    for (int w = 0; w < BF_MAXW; ++w) {
        const int c = lane + 32 * w;
        const bool in = w < nw && c < d;
        kv[w] = in ? k[row * d + c] * scale : 0.f;
        vv[w] = in ? v[row * d + c] : 0.f;
        ak[w] = av[w] = 0.f;
    }
    for (int s = 0; s < N; ++s) {
        const int i = (j + s) % N;
        const int cls = ra_block_class(layout, causal, i, j);
        if (cls == RA_CLS_SKIP)
            continue;
        // key bl is visible to query a iff bl < ra_key_limit(cls, a, L)
        const int a0 = cls == RA_CLS_FULL ? 0 : (cls == RA_CLS_DIAG_INCL ? bl : bl + 1);
        for (int hh = 0; hh < grp; ++hh) {
            const long long bh = b * H + (long long)g * grp + hh;
            for (int a = a0; a < L; ++a) {
                const long long qr = bh * S + (long long)i * L + a;
                float sc = 0.f, dp = 0.f;
#pragma unroll
                for (int w = 0; w < BF_MAXW; ++w) {
                    const int c = lane + 32 * w;
                    if (w < nw && c < d) {
                        sc = fmaf(kv[w], q[qr * d + c], sc);
                        dp = fmaf(vv[w], dout[qr * d + c], dp);
                    }
                }
                sc = warp_sum(sc);
                dp = warp_sum(dp);
                const float pr = expf(sc - lse[qr]);
                const float ds = pr * (dp - delta[qr]);
#pragma unroll
                for (int w = 0; w < BF_MAXW; ++w) {
                    const int c = lane + 32 * w;
                    if (w < nw && c < d) {
                        av[w] = fmaf(pr, dout[qr * d + c], av[w]);
                        ak[w] = fmaf(ds, q[qr * d + c], ak[w]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int w = 0; w < BF_MAXW; ++w) {
        const int c = lane + 32 * w;
        if (w < nw && c < d) {
            dk[row * d + c] = ak[w] * scale;
            dv[row * d + c] = av[w];
        }
    }
}

}  // namespace

void launch_bwd_f32(const BwdLaunch &a, cudaStream_t st)
{
    const int L = a.S / a.N;
    const long long rows = (long long)a.B * a.H * a.S;
    const float scale = 1.0f / sqrtf((float)a.d);
    ra_bwd_delta_f32_kernel<<<(unsigned)((rows + BF_WARPS - 1) / BF_WARPS), BF_WARPS * 32, 0, st>>>(
        static_cast<const float *>(a.out), static_cast<const float *>(a.dout), a.delta, rows, a.d);
    dim3 gq((L + BF_WARPS - 1) / BF_WARPS, a.N, a.B * a.H);
    ra_bwd_dq_f32_kernel<<<gq, BF_WARPS * 32, 0, st>>>(
        static_cast<const float *>(a.q), static_cast<const float *>(a.k), static_cast<const float *>(a.v),
        static_cast<const float *>(a.dout), a.lse, a.delta, static_cast<float *>(a.dq), a.H, a.Hkv, a.S, a.d, L,
        a.N, a.layout, a.causal, scale);
    dim3 gk((L + BF_WARPS - 1) / BF_WARPS, a.N, a.B * a.Hkv);
    ra_bwd_dkdv_f32_kernel<<<gk, BF_WARPS * 32, 0, st>>>(
        static_cast<const float *>(a.q), static_cast<const float *>(a.k), static_cast<const float *>(a.v),
        static_cast<const float *>(a.dout), a.lse, a.delta, static_cast<float *>(a.dk), static_cast<float *>(a.dv),
        a.H, a.Hkv, a.S, a.d, L, a.N, a.layout, a.causal, scale);
}

}  // namespace ra
