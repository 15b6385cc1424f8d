// Internal launchers shared by the C-ABI layer (ra_api.cu) and the kernel
// translation units.  Not part of the public interface.
#pragma once

#include <atomic>
#include <cstddef>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ra_schedule.h"

namespace ra {

// Status code the device error word carries for a bounded wait that ran out.
constexpr unsigned int RA_DEV_TIMEOUT_CODE = 5;

// One-time launch state (function attributes, occupancy queries) is kept per
// device: a process that calls on several devices sets each device's up once.
constexpr int RA_MAX_DEVICES = 64;

// The current device, or -1 when it cannot be read or has no cache slot.
inline int current_device_slot()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return dev >= 0 && dev < RA_MAX_DEVICES ? dev : -1;
}

// Runs set_up() once per device (again after a failure); returns its error.
template <class F>
cudaError_t once_per_device(std::atomic<int> (&done)[RA_MAX_DEVICES], F set_up)
{
    const int dev = current_device_slot();
    if (dev < 0)
        return cudaErrorInvalidDevice;
    if (done[dev].load(std::memory_order_acquire))
        return cudaSuccess;
    const cudaError_t e = set_up();
    if (e == cudaSuccess)
        done[dev].store(1, std::memory_order_release);
    return e;
}

void launch_attn_f32(const float *q, const float *k, const float *v, float *out, float *lse,
                     int B, int H, int Hkv, int S, int d, int N, int layout, int causal,
                     int s_begin, int s_end, int rank_lo, int rank_hi, cudaStream_t st);
// Sequence-sharded [n][B][Hn][S/n][d] <-> head-sharded [n][B][Hn/n][S][d]
// (inverse = 1 goes back); rows of row_bytes bytes, bit-exact.
void launch_all_to_all(const void *src, void *dst, int B, int Hn, int S, int n_dev, long long row_bytes,
                       int inverse, int sm_count, cudaStream_t st);
// out[bh, row0 + r, :] = 0 and lse[bh, row0 + r] = -inf for r < nrows: the
// partial of query rows that see no key at this step.
void launch_fill_empty(float *out, float *lse, long long BH, int S, long long row0, long long nrows,
                       int d, int sm_count, cudaStream_t st);

void launch_permute(const void *src, void *dst, long long rows_total, int S, int N,
                    long long row_bytes, int inverse, int sm_count, cudaStream_t st);

void launch_merge(float *out_run, float *lse_run, const float *out_s, const float *lse_s,
                  long long outer, long long stride, long long begin, long long count, int d,
                  int sm_count, cudaStream_t st);

void launch_finalize(const float *run, const float *run_lse, void *out, float *lse, int out_bf16,
                     long long rows_total, int S, int N, int striped, int d, int sm_count,
                     cudaStream_t st);

// Tensor-core attention; the work units (see RaUnitSpace) are enumerated in
// the kernel, so the launch needs no device-side list.
struct TcLaunch {
    const void *q, *k, *v;       // bf16, kernel (possibly striped) order
    void *out;                   // bf16 (out_f32 = 0) or fp32 normalised partial
    float *lse;
    int B, H, Hkv, S, d, N;
    int layout, causal;
    int s_begin, s_end;          // ring steps walked by every unit
    int rank_lo, rank_hi;        // query blocks (ranks) computed: [rank_lo, rank_hi)
    int out_f32;
    unsigned long long timeout_ns;
    int sm_count;
    int cluster;                 // 2: share K/V loads between CTA pairs where the units allow
    // > 1: cut every unit's walk over its key tiles into nsplit pieces, each
    // a work item writing its own normalised fp32 partial (out_f32 = 1) at
    // out + k split_out_bytes and lse + k split_lse_stride (k = piece)
    int nsplit;
    long long split_out_bytes, split_lse_stride;
};

// Folds nsplit normalised fp32 partials per row (kernel order; partial k of
// row r at part[(k part_stride + r) d], lse at part_lse[k part_stride + r])
// into the output in natural order (bf16 or fp32) and its lse.
void launch_combine(const float *part, const float *part_lse, int nsplit, long long part_stride, void *out,
                    float *lse, int out_bf16, long long rows_total, int S, int N, int striped, int d,
                    int sm_count, cudaStream_t st);

// Backward pass (bf16, d in {64, 128}): delta = rowsum(dout * out), then the
// dK/dV and dQ tensor-core kernels.  All tensors in the layout's rank-major
// order; lse and delta fp32 [B H S].
struct BwdLaunch {
    const void *q, *k, *v, *out, *dout;
    const float *lse;
    float *delta;                // written
    void *dq, *dk, *dv;          // written, bf16 (fp32 for launch_bwd_f32)
    int B, H, Hkv, S, d, N;
    int layout, causal;
    unsigned long long timeout_ns;
};
cudaError_t launch_bwd(const BwdLaunch &a, cudaStream_t st);
// The same pass in fp32 on the SIMT cores (any d <= 256): delta, dQ, dK/dV.
void launch_bwd_f32(const BwdLaunch &a, cudaStream_t st);

// Device address of the library's status word on the current device (the
// word ra_check reads); kernels in other translation units get it as a
// parameter.  nullptr if it cannot be looked up.
unsigned int *device_status_ptr();

// Returns cudaSuccess or the first CUDA error met while encoding tensor maps
// or launching.
cudaError_t launch_attn_tc(const TcLaunch &a, cudaStream_t st);

// Device-side error word helpers (defined in ra_attn_sm103.cu).
cudaError_t read_and_clear_device_status(unsigned int *status);

// One-thread kernel whose bounded wait on a never-completed mbarrier runs out.
cudaError_t launch_wait_probe(unsigned long long timeout_ns, cudaStream_t st);

}  // namespace ra
