// sv_refine.cu -- test hooks of the re-draw's building blocks: its bounded waits and its
// double-float exponential.  The re-draw itself runs inside the cooperative draw kernel
// (sv_refine.cuh, sv_sample.cu).
#include "spec_verify.h"
#include "sv_device.cuh"
#include "sv_df.cuh"
#include "sv_grid.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

// Test hook of the bounded waits: one CTA waits for the flag ctl[5] (which it sets itself
// first when expected == 1) and then meets the grid barrier expecting `expected` arrivals;
// with expected == 2 nobody sets the flag and nobody else comes, each wait runs out after
// limit_ns and records SV_ERR_TIMEOUT in ctl[kBarStatus].
__global__ void wait_selftest_kernel(int *ctl, int expected, uint64_t limit_ns) {
    constexpr int kFlag = 5;
    if (threadIdx.x == 0) {
        ctl[kBarCount] = 0;
        ctl[kBarStatus] = 0;
        ctl[kFlag] = expected == 1 ? 1 : 0;
        __threadfence();
        wait_nonzero(ctl + kFlag, ctl + kBarStatus, limit_ns);
    }
    __syncthreads();
    grid_barrier(ctl, expected, limit_ns);
}

__global__ void exp_df_kernel(const float *__restrict__ y_hi, const float *__restrict__ y_lo, int n,
                              float *__restrict__ out_hi, float *__restrict__ out_lo) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const df e = exp_df(df{y_hi[i], y_lo[i]});
    out_hi[i] = e.hi;
    out_lo[i] = e.lo;
}

}  // namespace

cudaError_t launch_wait_selftest(int *ctl, int expected, uint64_t limit_ns, cudaStream_t s) {
    wait_selftest_kernel<<<1, 32, 0, s>>>(ctl, expected, limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_exp_df(const float *y_hi, const float *y_lo, int n, float *out_hi, float *out_lo,
                          cudaStream_t s) {
    exp_df_kernel<<<unsigned((n + 255) / 256), 256, 0, s>>>(y_hi, y_lo, n, out_hi, out_lo);
    return cudaGetLastError();
}

}  // namespace sv
