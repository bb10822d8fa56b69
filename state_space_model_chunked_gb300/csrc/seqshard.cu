// One long sequence split over GPUs by tokens: the two small kernels of the
// exchange.  Step-3 of the CGLA kernel page (section III.A: the state carried
// sequentially across chunks, with the input-dependent diagonal decay)
// applied at the granularity of one GPU's token range:
//
//   H_in[0] = init,  H_in[r+1] = exp(a_r) H_in[r] + F_r,
//
// where a_r = A_h * (sum of dt over range r) is the range's log-decay and F_r
// the state range r reaches from a zero state (a scan of the range without
// an initial state).  Each GPU scans its range once from zero for F_r, the
// pairs (a_r, F_r) are exchanged (one all-gather), every GPU chains them to
// its own H_in, and scans its range again from H_in for y.
//
// Both kernels are small next to the scans: the log-decay reads dt once (4
// bytes per token and head), the chain reads R contributions and writes R
// entering states of H P N floats per batch row.
#include <cuda_runtime.h>
#include <stdint.h>

#include "launch.h"

namespace {

// out[b][h] = A_h * sum_t dt'[b][t][h], dt' the step size after the optional
// transform; summed in fp64.  A CTA of 32 x 8 threads takes 32 heads of one
// batch row: lanes walk consecutive heads (128-byte rows of dt), the 8 rows
// of threads stride over the tokens, and shared memory adds their sums.
template <bool kFuse>
__global__ void __launch_bounds__(256)
ssd_range_log_decay_kernel(const float *__restrict__ dt, const float *__restrict__ A, int L,
                           int H, SsdFuse fuse, float *__restrict__ out) {
    __shared__ double part[8][32];
    const int b = blockIdx.x;
    const int h = blockIdx.y * 32 + threadIdx.x;
    double acc = 0.0;
    if (h < H) {
        const float bias = ssd_dt_bias<kFuse>(fuse, h);
        const float *row = dt + (size_t)b * L * H + h;
        for (int t = threadIdx.y; t < L; t += 8)
            acc += (double)ssd_dt<kFuse>(fuse, row[(size_t)t * H], bias);
    }
    part[threadIdx.y][threadIdx.x] = acc;
    __syncthreads();
    if (threadIdx.y == 0 && h < H) {
        double s = 0.0;
#pragma unroll
        for (int i = 0; i < 8; ++i) s += part[i][threadIdx.x];
        out[(size_t)b * H + h] = (float)((double)A[h] * s);
    }
}

// entering[r] for r = 0 .. R-1, elementwise over (b, h, p, n): the chain of
// the ranges' contributions with their decays, from init (zeros when NULL).
__global__ void __launch_bounds__(256)
ssd_chain_states_kernel(const float *__restrict__ contrib, const float *__restrict__ log_decay,
                        const float *__restrict__ init, int R, size_t per_row, size_t n,
                        int BH, float *__restrict__ entering) {
    const size_t i = (size_t)blockIdx.x * 256 + threadIdx.x;
    if (i >= n) return;
    const size_t bh = i / per_row;             // (batch row, head) of this element
    float hs = init ? init[i] : 0.f;
    for (int r = 0; r < R; ++r) {
        entering[(size_t)r * n + i] = hs;
        hs = expf(log_decay[(size_t)r * BH + bh]) * hs + contrib[(size_t)r * n + i];
    }
}

}  // namespace

cudaError_t ssd_launch_range_log_decay(const float *dt, const float *A, int batch, int L, int H,
                                       const SsdFuse &fuse, float *out, cudaStream_t stream) {
    const dim3 grid((unsigned)batch, (unsigned)((H + 31) / 32)), block(32, 8);
    if (ssd_dt_transform_active(fuse))
        ssd_range_log_decay_kernel<true><<<grid, block, 0, stream>>>(dt, A, L, H, fuse, out);
    else
        ssd_range_log_decay_kernel<false><<<grid, block, 0, stream>>>(dt, A, L, H, fuse, out);
    return cudaGetLastError();
}

cudaError_t ssd_launch_chain_states(const float *contrib, const float *log_decay,
                                    const float *init, int R, int batch, int H, int P, int N,
                                    float *entering, cudaStream_t stream) {
    const size_t per_row = (size_t)P * N;
    const size_t n = (size_t)batch * H * per_row;
    if (n == 0) return cudaSuccess;
    ssd_chain_states_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(
        contrib, log_decay, init, R, per_row, n, batch * H, entering);
    return cudaGetLastError();
}
