// Decode: one token of the SSD recurrence for every (batch, head), the O(1)
// cached step of "Compiler-First State Space Duality and Portable O(1)
// Autoregressive Caching" (abstract); the per-head transition is the
// input-dependent diagonal of the CGLA kernel page, section III.A.
//
//   h[p][n] <- exp(dt*A_h) * h[p][n] + dt * B[n] * x[p]
//   y[p]     = sum_n C[n] * h[p][n] + D_h * x[p]
//
// The update is HBM-bound (0.75 flop per byte): every state byte is read once
// and written once.  One CTA owns one (batch, head) state of P x N floats; a
// row p is spread over TPR threads holding VPT float4 each, so a warp reads
// and writes whole 128-byte lines.  All of a thread's row loads are issued
// before any arithmetic to keep enough bytes in flight, and the state uses
// streaming (evict-first) loads and stores because it is touched once per
// call.  y reduces C . h across the TPR threads of a row with shuffles.
#include "common.cuh"
#include "launch.h"

namespace {

constexpr int kThreads = 256;
constexpr int kBatchRows = 8;   // rows each thread has in flight at once

template <typename T, int VPT>
__global__ void __launch_bounds__(kThreads)
ssd_decode_kernel(float *__restrict__ state, const T *__restrict__ x,
                  const float *__restrict__ dt, const float *__restrict__ A,
                  const T *__restrict__ Bm, const T *__restrict__ Cm,
                  const float *__restrict__ D, T *__restrict__ y, int H, int P,
                  int N, int G) {
    const int bh = blockIdx.x;             // b * H + h
    const int b = bh / H, h = bh - b * H;
    const int g = h / (H / G);
    const int tpr = N / (4 * VPT);         // threads per row, power of two <= 32
    const int rpp = kThreads / tpr;        // rows per pass
    const int lane_n = threadIdx.x % tpr;
    const int r0 = threadIdx.x / tpr;

    const float dtv = dt[bh];
    const float decay = expf(dtv * A[h]);
    const float Dh = D ? D[h] : 0.0f;

    float4 Bv[VPT], Cv[VPT];
    const T *Bg = Bm + ((size_t)b * G + g) * N;
    const T *Cg = Cm + ((size_t)b * G + g) * N;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int n0 = 4 * (lane_n + v * tpr);
        Bv[v] = ssd_ld4(Bg + n0);
        Cv[v] = ssd_ld4(Cg + n0);
    }
    float *st = state + (size_t)bh * P * N;
    const T *xr = x + (size_t)bh * P;
    T *yr = y + (size_t)bh * P;

    // the loop bound is the same for every thread so the row shuffles below
    // always see full warps
    for (int pb0 = 0; pb0 < P; pb0 += kBatchRows * rpp) {
        const int pb = pb0 + r0;
        float4 s[kBatchRows][VPT];
        float xv[kBatchRows];
#pragma unroll
        for (int i = 0; i < kBatchRows; ++i) {
            const int p = pb + i * rpp;
            if (p < P) {
                xv[i] = ssd_ld(xr + p);
#pragma unroll
                for (int v = 0; v < VPT; ++v)
                    s[i][v] = __ldcs(reinterpret_cast<const float4 *>(
                        st + (size_t)p * N + 4 * (lane_n + v * tpr)));
            }
        }
#pragma unroll
        for (int i = 0; i < kBatchRows; ++i) {
            const int p = pb + i * rpp;
            float acc = 0.0f;
            if (p < P) {
                const float dx = dtv * xv[i];
#pragma unroll
                for (int v = 0; v < VPT; ++v) {
                    float4 q = s[i][v];
                    q.x = fmaf(decay, q.x, dx * Bv[v].x);
                    q.y = fmaf(decay, q.y, dx * Bv[v].y);
                    q.z = fmaf(decay, q.z, dx * Bv[v].z);
                    q.w = fmaf(decay, q.w, dx * Bv[v].w);
                    __stcs(reinterpret_cast<float4 *>(st + (size_t)p * N +
                                                      4 * (lane_n + v * tpr)),
                           q);
                    acc = fmaf(Cv[v].x, q.x, acc);
                    acc = fmaf(Cv[v].y, q.y, acc);
                    acc = fmaf(Cv[v].z, q.z, acc);
                    acc = fmaf(Cv[v].w, q.w, acc);
                }
            }
            // reduce over the tpr threads of this row (aligned power-of-two group)
            for (int off = tpr >> 1; off > 0; off >>= 1)
                acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (p < P && lane_n == 0) ssd_st(yr + p, acc + Dh * xv[i]);
        }
    }
}

template <typename T>
cudaError_t launch_t(float *state, const void *x, const float *dt, const float *A,
                     const void *B, const void *C, const float *D, void *y, int batch,
                     int H, int P, int N, int G, cudaStream_t stream) {
    const unsigned grid = (unsigned)((size_t)batch * H);
    if (N <= 128) {
        ssd_decode_kernel<T, 1><<<grid, kThreads, 0, stream>>>(
            state, (const T *)x, dt, A, (const T *)B, (const T *)C, D, (T *)y, H, P, N, G);
    } else {
        ssd_decode_kernel<T, 2><<<grid, kThreads, 0, stream>>>(
            state, (const T *)x, dt, A, (const T *)B, (const T *)C, D, (T *)y, H, P, N, G);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t ssd_launch_decode(float *state, const void *x, const float *dt,
                              const float *A, const void *B, const void *C,
                              const float *D, void *y, bool bf16, int batch,
                              int H, int P, int N, int G, cudaStream_t stream) {
    if (bf16)
        return launch_t<__nv_bfloat16>(state, x, dt, A, B, C, D, y, batch, H, P, N, G, stream);
    return launch_t<float>(state, x, dt, A, B, C, D, y, batch, H, P, N, G, stream);
}
