// fp8 (E4M3) -> bfloat16 widening of prefill inputs.
//
// An fp8 prefill call widens x, B and C once into bfloat16 copies in its
// workspace, then runs the bf16 path on them.  Every E4M3 value (3
// significand bits, exponents 2^-9 .. 2^8) is exactly a bfloat16 value (7
// significand bits, fp32's exponent range), so the widening is exact; the
// conversion goes through the hardware E4M3x2 -> f16x2 convert (f16 holds
// every E4M3 value exactly too) and fp32.
//
// The kernel is HBM-bound: 1 byte read and 2 bytes written per value.  Each
// thread moves four independent 16-value vectors per step (64 bytes in, 128
// out) so that enough loads are in flight per SM, on a grid of a few CTAs per
// SM striding over up to three arrays in one launch.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "launch.h"

namespace {

constexpr int kWidenThreads = 256;
constexpr int kWidenUnroll = 4;

// 16 E4M3 values (one 16-byte vector) -> 16 bfloat16 values (two vectors)
__device__ __forceinline__ void widen16(uint4 v, uint4 &lo, uint4 &hi) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)(w[i] >> (16 * k));
            const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
            const __nv_bfloat162 b = __float22bfloat162_rn(f);
            o[2 * i + k] = *reinterpret_cast<const uint32_t *>(&b);
        }
    }
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}

__device__ __forceinline__ __nv_bfloat16 widen1(uint8_t c) {
    const __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
    return __float2bfloat16_rn(__half2float(*reinterpret_cast<const __half *>(&hr)));
}

__global__ void __launch_bounds__(kWidenThreads)
ssd_fp8_widen_kernel(SsdWidenJobs jobs) {
    const size_t stride = (size_t)gridDim.x * kWidenThreads;
    const size_t tid = (size_t)blockIdx.x * kWidenThreads + threadIdx.x;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        if (j >= jobs.count) break;
        const uint8_t *src = static_cast<const uint8_t *>(jobs.job[j].src);
        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(jobs.job[j].dst);
        const size_t n = jobs.job[j].n;
        const size_t nv = n / 16;                  // whole 16-value vectors
        const uint4 *sv = reinterpret_cast<const uint4 *>(src);
        uint4 *dv = reinterpret_cast<uint4 *>(dst);
        size_t i = tid;
        for (; i + (kWidenUnroll - 1) * stride < nv; i += kWidenUnroll * stride) {
            uint4 v[kWidenUnroll];
#pragma unroll
            for (int u = 0; u < kWidenUnroll; ++u) v[u] = __ldcs(sv + i + u * stride);
#pragma unroll
            for (int u = 0; u < kWidenUnroll; ++u) {
                uint4 lo, hi;
                widen16(v[u], lo, hi);
                dv[2 * (i + u * stride)] = lo;
                dv[2 * (i + u * stride) + 1] = hi;
            }
        }
        for (; i < nv; i += stride) {
            uint4 lo, hi;
            widen16(__ldcs(sv + i), lo, hi);
            dv[2 * i] = lo;
            dv[2 * i + 1] = hi;
        }
        // ragged tail of fewer than 16 values
        const size_t t = 16 * nv + tid;
        if (t < n) dst[t] = widen1(src[t]);
    }
}

}  // namespace

cudaError_t ssd_launch_widen_fp8(const SsdWidenJobs &jobs, int num_sms, cudaStream_t stream) {
    size_t total = 0, vecs = 0;
    for (int j = 0; j < jobs.count; ++j) {
        total += jobs.job[j].n;
        vecs += jobs.job[j].n / 16;
    }
    if (total == 0) return cudaSuccess;
    // a few CTAs per SM; at least one, whose first 16 threads cover the tails
    const size_t want = (vecs + kWidenThreads - 1) / kWidenThreads;
    const size_t cap = (size_t)(num_sms > 0 ? num_sms : 1) * 8;
    const unsigned grid = (unsigned)(want == 0 ? 1 : (want < cap ? want : cap));
    ssd_fp8_widen_kernel<<<grid, kWidenThreads, 0, stream>>>(jobs);
    return cudaGetLastError();
}
