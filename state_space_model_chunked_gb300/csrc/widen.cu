// fp8 (E4M3) -> bfloat16 widening of prefill inputs.
//
// An fp8 prefill call widens x, B and C once into bfloat16 copies in its
// workspace, then runs the bf16 path on them.  Every E4M3 value (3
// significand bits, exponents 2^-9 .. 2^8) is exactly a bfloat16 value (7
// significand bits, fp32's exponent range), so the widening is exact; the
// conversion goes through the hardware E4M3x2 -> f16x2 convert (f16 holds
// every E4M3 value exactly too) and fp32.
//
// The kernel is HBM-bound: 1 byte read and 2 bytes written per value.  It
// makes one pass over its arrays, CTA after CTA in address order (a grid that
// strides over them instead reached 0.72 of the HBM copy rate; one pass
// reaches it): each thread widens two 8-value chunks 256 chunks apart, so a
// warp's load covers 256 contiguous bytes and its store 512.  Up to three
// arrays share one launch, each on its own run of CTAs.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "launch.h"

namespace {

constexpr int kWidenThreads = 256;
constexpr size_t kChunksPerCta = 2 * kWidenThreads;    // 8-value chunks per CTA

// 8 E4M3 values (8 bytes) -> 8 bfloat16 values (16 bytes)
__device__ __forceinline__ uint4 widen8(uint2 v) {
    const uint32_t w[2] = {v.x, v.y};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)(w[i] >> (16 * k));
            const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
            const __nv_bfloat162 b = __float22bfloat162_rn(f);
            o[2 * i + k] = *reinterpret_cast<const uint32_t *>(&b);
        }
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ __nv_bfloat16 widen1(uint8_t c) {
    const __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
    return __float2bfloat16_rn(__half2float(*reinterpret_cast<const __half *>(&hr)));
}

size_t ctas_of(size_t n) { return (n / 8 + kChunksPerCta - 1) / kChunksPerCta; }

// CTAs [first[j], first[j + 1]) widen job j; the job's first CTA also takes
// its ragged tail of fewer than 8 values
__global__ void __launch_bounds__(kWidenThreads)
ssd_fp8_widen_kernel(SsdWidenJobs jobs, SsdWidenFirst first) {
    const size_t cta = blockIdx.x;
    const int j = cta < first.cta[1] ? 0 : (cta < first.cta[2] ? 1 : 2);
    const SsdWidenJob job = j == 0 ? jobs.job[0] : (j == 1 ? jobs.job[1] : jobs.job[2]);
    const size_t n8 = job.n / 8;
    const size_t c0 = (cta - (j == 0 ? first.cta[0] : (j == 1 ? first.cta[1] : first.cta[2]))) *
                          kChunksPerCta + threadIdx.x;
    const size_t c1 = c0 + kWidenThreads;
    const uint2 *src = static_cast<const uint2 *>(job.src);
    uint4 *dst = static_cast<uint4 *>(job.dst);
    uint2 a = make_uint2(0u, 0u), b = make_uint2(0u, 0u);
    if (c0 < n8) a = __ldcs(src + c0);
    if (c1 < n8) b = __ldcs(src + c1);
    if (c0 < n8) dst[c0] = widen8(a);
    if (c1 < n8) dst[c1] = widen8(b);
    if (c0 < 8 && 8 * n8 + c0 < job.n) {
        const size_t t = 8 * n8 + c0;
        static_cast<__nv_bfloat16 *>(job.dst)[t] = widen1(static_cast<const uint8_t *>(job.src)[t]);
    }
}

}  // namespace

cudaError_t ssd_launch_widen_fp8(const SsdWidenJobs &jobs, cudaStream_t stream) {
    SsdWidenJobs js{};
    SsdWidenFirst first{};
    size_t total = 0;
    for (int j = 0; j < 3; ++j) {
        // unused slots are empty jobs of no CTAs
        js.job[j] = j < jobs.count ? jobs.job[j] : SsdWidenJob{nullptr, nullptr, 0};
        first.cta[j] = total;
        // a job with values but no whole chunk still needs a CTA for its tail
        total += js.job[j].n > 0 ? (ctas_of(js.job[j].n) > 0 ? ctas_of(js.job[j].n) : 1) : 0;
    }
    js.count = jobs.count;
    if (total == 0) return cudaSuccess;
    if (total > 0x7fffffffu) return cudaErrorInvalidValue;
    ssd_fp8_widen_kernel<<<(unsigned)total, kWidenThreads, 0, stream>>>(js, first);
    return cudaGetLastError();
}
