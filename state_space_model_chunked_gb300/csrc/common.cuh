// Shared device helpers for the SSD kernels (no arithmetic of the method).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

// Codes a kernel writes into the device error word (first writer wins).
enum : unsigned int {
    SSD_DEVERR_NONE = 0,
    SSD_DEVERR_TIMEOUT = 1,        // a bounded mbarrier / flag wait ran out
    SSD_DEVERR_SMEM_ALIGN = 2,     // dynamic shared memory not 1024-byte aligned
    SSD_DEVERR_TMEM = 3,           // tensor-memory allocation returned an unusable address
};

__device__ __forceinline__ void ssd_report(unsigned int *err, unsigned int code) {
    if (err) atomicCAS(err, 0u, code);
}

// Optional transform of the raw step size before it is used, the usual
// parameterisation of a positive step from the input projection's output:
//   dt <- clamp(sp(dt_raw + bias[h]), lo, hi),  sp = softplus when enabled,
// softplus(u) = log(1 + e^u) (u itself above 20, where they agree in fp32).
// bias = nullptr, softplus = 0, lo = -inf, hi = +inf is the identity.
struct SsdDt {
    const float *bias;
    int softplus;
    float lo, hi;
};

// Kernels are instantiated with and without the transform (kOn): its code,
// even untaken, costs the scan kernel a quarter of its speed, so the identity
// instantiation carries none of it.
template <bool kOn>
__device__ __forceinline__ float ssd_dt(const SsdDt &t, float raw, int h) {
    if constexpr (!kOn) {
        (void)t;
        (void)h;
        return raw;
    } else {
        float v = raw;
        if (t.bias) v += t.bias[h];
        if (t.softplus) v = v > 20.f ? v : log1pf(expf(v));
        return fminf(fmaxf(v, t.lo), t.hi);
    }
}

inline bool ssd_dt_active(const SsdDt &t) {
    return t.bias != nullptr || t.softplus != 0 || t.lo > -INFINITY || t.hi < INFINITY;
}

// Element loads/stores for the two input dtypes.
__device__ __forceinline__ float ssd_ld(const float *p) { return *p; }
__device__ __forceinline__ float ssd_ld(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void ssd_st(float *p, float v) { *p = v; }
__device__ __forceinline__ void ssd_st(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

// Four consecutive elements starting at a 4-element-aligned index.
__device__ __forceinline__ float4 ssd_ld4(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
__device__ __forceinline__ float4 ssd_ld4(const __nv_bfloat16 *p) {
    uint2 u = *reinterpret_cast<const uint2 *>(p);
    float4 r;
    r.x = __uint_as_float(u.x << 16);
    r.y = __uint_as_float(u.x & 0xffff0000u);
    r.z = __uint_as_float(u.y << 16);
    r.w = __uint_as_float(u.y & 0xffff0000u);
    return r;
}
