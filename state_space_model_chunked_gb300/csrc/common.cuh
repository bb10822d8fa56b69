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

// Limit of a bounded device-side wait unless the host sets another one
// (nanoseconds of the global timer).
constexpr unsigned long long kSsdDefaultWaitNs = 2000000000ull;
// Host-set fault injection for tests of the timeout path (ssd_fault in the C
// ABI): the tensor-core scan kernel's factor warp withholds its first signal.
constexpr int kSsdFaultWithholdSignal = 1;

// The neighbouring steps of a Mamba-2 layer fused into the kernels.
// Input side, the transform of the raw step size (the usual parameterisation
// of a positive step from the input projection's output):
//   dt <- clamp(sp(dt_raw + bias[h]), lo, hi),  sp = softplus when enabled,
// softplus(u) = log(1 + e^u) (u itself above 20, where they agree in fp32);
// bias = nullptr, softplus = 0, lo = -inf, hi = +inf is the identity.
// Output side, the gate: y <- y * silu(z), silu(z) = z / (1 + e^-z), with z
// (the input dtype, y's layout) from the same projection; nullptr = no gate.
struct SsdFuse {
    const float *bias;
    int softplus;
    float lo, hi;
    const void *z;
};

// softplus(u) = log(1 + e^u) = max(u, 0) + log1p(e^-|u|) from the hardware
// exponential and logarithm approximations: log1p(e) by its Taylor series
// e - e^2/2 + e^3/3 - e^4/4 below e = 1/16 (truncation below e^5/5, relative
// error under 3e-6), else log(1 + e), whose argument is then at least 1/16
// away from 1 (relative error near 1e-5).  A few instructions instead of the
// libm pair, for the single warps that compute per-token factors.
__device__ __forceinline__ float ssd_softplus_fast(float u) {
    const float e = __expf(-fabsf(u));
    const float l = e < 0.0625f ? e * (1.f - e * (0.5f - e * (0.33333334f - 0.25f * e)))
                                : __logf(1.f + e);
    return fmaxf(u, 0.f) + l;
}

// The transform's per-head bias, read once per kernel and head (0 without).
template <bool kOn>
__device__ __forceinline__ float ssd_dt_bias(const SsdFuse &t, int h) {
    if constexpr (!kOn) {
        (void)t;
        (void)h;
        return 0.f;
    } else {
        return t.bias ? t.bias[h] : 0.f;
    }
}

// Kernels are instantiated with and without these steps (kOn): their code,
// even untaken, costs the scan kernel a quarter of its speed, so the plain
// instantiation carries none of it.  kFast selects ssd_softplus_fast (the
// tensor-core kernels) over the libm form (fp32 paths).
template <bool kOn, bool kFast = false>
__device__ __forceinline__ float ssd_dt(const SsdFuse &t, float raw, float bias) {
    if constexpr (!kOn) {
        (void)t;
        (void)bias;
        return raw;
    } else {
        float v = raw + bias;
        if (t.softplus) {
            if constexpr (kFast) v = ssd_softplus_fast(v);
            else v = v > 20.f ? v : log1pf(expf(v));
        }
        return fminf(fmaxf(v, t.lo), t.hi);
    }
}

inline bool ssd_dt_transform_active(const SsdFuse &t) {
    return t.bias != nullptr || t.softplus != 0 || t.lo > -INFINITY || t.hi < INFINITY;
}
inline bool ssd_fuse_active(const SsdFuse &t) { return ssd_dt_transform_active(t) || t.z != nullptr; }

// silu(z) = z * sigmoid(z) = z / (1 + e^-z) with the hardware exponential and
// reciprocal approximations (relative error near 1e-6); for very negative z,
// e^-z overflows to inf and the quotient is 0.
__device__ __forceinline__ float ssd_silu(float z) { return __fdividef(z, 1.f + __expf(-z)); }

// Element loads/stores for the two input dtypes.
__device__ __forceinline__ float ssd_ld(const float *p) { return *p; }
__device__ __forceinline__ float ssd_ld(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void ssd_st(float *p, float v) { *p = v; }
__device__ __forceinline__ void ssd_st(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

// The output gate applied to y at flat element index i of the y layout.
template <bool kOn, typename T>
__device__ __forceinline__ float ssd_gate(const SsdFuse &f, float y, size_t i) {
    if constexpr (!kOn) {
        (void)f;
        (void)i;
        return y;
    } else {
        return f.z ? y * ssd_silu(ssd_ld(static_cast<const T *>(f.z) + i)) : y;
    }
}

// Four consecutive state elements stored as float or as bfloat16 (rounded to
// nearest even); the arithmetic is fp32 either way.
__device__ __forceinline__ void ssd_st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void ssd_st4(__nv_bfloat16 *p, float4 v) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t *>(&lo);
    u.y = *reinterpret_cast<const uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(p) = u;
}
// Streaming (evict-first) forms for state touched once per call.
__device__ __forceinline__ float4 ssd_ld4_cs(const float *p) {
    return __ldcs(reinterpret_cast<const float4 *>(p));
}
__device__ __forceinline__ float4 ssd_ld4_cs(const __nv_bfloat16 *p) {
    const uint2 u = __ldcs(reinterpret_cast<const uint2 *>(p));
    float4 r;
    r.x = __uint_as_float(u.x << 16);
    r.y = __uint_as_float(u.x & 0xffff0000u);
    r.z = __uint_as_float(u.y << 16);
    r.w = __uint_as_float(u.y & 0xffff0000u);
    return r;
}
__device__ __forceinline__ void ssd_st4_cs(float *p, float4 v) {
    __stcs(reinterpret_cast<float4 *>(p), v);
}
__device__ __forceinline__ void ssd_st4_cs(__nv_bfloat16 *p, float4 v) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t *>(&lo);
    u.y = *reinterpret_cast<const uint32_t *>(&hi);
    __stcs(reinterpret_cast<uint2 *>(p), u);
}

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
