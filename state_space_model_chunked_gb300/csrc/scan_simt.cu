// SIMT chunked SSD scan: exact fp32 FFMA arithmetic for any shape.
//
// The chunk steps are those of "Mamba-Family State-Space Model Kernels on a
// Programmable CGLA", section III.A: Step-1 inside a chunk is GEMM1 (C.B^T,
// reduction over the state size N), the Hadamard decay mask, and GEMM2
// (reduction over the chunk); Step-3 carries the N x P state across chunks
// sequentially.  Per chunk of T tokens starting at t0, with a_t the
// chunk-local inclusive cumulative sum of dt*A:
//
//   M[t][s]  = (C_t . B_s) * exp(a_t - a_s) * dt_s          (s <= t)
//   y_t[p]   = sum_s M[t][s] x_s[p] + exp(a_t) * C_t . H[p][:] + D x_t[p]
//   H[p][n] <- exp(a_end) * H[p][n] + sum_s exp(a_end - a_s) dt_s x_s[p] B_s[n]
//
// Exponents are always differences a_t - a_s <= 0 (never a ratio of two
// exponentials), so nothing overflows however long the decay runs.
//
// One CTA owns one (batch, head, block of PB state rows).  Rows of the state
// (and columns p of y) are independent given C, B and dt, so splitting P
// across CTAs multiplies the parallelism; the C.B^T product is recomputed by
// every CTA of a head, which is the price of that split on this path.  The
// state block stays in shared memory for the whole sequence.  The tile T is
// this kernel's own block size; the result does not depend on it.
#include "common.cuh"
#include "launch.h"

namespace {

constexpr int kT = 64;          // tokens per tile
constexpr int kPB = 16;         // state rows (headdim columns) per CTA
constexpr int kThreads = 256;
constexpr int kMS = kT + 16;    // row stride of the mask tile (bank spread)

struct SimtSmem {
    int np;                     // padded row stride of the C/B/H tiles (floats)
    size_t bytes;
};

__host__ __device__ inline int simt_np(int N) { return N + 4; }

__host__ inline size_t simt_smem_bytes(int N) {
    const int np = simt_np(N);
    return sizeof(float) * ((size_t)2 * kT * np + (size_t)kT * kPB + (size_t)kPB * np +
                            (size_t)kT * kMS + 4 * kT);
}

template <typename T, bool kFuse>
__global__ void __launch_bounds__(kThreads)
ssd_scan_simt_kernel(const T *__restrict__ x, const float *__restrict__ dt,
                     const float *__restrict__ A, const T *__restrict__ Bm,
                     const T *__restrict__ Cm, const float *__restrict__ D,
                     const float *__restrict__ init, T *__restrict__ y,
                     float *__restrict__ fin, int L, int H, int P, int N, int G,
                     const SsdFuse fuse, const int *__restrict__ cu) {
    extern __shared__ __align__(16) float sm[];
    const int np = simt_np(N);
    float *Cs = sm;                       // [kT][np]
    float *Bs = Cs + kT * np;             // [kT][np]
    float *Xs = Bs + kT * np;             // [kT][kPB]
    float *Hs = Xs + kT * kPB;            // [kPB][np]
    float *Ms = Hs + kPB * np;            // [kT][kMS]
    float *a_s = Ms + kT * kMS;           // [kT] chunk-local inclusive cumsum
    float *ea = a_s + kT;                 // [kT] exp(a_t)
    float *wS = ea + kT;                  // [kT] exp(a_end - a_s) * dt_s
    float *dts = wS + kT;                 // [kT] dt_s

    const int tid = threadIdx.x;
    const int p0 = blockIdx.x * kPB;
    const int h = blockIdx.y;
    const int b = blockIdx.z;             // sequence (a batch row, or one of cu's)
    // packed sequences: tokens cu[b] .. cu[b+1]-1 of the flattened token axis
    const size_t grow0 = cu ? (size_t)cu[b] : (size_t)b * L;
    const int Ls = cu ? cu[b + 1] - cu[b] : L;
    const int g = h / (H / G);
    const int pw = min(kPB, P - p0);
    const float Ah = A[h];
    const float dtb = ssd_dt_bias<kFuse>(fuse, h);
    const float Dh = D ? D[h] : 0.0f;
    const int nq = N / 4;

    // entering state
    for (int i = tid; i < kPB * nq; i += kThreads) {
        const int p = i / nq, n4 = (i - p * nq) * 4;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (init && p < pw)
            v = *reinterpret_cast<const float4 *>(init + (((size_t)b * H + h) * P + p0 + p) * N + n4);
        *reinterpret_cast<float4 *>(Hs + p * np + n4) = v;
    }

    for (int t0 = 0; t0 < Ls; t0 += kT) {
        const int len = min(kT, Ls - t0);
        __syncthreads();   // previous tile fully consumed
        // ---- load the tile: dt, C, B (all N), x (this CTA's PB columns)
        for (int i = tid; i < kT * nq; i += kThreads) {
            const int t = i / nq, n4 = (i - t * nq) * 4;
            float4 c = make_float4(0.f, 0.f, 0.f, 0.f), bb = c;
            if (t < len) {
                const size_t row = ((grow0 + t0 + t) * G + g) * N + n4;
                c = ssd_ld4(Cm + row);
                bb = ssd_ld4(Bm + row);
            }
            *reinterpret_cast<float4 *>(Cs + t * np + n4) = c;
            *reinterpret_cast<float4 *>(Bs + t * np + n4) = bb;
        }
        for (int i = tid; i < kT * kPB; i += kThreads) {
            const int t = i / kPB, p = i - t * kPB;
            float v = 0.f;
            if (t < len && p < pw) v = ssd_ld(x + ((grow0 + t0 + t) * H + h) * P + p0 + p);
            Xs[i] = v;
        }
        if (tid < 32) {
            // inclusive cumsum of dt*A over the tile: two tokens per lane
            const int ta = 2 * tid, tb = 2 * tid + 1;
            const float da = ta < len ? ssd_dt<kFuse>(fuse, dt[(grow0 + t0 + ta) * H + h], dtb) : 0.f;
            const float db = tb < len ? ssd_dt<kFuse>(fuse, dt[(grow0 + t0 + tb) * H + h], dtb) : 0.f;
            const float va = da * Ah, vb = db * Ah;
            float pair = va + vb;
            float incl = pair;
            for (int off = 1; off < 32; off <<= 1) {
                const float o = __shfl_up_sync(0xffffffffu, incl, off);
                if (tid >= off) incl += o;
            }
            const float excl = incl - pair;
            a_s[ta] = excl + va;
            a_s[tb] = excl + va + vb;
            dts[ta] = da;
            dts[tb] = db;
        }
        __syncthreads();
        const float a_end = a_s[len - 1];
        if (tid < kT) {
            ea[tid] = expf(a_s[tid]);
            wS[tid] = tid < len ? expf(a_end - a_s[tid]) * dts[tid] : 0.f;
        }
        // ---- GEMM1 + mask: M[t][s] for t = ty + 16i, s = tx + 16j
        {
            const int ty = tid / 16, tx = tid % 16;
            float acc[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
            for (int n = 0; n < N; n += 4) {
                float4 c[4], bv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) c[i] = *reinterpret_cast<const float4 *>(Cs + (ty + 16 * i) * np + n);
#pragma unroll
                for (int j = 0; j < 4; ++j) bv[j] = *reinterpret_cast<const float4 *>(Bs + (tx + 16 * j) * np + n);
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        acc[i][j] = fmaf(c[i].x, bv[j].x, acc[i][j]);
                        acc[i][j] = fmaf(c[i].y, bv[j].y, acc[i][j]);
                        acc[i][j] = fmaf(c[i].z, bv[j].z, acc[i][j]);
                        acc[i][j] = fmaf(c[i].w, bv[j].w, acc[i][j]);
                    }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int t = ty + 16 * i, s = tx + 16 * j;
                    float m = 0.f;
                    if (s <= t && t < len) m = acc[i][j] * expf(a_s[t] - a_s[s]) * dts[s];
                    Ms[t * kMS + s] = m;
                }
        }
        __syncthreads();
        // ---- outputs: intra-chunk GEMM2 + off-diagonal from the entering state + D skip
        {
            const int p = tid % 16;
            for (int t = tid / 16; t < len; t += 16) {
                float acc = 0.f;
                for (int s = 0; s <= t; ++s) acc = fmaf(Ms[t * kMS + s], Xs[s * kPB + p], acc);
                float off = 0.f;
                for (int n = 0; n < N; n += 4) {
                    const float4 c = *reinterpret_cast<const float4 *>(Cs + t * np + n);
                    const float4 hh = *reinterpret_cast<const float4 *>(Hs + p * np + n);
                    off = fmaf(c.x, hh.x, off);
                    off = fmaf(c.y, hh.y, off);
                    off = fmaf(c.z, hh.z, off);
                    off = fmaf(c.w, hh.w, off);
                }
                const float v = acc + ea[t] * off + Dh * Xs[t * kPB + p];
                if (p < pw) {
                    const size_t yi = ((grow0 + t0 + t) * H + h) * P + p0 + p;
                    ssd_st(y + yi, ssd_gate<kFuse, T>(fuse, v, yi));
                }
            }
        }
        __syncthreads();   // all reads of the entering state done
        // ---- Step-3: H <- exp(a_end) H + sum_s w_s x_s B_s^T
        {
            const float de = expf(a_end);
            for (int i = tid; i < kPB * nq; i += kThreads) {
                const int p = i / nq, n4 = (i - p * nq) * 4;
                float4 acc = *reinterpret_cast<const float4 *>(Hs + p * np + n4);
                acc.x *= de; acc.y *= de; acc.z *= de; acc.w *= de;
                for (int s = 0; s < len; ++s) {
                    const float wx = wS[s] * Xs[s * kPB + p];
                    const float4 bb = *reinterpret_cast<const float4 *>(Bs + s * np + n4);
                    acc.x = fmaf(wx, bb.x, acc.x);
                    acc.y = fmaf(wx, bb.y, acc.y);
                    acc.z = fmaf(wx, bb.z, acc.z);
                    acc.w = fmaf(wx, bb.w, acc.w);
                }
                *reinterpret_cast<float4 *>(Hs + p * np + n4) = acc;
            }
        }
    }
    __syncthreads();
    if (fin) {
        for (int i = tid; i < kPB * nq; i += kThreads) {
            const int p = i / nq, n4 = (i - p * nq) * 4;
            if (p < pw)
                *reinterpret_cast<float4 *>(fin + (((size_t)b * H + h) * P + p0 + p) * N + n4) =
                    *reinterpret_cast<const float4 *>(Hs + p * np + n4);
        }
    }
}

template <typename T, bool kFuse>
cudaError_t launch_t(const void *x, const float *dt, const float *A, const void *B,
                     const void *C, const float *D, const float *init, void *y,
                     float *fin, int batch, int L, int H, int P, int N, int G,
                     const SsdFuse &fuse, const int *cu, SsdProfileEvents prof,
                     cudaStream_t stream) {
    const size_t smem = simt_smem_bytes(N);
    cudaError_t e = cudaFuncSetAttribute(ssd_scan_simt_kernel<T, kFuse>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((P + kPB - 1) / kPB, H, batch);
    if (prof.before && prof.after && (e = ssd_record_event(prof.before, stream)) != cudaSuccess)
        return e;
    ssd_scan_simt_kernel<T, kFuse><<<grid, kThreads, smem, stream>>>(
        (const T *)x, dt, A, (const T *)B, (const T *)C, D, init, (T *)y, fin, L, H, P, N, G,
        fuse, cu);
    e = cudaGetLastError();
    if (e == cudaSuccess && prof.before && prof.after) e = ssd_record_event(prof.after, stream);
    return e;
}

}  // namespace

size_t ssd_simt_smem_bytes(int N) { return simt_smem_bytes(N); }

cudaError_t ssd_launch_scan_simt(const void *x, const float *dt, const float *A,
                                 const void *B, const void *C, const float *D,
                                 const float *init, void *y, float *fin, bool bf16,
                                 int batch, int L, int H, int P, int N, int G,
                                 const SsdFuse &fuse, const int *cu, SsdProfileEvents prof,
                                 cudaStream_t stream) {
    const bool fused = ssd_fuse_active(fuse);
    if (bf16)
        return fused ? launch_t<__nv_bfloat16, true>(x, dt, A, B, C, D, init, y, fin, batch, L, H,
                                                   P, N, G, fuse, cu, prof, stream)
                   : launch_t<__nv_bfloat16, false>(x, dt, A, B, C, D, init, y, fin, batch, L,
                                                    H, P, N, G, fuse, cu, prof, stream);
    return fused ? launch_t<float, true>(x, dt, A, B, C, D, init, y, fin, batch, L, H, P, N, G,
                                       fuse, cu, prof, stream)
               : launch_t<float, false>(x, dt, A, B, C, D, init, y, fin, batch, L, H, P, N, G,
                                        fuse, cu, prof, stream);
}
