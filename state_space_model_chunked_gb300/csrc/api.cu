// C ABI of libssd.so (declarations and contracts: include/ssd.h).
//
// This layer validates every argument on the host, picks the kernel path,
// and enqueues launches on the caller's stream.  It never allocates device
// memory and never synchronises (except ssd_last_device_error, which must).
#include <stdint.h>
#include <stdio.h>

#include "../../include/ssd.h"
#include "common.cuh"
#include "launch.h"

namespace {

// One error word per device: kernels report self-detected faults here.
__device__ unsigned int g_ssd_device_error;

constexpr int kMaxDevices = 64;
unsigned int *g_err_ptr[kMaxDevices];   // cached device address per device ordinal

unsigned int *device_error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    unsigned int *p = __atomic_load_n(&g_err_ptr[dev], __ATOMIC_ACQUIRE);
    if (p) return p;
    void *addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_ssd_device_error) != cudaSuccess) return nullptr;
    __atomic_store_n(&g_err_ptr[dev], (unsigned int *)addr, __ATOMIC_RELEASE);
    return (unsigned int *)addr;
}

int current_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

SsdProfileEvents g_profile = {nullptr, nullptr};
// test hooks (ssd_debug_inject_fault): written by the host between calls
SsdDebug g_debug = {0, kSsdDefaultWaitNs};

bool valid_chunk(int q) {
    return q == 16 || q == 32 || q == 64 || q == 128 || q == 256;
}

bool pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

ssd_status check_scan_args(const void *x, const float *dt, const float *A, const void *B,
                           const void *C, const float *D, ssd_dtype dtype, int batch,
                           int L, int H, int P, int N, int G, int chunk,
                           const float *init, const void *y, const float *fin) {
    if (!x || !dt || !A || !B || !C || !y) return SSD_ERR_INVALID_ARG;
    if (dtype != SSD_F32 && dtype != SSD_BF16 && dtype != SSD_FP8_E4M3) return SSD_ERR_INVALID_ARG;
    if (batch <= 0 || L <= 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0) return SSD_ERR_INVALID_ARG;
    if (H % G != 0) return SSD_ERR_INVALID_ARG;
    if (!valid_chunk(chunk)) return SSD_ERR_INVALID_ARG;
    if (N % 4 != 0 || N > 256) return SSD_ERR_UNSUPPORTED;
    const void *ptrs[] = {x, dt, A, B, C, D, init, y, fin};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return SSD_ERR_INVALID_ARG;
    if ((size_t)batch * L * H * P >= ((size_t)1 << 40)) return SSD_ERR_UNSUPPORTED;
    return SSD_OK;
}

// The device-side form of a caller's dt transform; NULL is the identity.
ssd_status dt_transform_of(const ssd_dt_transform *t, SsdFuse *out) {
    out->bias = nullptr;
    out->softplus = 0;
    out->lo = -INFINITY;
    out->hi = INFINITY;
    out->z = nullptr;
    if (!t) return SSD_OK;
    if (!(t->dt_min <= t->dt_max)) return SSD_ERR_INVALID_ARG;   // also rejects NaN
    out->bias = t->dt_bias;
    out->softplus = t->softplus != 0;
    out->lo = t->dt_min;
    out->hi = t->dt_max;
    return SSD_OK;
}

// Packed sequence offsets: nseq + 1 host ints from 0, non-decreasing, the
// total within the int range the kernels index tokens with.
ssd_status check_cu(int nseq, const int *cu) {
    if (nseq <= 0 || !cu || cu[0] != 0) return SSD_ERR_INVALID_ARG;
    for (int s = 0; s < nseq; ++s)
        if (cu[s + 1] < cu[s]) return SSD_ERR_INVALID_ARG;
    return SSD_OK;
}

// Workspace carve-out of an fp8 call: bfloat16 copies of x, B and C (each
// rounded up to 256 bytes) in front of the bf16 call's own workspace.
struct Fp8Copies {
    size_t b_off, c_off, total;
};
Fp8Copies fp8_copies(size_t rows, int H, int P, int G, int N) {
    auto up = [](size_t v) { return (v + 255) / 256 * 256; };
    Fp8Copies c;
    c.b_off = up(rows * (size_t)H * P * 2);
    c.c_off = c.b_off + up(rows * (size_t)G * N * 2);
    c.total = c.c_off + up(rows * (size_t)G * N * 2);
    return c;
}

ssd_status scan_any(ssd_algo algo, const void *x, const float *dt, const float *A,
                    const void *B, const void *C, const float *D,
                    const ssd_dt_transform *dt_transform, const void *z, ssd_dtype in_dtype,
                    int batch, int L, int nheads, int headdim, int dstate, int ngroups, int chunk,
                    const int *cu_host, const int *cu_dev, const float *init_state, void *y,
                    float *final_state, void *workspace, size_t workspace_bytes,
                    cudaStream_t stream, bool launch = true);

// fp8 inputs: x, B and C widened to bfloat16 copies at the front of the
// workspace, then the bf16 call on the copies with the rest of it.  Every
// check of that call runs before the widening is enqueued.
ssd_status scan_fp8(ssd_algo algo, const void *x, const float *dt, const float *A,
                    const void *B, const void *C, const float *D,
                    const ssd_dt_transform *dt_transform, const void *z, int batch, int L,
                    int nheads, int headdim, int dstate, int ngroups, int chunk,
                    const int *cu_host, const int *cu_dev, const float *init_state, void *y,
                    float *final_state, void *workspace, size_t workspace_bytes,
                    cudaStream_t stream) {
    const bool packed = cu_host != nullptr;
    const size_t rows = packed ? (size_t)L : (size_t)batch * L;
    if (rows == 0)   // a packed batch of empty sequences: no token values to widen
        return scan_any(algo, x, dt, A, B, C, D, dt_transform, z, SSD_BF16, batch, L, nheads,
                        headdim, dstate, ngroups, chunk, cu_host, cu_dev, init_state, y,
                        final_state, workspace, workspace_bytes, stream);
    ssd_status st = check_scan_args(x, dt, A, B, C, D, SSD_FP8_E4M3, packed ? 1 : batch, L,
                                    nheads, headdim, dstate, ngroups, chunk, init_state, y,
                                    final_state);
    if (st != SSD_OK) return st;
    const Fp8Copies cp = fp8_copies(rows, nheads, headdim, ngroups, dstate);
    if (!workspace || workspace_bytes < cp.total) return SSD_ERR_WORKSPACE;
    if (((uintptr_t)workspace & 255u) != 0) return SSD_ERR_INVALID_ARG;
    char *ws = static_cast<char *>(workspace);
    void *x16 = ws, *b16 = ws + cp.b_off, *c16 = ws + cp.c_off;
    void *rest = workspace_bytes > cp.total ? ws + cp.total : nullptr;
    const size_t rest_bytes = workspace_bytes - cp.total;
    st = scan_any(algo, x16, dt, A, b16, c16, D, dt_transform, z, SSD_BF16, batch, L, nheads,
                  headdim, dstate, ngroups, chunk, cu_host, cu_dev, init_state, y, final_state,
                  rest, rest_bytes, stream, false);
    if (st != SSD_OK) return st;
    SsdWidenJobs jobs{};
    jobs.job[0] = {x, x16, rows * (size_t)nheads * headdim};
    jobs.job[1] = {B, b16, rows * (size_t)ngroups * dstate};
    jobs.job[2] = {C, c16, rows * (size_t)ngroups * dstate};
    jobs.count = 3;
    if (ssd_launch_widen_fp8(jobs, stream) != cudaSuccess) return SSD_ERR_CUDA;
    return scan_any(algo, x16, dt, A, b16, c16, D, dt_transform, z, SSD_BF16, batch, L, nheads,
                    headdim, dstate, ngroups, chunk, cu_host, cu_dev, init_state, y, final_state,
                    rest, rest_bytes, stream);
}

// Both scan entry points: batched (cu_host == NULL; `batch` rows of `L`
// tokens) and packed (`batch` sequences on one axis of L = cu_host[batch]).
// With launch == false every check runs and nothing is enqueued.
ssd_status scan_any(ssd_algo algo, const void *x, const float *dt, const float *A,
                    const void *B, const void *C, const float *D,
                    const ssd_dt_transform *dt_transform, const void *z, ssd_dtype in_dtype,
                    int batch, int L, int nheads, int headdim, int dstate, int ngroups, int chunk,
                    const int *cu_host, const int *cu_dev, const float *init_state, void *y,
                    float *final_state, void *workspace, size_t workspace_bytes,
                    cudaStream_t stream, bool launch) {
    if (in_dtype == SSD_FP8_E4M3)
        return scan_fp8(algo, x, dt, A, B, C, D, dt_transform, z, batch, L, nheads, headdim,
                        dstate, ngroups, chunk, cu_host, cu_dev, init_state, y, final_state,
                        workspace, workspace_bytes, stream);
    const bool packed = cu_host != nullptr;
    // an all-empty packed batch has no token rows (the token arrays may be
    // NULL): only final states are written
    const bool rowless = packed && L == 0;
    const void *tok = A;   // stands in for absent token arrays in the checks
    ssd_status st = check_scan_args(rowless && !x ? tok : x, rowless && !dt ? A : dt, A,
                                    rowless && !B ? tok : B, rowless && !C ? tok : C, D,
                                    in_dtype, packed ? 1 : batch, rowless ? 1 : L, nheads,
                                    headdim, dstate, ngroups, chunk, init_state,
                                    rowless && !y ? tok : y, final_state);
    if (st != SSD_OK) return st;
    if (z && !aligned16(z)) return SSD_ERR_INVALID_ARG;
    SsdFuse fuse;
    if ((st = dt_transform_of(dt_transform, &fuse)) != SSD_OK) return st;
    fuse.z = z;
    if (algo != SSD_ALGO_AUTO && algo != SSD_ALGO_SIMT && algo != SSD_ALGO_TCGEN05)
        return SSD_ERR_INVALID_ARG;
    const bool bf16 = in_dtype == SSD_BF16;
    bool use_tc = false;
    SsdTcPlan plan{};
    if (algo != SSD_ALGO_SIMT && bf16) {
        plan = packed ? ssd_tc_plan_varlen(batch, cu_host, nheads, headdim, dstate, ngroups,
                                           current_sm_count())
                      : ssd_tc_plan(batch, L, nheads, headdim, dstate, ngroups,
                                    current_sm_count());
        use_tc = plan.supported;
    }
    if (algo == SSD_ALGO_TCGEN05 && !use_tc) return SSD_ERR_UNSUPPORTED;
    if (!use_tc && batch > 65535) return SSD_ERR_UNSUPPORTED;   // grid z: one per sequence
    cudaError_t e;
    if (use_tc) {
        // the transformed step sizes take the workspace's last region, needed
        // only with a dt transform
        const size_t need = ssd_dt_transform_active(fuse) ? plan.workspace : plan.dt_offset;
        if (need > 0) {
            if (!workspace || workspace_bytes < need) return SSD_ERR_WORKSPACE;
            if (((uintptr_t)workspace & 255u) != 0) return SSD_ERR_INVALID_ARG;
        }
        if (!launch) return SSD_OK;
        e = ssd_launch_scan_tc(plan, x, dt, A, B, C, D, init_state, y, final_state, batch, L,
                               nheads, headdim, dstate, ngroups, workspace, device_error_word(),
                               fuse, g_profile, stream, cu_dev);
    } else {
        if (!launch) return SSD_OK;
        e = ssd_launch_scan_simt(x, dt, A, B, C, D, init_state, y, final_state, bf16, batch, L,
                                 nheads, headdim, dstate, ngroups, fuse, cu_dev, g_profile,
                                 stream);
    }
    return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

// Workspace of one batched call on the current device: the tensor-core
// plan's segment states and decays, plus the transformed step sizes only for
// a call with a dt transform; fp32 inputs take the SIMT path, which needs none.
size_t scan_workspace(int batch, int seqlen, int nheads, int headdim, int dstate, int ngroups,
                      int chunk, ssd_dtype in_dtype, bool with_dt) {
    if (batch <= 0 || seqlen <= 0 || nheads <= 0 || headdim <= 0 || dstate <= 0 ||
        ngroups <= 0 || nheads % ngroups != 0 || !valid_chunk(chunk))
        return (size_t)-1;
    if (in_dtype == SSD_FP8_E4M3)
        return fp8_copies((size_t)batch * seqlen, nheads, headdim, ngroups, dstate).total +
               scan_workspace(batch, seqlen, nheads, headdim, dstate, ngroups, chunk, SSD_BF16,
                              with_dt);
    if (in_dtype != SSD_BF16) return 0;
    const SsdTcPlan plan = ssd_tc_plan(batch, seqlen, nheads, headdim, dstate, ngroups,
                                       current_sm_count());
    if (!plan.supported) return 0;
    return with_dt ? plan.workspace : plan.dt_offset;
}

}  // namespace

SsdDebug ssd_debug_config() { return g_debug; }

extern "C" {

const char *ssd_status_string(ssd_status s) {
    switch (s) {
        case SSD_OK: return "SSD_OK";
        case SSD_ERR_INVALID_ARG: return "SSD_ERR_INVALID_ARG: invalid argument";
        case SSD_ERR_UNSUPPORTED: return "SSD_ERR_UNSUPPORTED: shape not handled by this kernel";
        case SSD_ERR_CUDA: return "SSD_ERR_CUDA: CUDA runtime or launch failure";
        case SSD_ERR_TIMEOUT: return "SSD_ERR_TIMEOUT: a bounded device-side wait ran out";
        case SSD_ERR_WORKSPACE: return "SSD_ERR_WORKSPACE: workspace missing or too small";
    }
    return "SSD_ERR_UNKNOWN";
}

ssd_status ssd_scan_profile_events(cudaEvent_t before, cudaEvent_t after) {
    g_profile.before = before;
    g_profile.after = after;
    return SSD_OK;
}

ssd_status ssd_last_device_error(void) {
    unsigned int *p = device_error_word();
    if (!p) return SSD_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return SSD_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return SSD_ERR_CUDA;
    const unsigned int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return SSD_ERR_CUDA;
    if (v == SSD_DEVERR_NONE) return SSD_OK;
    if (v == SSD_DEVERR_TIMEOUT) return SSD_ERR_TIMEOUT;
    return SSD_ERR_CUDA;
}

size_t ssd_scan_workspace_bytes(int batch, int seqlen, int nheads, int headdim, int dstate,
                                int ngroups, int chunk) {
    return scan_workspace(batch, seqlen, nheads, headdim, dstate, ngroups, chunk, SSD_BF16,
                          false);
}

size_t ssd_scan_fused_workspace_bytes(int batch, int seqlen, int nheads, int headdim,
                                      int dstate, int ngroups, int chunk, ssd_dtype in_dtype,
                                      int with_dt_transform) {
    return scan_workspace(batch, seqlen, nheads, headdim, dstate, ngroups, chunk, in_dtype,
                          with_dt_transform != 0);
}

ssd_status ssd_fp8_e4m3_to_bf16(const void *src, void *dst, size_t n, cudaStream_t stream) {
    if (n == 0) return SSD_OK;
    if (!src || !dst || !aligned16(src) || !aligned16(dst)) return SSD_ERR_INVALID_ARG;
    SsdWidenJobs jobs{};
    jobs.job[0] = {src, dst, n};
    jobs.count = 1;
    return ssd_launch_widen_fp8(jobs, stream) == cudaSuccess ? SSD_OK
                                                                                 : SSD_ERR_CUDA;
}

ssd_status ssd_range_log_decay(const float *dt, const float *A,
                               const ssd_dt_transform *dt_transform, int batch, int seqlen,
                               int nheads, float *log_decay, cudaStream_t stream) {
    if (!dt || !A || !log_decay) return SSD_ERR_INVALID_ARG;
    if (batch <= 0 || seqlen <= 0 || nheads <= 0) return SSD_ERR_INVALID_ARG;
    if ((nheads + 31) / 32 > 65535) return SSD_ERR_UNSUPPORTED;   // grid rows of 32 heads
    SsdFuse fuse;
    const ssd_status st = dt_transform_of(dt_transform, &fuse);
    if (st != SSD_OK) return st;
    return ssd_launch_range_log_decay(dt, A, batch, seqlen, nheads, fuse, log_decay, stream) ==
                   cudaSuccess
               ? SSD_OK
               : SSD_ERR_CUDA;
}

ssd_status ssd_chain_states(const float *contrib, const float *log_decay, const float *init,
                            int nranges, int batch, int nheads, int headdim, int dstate,
                            float *entering, cudaStream_t stream) {
    if (!contrib || !log_decay || !entering) return SSD_ERR_INVALID_ARG;
    if (nranges <= 0 || batch <= 0 || nheads <= 0 || headdim <= 0 || dstate <= 0)
        return SSD_ERR_INVALID_ARG;
    if ((size_t)batch * nheads * headdim * dstate >= ((size_t)1 << 38)) return SSD_ERR_UNSUPPORTED;
    return ssd_launch_chain_states(contrib, log_decay, init, nranges, batch, nheads, headdim,
                                   dstate, entering, stream) == cudaSuccess
               ? SSD_OK
               : SSD_ERR_CUDA;
}

ssd_status ssd_debug_inject_fault(ssd_fault fault, unsigned long long wait_limit_ns) {
    if (fault != SSD_FAULT_NONE && fault != SSD_FAULT_WITHHOLD_SIGNAL) return SSD_ERR_INVALID_ARG;
    g_debug.fault = (int)fault;
    g_debug.wait_ns = wait_limit_ns ? wait_limit_ns : kSsdDefaultWaitNs;
    return SSD_OK;
}

int ssd_scan_kernel_launches(int batch, int seqlen, int nheads, int headdim, int dstate,
                             int ngroups, int chunk, ssd_dtype in_dtype) {
    if (batch <= 0 || seqlen <= 0 || nheads <= 0 || headdim <= 0 || dstate <= 0 ||
        ngroups <= 0 || nheads % ngroups != 0 || !valid_chunk(chunk))
        return -1;
    if (in_dtype == SSD_FP8_E4M3)   // the widening, then the bf16 call
        return 1 + ssd_scan_kernel_launches(batch, seqlen, nheads, headdim, dstate, ngroups,
                                            chunk, SSD_BF16);
    if (in_dtype != SSD_BF16) return 1;
    const SsdTcPlan plan = ssd_tc_plan(batch, seqlen, nheads, headdim, dstate, ngroups,
                                       current_sm_count());
    return plan.supported ? plan.launches : 1;
}

ssd_status ssd_scan_fwd_fused(ssd_algo algo, const void *x, const float *dt, const float *A,
                              const void *B, const void *C, const float *D,
                              const ssd_dt_transform *dt_transform, const void *z,
                              ssd_dtype in_dtype, int batch, int seqlen, int nheads, int headdim,
                              int dstate, int ngroups, int chunk, const float *init_state,
                              void *y, float *final_state, void *workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
    return scan_any(algo, x, dt, A, B, C, D, dt_transform, z, in_dtype, batch, seqlen, nheads,
                    headdim, dstate, ngroups, chunk, nullptr, nullptr, init_state, y,
                    final_state, workspace, workspace_bytes, stream);
}

ssd_status ssd_scan_fwd_dt(ssd_algo algo, const void *x, const float *dt, const float *A,
                           const void *B, const void *C, const float *D,
                           const ssd_dt_transform *dt_transform, ssd_dtype in_dtype, int batch,
                           int seqlen, int nheads, int headdim, int dstate, int ngroups,
                           int chunk, const float *init_state, void *y, float *final_state,
                           void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    return ssd_scan_fwd_fused(algo, x, dt, A, B, C, D, dt_transform, nullptr, in_dtype, batch,
                              seqlen, nheads, headdim, dstate, ngroups, chunk, init_state, y,
                              final_state, workspace, workspace_bytes, stream);
}

size_t ssd_scan_varlen_workspace_bytes(int nseq, const int *cu_seqlens_host, int nheads,
                                       int headdim, int dstate, int ngroups, int chunk,
                                       ssd_dtype in_dtype) {
    if (check_cu(nseq, cu_seqlens_host) != SSD_OK || nheads <= 0 || headdim <= 0 ||
        dstate <= 0 || ngroups <= 0 || nheads % ngroups != 0 || !valid_chunk(chunk))
        return (size_t)-1;
    if (in_dtype == SSD_FP8_E4M3) {
        const size_t rows = (size_t)cu_seqlens_host[nseq];
        return (rows ? fp8_copies(rows, nheads, headdim, ngroups, dstate).total : 0) +
               ssd_scan_varlen_workspace_bytes(nseq, cu_seqlens_host, nheads, headdim, dstate,
                                               ngroups, chunk, SSD_BF16);
    }
    if (in_dtype != SSD_BF16) return 0;
    const SsdTcPlan plan = ssd_tc_plan_varlen(nseq, cu_seqlens_host, nheads, headdim, dstate,
                                              ngroups, current_sm_count());
    return plan.supported ? plan.workspace : 0;
}

int ssd_scan_varlen_kernel_launches(int nseq, const int *cu_seqlens_host, int nheads,
                                    int headdim, int dstate, int ngroups, int chunk,
                                    ssd_dtype in_dtype) {
    if (check_cu(nseq, cu_seqlens_host) != SSD_OK || nheads <= 0 || headdim <= 0 ||
        dstate <= 0 || ngroups <= 0 || nheads % ngroups != 0 || !valid_chunk(chunk))
        return -1;
    if (in_dtype == SSD_FP8_E4M3)   // the widening (when there are tokens), then the bf16 call
        return (cu_seqlens_host[nseq] > 0 ? 1 : 0) +
               ssd_scan_varlen_kernel_launches(nseq, cu_seqlens_host, nheads, headdim, dstate,
                                               ngroups, chunk, SSD_BF16);
    if (in_dtype != SSD_BF16) return 1;
    const SsdTcPlan plan = ssd_tc_plan_varlen(nseq, cu_seqlens_host, nheads, headdim, dstate,
                                              ngroups, current_sm_count());
    return plan.supported ? plan.launches : 1;
}

ssd_status ssd_scan_fwd_varlen(ssd_algo algo, const void *x, const float *dt, const float *A,
                               const void *B, const void *C, const float *D,
                               const ssd_dt_transform *dt_transform, const void *z,
                               ssd_dtype in_dtype, int nseq, const int *cu_seqlens_host,
                               const int *cu_seqlens_dev, int nheads, int headdim, int dstate,
                               int ngroups, int chunk, const float *init_state, void *y,
                               float *final_state, void *workspace, size_t workspace_bytes,
                               cudaStream_t stream) {
    ssd_status st = check_cu(nseq, cu_seqlens_host);
    if (st != SSD_OK) return st;
    if (!cu_seqlens_dev || ((uintptr_t)cu_seqlens_dev & 3u) != 0) return SSD_ERR_INVALID_ARG;
    return scan_any(algo, x, dt, A, B, C, D, dt_transform, z, in_dtype, nseq,
                    cu_seqlens_host[nseq], nheads, headdim, dstate, ngroups, chunk,
                    cu_seqlens_host, cu_seqlens_dev, init_state, y, final_state, workspace,
                    workspace_bytes, stream);
}

ssd_status ssd_scan_fwd_algo(ssd_algo algo, const void *x, const float *dt, const float *A,
                             const void *B, const void *C, const float *D,
                             ssd_dtype in_dtype, int batch, int seqlen, int nheads,
                             int headdim, int dstate, int ngroups, int chunk,
                             const float *init_state, void *y, float *final_state,
                             void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    return ssd_scan_fwd_dt(algo, x, dt, A, B, C, D, nullptr, in_dtype, batch, seqlen, nheads,
                           headdim, dstate, ngroups, chunk, init_state, y, final_state,
                           workspace, workspace_bytes, stream);
}

ssd_status ssd_scan_fwd(const void *x, const float *dt, const float *A, const void *B,
                        const void *C, const float *D, ssd_dtype in_dtype, int batch,
                        int seqlen, int nheads, int headdim, int dstate, int ngroups,
                        int chunk, const float *init_state, void *y, float *final_state,
                        void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    return ssd_scan_fwd_algo(SSD_ALGO_AUTO, x, dt, A, B, C, D, in_dtype, batch, seqlen,
                             nheads, headdim, dstate, ngroups, chunk, init_state, y,
                             final_state, workspace, workspace_bytes, stream);
}

ssd_status ssd_state_update_fused(void *state, ssd_dtype state_dtype, const void *x,
                                  const float *dt, const float *A, const void *B, const void *C,
                                  const float *D, const ssd_dt_transform *dt_transform,
                                  const void *z, ssd_dtype in_dtype, int batch, int nheads,
                                  int headdim, int dstate, int ngroups, void *y,
                                  cudaStream_t stream) {
    if (!state || !x || !dt || !A || !B || !C || !y) return SSD_ERR_INVALID_ARG;
    if (in_dtype == SSD_FP8_E4M3) return SSD_ERR_UNSUPPORTED;   // prefill only
    if (in_dtype != SSD_F32 && in_dtype != SSD_BF16) return SSD_ERR_INVALID_ARG;
    if (state_dtype != SSD_F32 && state_dtype != SSD_BF16) return SSD_ERR_INVALID_ARG;
    if (batch <= 0 || nheads <= 0 || headdim <= 0 || dstate <= 0 || ngroups <= 0)
        return SSD_ERR_INVALID_ARG;
    if (nheads % ngroups != 0) return SSD_ERR_INVALID_ARG;
    if (!pow2(dstate) || dstate < 4 || dstate > 256) return SSD_ERR_UNSUPPORTED;
    if (state_dtype == SSD_BF16 && in_dtype != SSD_BF16) return SSD_ERR_UNSUPPORTED;
    const void *ptrs[] = {state, x, dt, A, B, C, D, y, z};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return SSD_ERR_INVALID_ARG;
    if ((size_t)batch * nheads >= ((size_t)1 << 31)) return SSD_ERR_UNSUPPORTED;
    SsdFuse fuse;
    const ssd_status st = dt_transform_of(dt_transform, &fuse);
    if (st != SSD_OK) return st;
    fuse.z = z;
    cudaError_t e = ssd_launch_decode(state, state_dtype == SSD_BF16, x, dt, A, B, C, D, y,
                                      in_dtype == SSD_BF16, batch, nheads, headdim, dstate,
                                      ngroups, current_sm_count(), device_error_word(), fuse,
                                      stream);
    return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status ssd_state_update_multi(void *state, ssd_dtype state_dtype, const void *x,
                                  const float *dt, const float *A, const void *B, const void *C,
                                  const float *D, const ssd_dt_transform *dt_transform,
                                  const void *z, ssd_dtype in_dtype, int batch, int ntokens,
                                  int nheads, int headdim, int dstate, int ngroups, void *y,
                                  cudaStream_t stream) {
    if (!state || !x || !dt || !A || !B || !C || !y) return SSD_ERR_INVALID_ARG;
    if (in_dtype == SSD_FP8_E4M3) return SSD_ERR_UNSUPPORTED;   // prefill only
    if (in_dtype != SSD_F32 && in_dtype != SSD_BF16) return SSD_ERR_INVALID_ARG;
    if (state_dtype != SSD_F32 && state_dtype != SSD_BF16) return SSD_ERR_INVALID_ARG;
    if (batch <= 0 || ntokens <= 0 || nheads <= 0 || headdim <= 0 || dstate <= 0 ||
        ngroups <= 0)
        return SSD_ERR_INVALID_ARG;
    if (nheads % ngroups != 0) return SSD_ERR_INVALID_ARG;
    if (!pow2(dstate) || dstate < 4 || dstate > 256) return SSD_ERR_UNSUPPORTED;
    if (headdim > ssd_decode_multi_max_headdim(dstate)) return SSD_ERR_UNSUPPORTED;
    if (state_dtype == SSD_BF16 && in_dtype != SSD_BF16) return SSD_ERR_UNSUPPORTED;
    const void *ptrs[] = {state, x, dt, A, B, C, D, y, z};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return SSD_ERR_INVALID_ARG;
    if ((size_t)batch * nheads >= ((size_t)1 << 31)) return SSD_ERR_UNSUPPORTED;
    if ((size_t)batch * ntokens * nheads * headdim >= ((size_t)1 << 40)) return SSD_ERR_UNSUPPORTED;
    SsdFuse fuse;
    const ssd_status st = dt_transform_of(dt_transform, &fuse);
    if (st != SSD_OK) return st;
    fuse.z = z;
    cudaError_t e = ssd_launch_decode_multi(state, state_dtype == SSD_BF16, x, dt, A, B, C, D, y,
                                            in_dtype == SSD_BF16, batch, ntokens, nheads,
                                            headdim, dstate, ngroups, current_sm_count(), fuse,
                                            stream);
    return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status ssd_state_update_dt(float *state, const void *x, const float *dt, const float *A,
                               const void *B, const void *C, const float *D,
                               const ssd_dt_transform *dt_transform, ssd_dtype in_dtype,
                               int batch, int nheads, int headdim, int dstate, int ngroups,
                               void *y, cudaStream_t stream) {
    return ssd_state_update_fused(state, SSD_F32, x, dt, A, B, C, D, dt_transform, nullptr,
                                  in_dtype, batch, nheads, headdim, dstate, ngroups, y, stream);
}

ssd_status ssd_state_update(float *state, const void *x, const float *dt, const float *A,
                            const void *B, const void *C, const float *D, ssd_dtype in_dtype,
                            int batch, int nheads, int headdim, int dstate, int ngroups,
                            void *y, cudaStream_t stream) {
    return ssd_state_update_dt(state, x, dt, A, B, C, D, nullptr, in_dtype, batch, nheads,
                               headdim, dstate, ngroups, y, stream);
}

}  // extern "C"
