// Prefill scan for callers that cannot allocate device memory.
//
// Some callers are not allowed to call cudaMalloc when they run the scan:
// code whose memory plan is fixed at start-up (an inference engine plugin
// that is handed only its inputs and outputs), runtimes that forbid device
// allocation after initialisation, or code running where an allocation could
// block or fail mid-step.  ssd_scan_fwd needs a caller-provided workspace for
// long sequences; this entry point instead uses a fixed scratch array that
// lives in the library itself.
//
// The scratch is a file-scope __device__ array of SSD_STATIC_SCRATCH_BYTES.
// Every GPU that loads this library holds it until the process exits.  Host
// code cannot use the array's name as a device address, so the first call on
// each device looks up the real address with cudaGetSymbolAddress (with that
// device current) and caches it; that first call should therefore come
// before any stream capture.  All calls share the one array: calls whose
// kernels overlap on the GPU (different streams, no ordering between them)
// race on it.  Nothing in the scratch needs to start at zero: every element
// a call reads was written earlier in the same call.
#include <stdint.h>

#include <mutex>

#include "../../include/ssd.h"
#include "launch.h"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[SSD_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (looked up once
// per device), or nullptr on failure.
void *scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) return nullptr;
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" ssd_status ssd_scan_fwd_static(const void *x, const float *dt, const float *A,
                                          const void *B, const void *C, const float *D,
                                          ssd_dtype in_dtype, int batch, int seqlen, int nheads,
                                          int headdim, int dstate, int ngroups, int chunk,
                                          const float *init_state, void *y, float *final_state,
                                          cudaStream_t stream) {
    // this entry point takes no dt transform: the scratch it needs excludes
    // the transformed step sizes
    const size_t need = ssd_scan_fused_workspace_bytes(batch, seqlen, nheads, headdim, dstate,
                                                       ngroups, chunk, in_dtype, 0);
    if (need == (size_t)-1) return SSD_ERR_INVALID_ARG;
    if (need > (size_t)SSD_STATIC_SCRATCH_BYTES) return SSD_ERR_WORKSPACE;
    void *scratch = scratch_address();
    if (!scratch) return SSD_ERR_CUDA;
    return ssd_scan_fwd(x, dt, A, B, C, D, in_dtype, batch, seqlen, nheads, headdim, dstate,
                        ngroups, chunk, init_state, y, final_state, scratch,
                        (size_t)SSD_STATIC_SCRATCH_BYTES, stream);
}
