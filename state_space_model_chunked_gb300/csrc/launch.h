// Internal launchers behind the C ABI (include/ssd.h).  Arguments are
// validated by the ABI layer before any of these is called.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "common.cuh"

cudaError_t ssd_launch_decode(void *state, bool bf16_state, const void *x, const float *dt,
                              const float *A, const void *B, const void *C,
                              const float *D, void *y, bool bf16, int batch,
                              int H, int P, int N, int G, int num_sms, unsigned int *err,
                              const SsdFuse &fuse, cudaStream_t stream);

// ntok consecutive tokens per (batch, head) in one launch (state read and
// written once); headdim must not exceed ssd_decode_multi_max_headdim(N)
// (0 for an unsupported dstate).
cudaError_t ssd_launch_decode_multi(void *state, bool bf16_state, const void *x, const float *dt,
                                    const float *A, const void *B, const void *C,
                                    const float *D, void *y, bool bf16, int batch, int ntok,
                                    int H, int P, int N, int G, int num_sms, const SsdFuse &fuse,
                                    cudaStream_t stream);
int ssd_decode_multi_max_headdim(int N);

size_t ssd_simt_smem_bytes(int N);

// fp8 (E4M3) -> bfloat16 widening of up to three arrays in one launch; every
// pointer 16-byte aligned (the ABI checks the sources, the workspace
// carve-out aligns the destinations).
struct SsdWidenJob {
    const void *src;
    void *dst;
    size_t n;
};
struct SsdWidenJobs {
    SsdWidenJob job[3];
    int count;
};
struct SsdWidenFirst {     // first CTA of each job in the widening launch
    size_t cta[3];
};
cudaError_t ssd_launch_widen_fp8(const SsdWidenJobs &jobs, cudaStream_t stream);

// Sequence split over GPUs by tokens: a token range's log-decay A_h * sum dt
// ([batch][H], dt transformed as the scan does), and the chain of R ranges'
// contributions into each range's entering state ([R][batch][H][P][N]).
cudaError_t ssd_launch_range_log_decay(const float *dt, const float *A, int batch, int L, int H,
                                       const SsdFuse &fuse, float *out, cudaStream_t stream);
cudaError_t ssd_launch_chain_states(const float *contrib, const float *log_decay,
                                    const float *init, int R, int batch, int H, int P, int N,
                                    float *entering, cudaStream_t stream);

// Test hooks of the ABI layer: the fault to inject (0 = none) and the limit
// of every bounded device wait, read by the launchers at each launch.
struct SsdDebug {
    int fault;
    unsigned long long wait_ns;
};
SsdDebug ssd_debug_config();

// Events recorded around the kernel that writes y (null = none).
struct SsdProfileEvents {
    cudaEvent_t before, after;
};

// Records a profiling event on `stream`; inside stream capture it becomes an
// event-record node of the graph (an external record), not a capture-internal
// dependency.
inline cudaError_t ssd_record_event(cudaEvent_t ev, cudaStream_t stream) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &st);
    if (e != cudaSuccess) return e;
    if (st == cudaStreamCaptureStatusActive)
        return cudaEventRecordWithFlags(ev, stream, cudaEventRecordExternal);
    return cudaEventRecord(ev, stream);
}

cudaError_t ssd_launch_scan_simt(const void *x, const float *dt, const float *A,
                                 const void *B, const void *C, const float *D,
                                 const float *init, void *y, float *fin, bool bf16,
                                 int batch, int L, int H, int P, int N, int G,
                                 const SsdFuse &fuse, const int *cu, SsdProfileEvents prof,
                                 cudaStream_t stream);

// Tensor-core (tcgen05/TMEM/TMA) chunked scan.
struct SsdTcPlan {
    bool supported;
    int tiles;            // 128-token tiles per sequence (last may be ragged)
    int heads_per_cta;    // heads sharing one C.B^T product
    int seg_tiles;        // tiles per segment (the unit of sequence parallelism)
    int nseg;             // segments per sequence
    int seg_heads;        // heads per CTA of the segment-contribution kernel
    int seg_split;        // batched, seg_heads 4: segments launched at four heads per
                          // CTA (the rest at two, in a second launch); 0 = one launch
    size_t workspace;     // bytes of workspace required
    int launches;         // kernels enqueued per call
    // work items: sequences, segment contributions (every segment but each
    // sequence's last) and scan segments; batched plans have nseqs equal
    // sequences of `tiles` tiles, packed plans (varlen) per-sequence lengths
    bool varlen;
    int nseqs, nslots, items;
    size_t dt_offset;     // workspace bytes before the transformed step sizes
};

SsdTcPlan ssd_tc_plan(int batch, int L, int H, int P, int N, int G, int num_sms);
// Plan for nseq packed sequences, token offsets cu_host[0..nseq] (host copy).
SsdTcPlan ssd_tc_plan_varlen(int nseq, const int *cu_host, int H, int P, int N, int G,
                             int num_sms);

cudaError_t ssd_launch_scan_tc(const SsdTcPlan &plan, const void *x, const float *dt,
                               const float *A, const void *B, const void *C,
                               const float *D, const float *init, void *y, float *fin,
                               int batch, int L, int H, int P, int N, int G,
                               void *workspace, unsigned int *err, const SsdFuse &fuse,
                               SsdProfileEvents prof, cudaStream_t stream,
                               const int *cu_dev = nullptr);
