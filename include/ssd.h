/*
 * ssd.h -- C ABI of libssd.so, the GB300 (sm_103a) Mamba-2 state-space-duality
 * (SSD) hot path: the chunked scan for prefill and the single-token state
 * update for decode.
 *
 * Where the operations come from:
 *   - "Mamba-Family State-Space Model Kernels on a Programmable CGLA",
 *     section III.A (Mamba-2 layer with three kernel shapes): SSD Step-1 is
 *     GEMM1 (reduction over the state size N) -> Hadamard mask -> GEMM2
 *     (reduction over the chunk length Q); Step-3 updates the recurrent state
 *     h sequentially across chunks, with an input-dependent diagonal
 *     transition A_c; section III.C: the per-chunk recurrence is an N x d
 *     product (128 x 64 for Mamba-370M).
 *   - "Compiler-First State Space Duality and Portable O(1) Autoregressive
 *     Caching for Inference", abstract: diagonal per-head dynamics,
 *     fixed-size chunking, and an O(1) cached decode step.
 *   - "Mambalaya: Einsum-Based Fusion Optimizations on State-Space Models",
 *     abstract and Figures 4-5: fuse neighbouring Einsums so intermediates
 *     do not round-trip off-chip memory.
 *
 * The recurrence, for each batch row b and head h (group g = h / (H / G)):
 *     h_t = exp(dt_t * A_h) * h_{t-1} + dt_t * B_t x_t^T      (state N x P)
 *     y_t = C_t . h_t + D_h * x_t                             (uses updated h)
 * with h_{-1} = init_state (or zero) and final_state = h_{L-1}.  dt is used
 * exactly as given unless a call passes a dt transform (ssd_dt_transform);
 * the fused entry points can also gate y by silu(z).
 *
 * Layouts (row-major, contiguous, element strides implied by the sizes):
 *     x, y            [batch][seqlen][nheads][headdim]          in_dtype
 *     dt              [batch][seqlen][nheads]                    float
 *     A, D            [nheads]                                   float
 *     B, C            [batch][seqlen][ngroups][dstate]           in_dtype
 *     init_state, final_state, decode state
 *                     [batch][nheads][headdim][dstate]           float
 *                     (a decode state may be bfloat16: ssd_state_update_fused)
 * For decode, drop the seqlen dimension.  Packed variable-length batches
 * (ssd_scan_fwd_varlen) drop the batch dimension of the token arrays.
 *
 * fp8 inputs (in_dtype SSD_FP8_E4M3, prefill entry points only): x, B and C
 * hold one byte per value in the E4M3 encoding -- sign bit, 4 exponent bits
 * with bias 7, 3 significand bits; exponent field 0 encodes the subnormals
 * m * 2^-9; no infinities; S.1111.111 is NaN; the largest finite value is
 * 448.  Every E4M3 value is exactly a bfloat16 value, so each call widens x,
 * B and C once into bfloat16 copies in its workspace (one elementwise kernel,
 * ssd_fp8_e4m3_to_bf16) and runs the bf16 path on the copies: the result is
 * the bf16 path's on the exactly decoded inputs.  y and the gate's z are
 * bfloat16 in such a call.  The pages name reduced precision as future work
 * (CGLA sections V.A and VI) without fixing a format; E4M3 is the common
 * 8-bit one.  The decode entry points return SSD_ERR_UNSUPPORTED for it.
 *
 * Ownership: every pointer is a DEVICE pointer owned by the caller, except
 * where an entry point says otherwise.  The library allocates no memory;
 * scratch memory is the caller's workspace, sized by
 * ssd_scan_workspace_bytes().
 *
 * Asynchrony: work is enqueued on `stream` and the call returns without
 * synchronising.  Argument errors are detected on the host before anything
 * is enqueued and are returned synchronously.  Device-side faults the kernels
 * detect themselves (a bounded wait that ran out, a misaligned shared-memory
 * carve-out) set a device error word read by ssd_last_device_error().
 *
 * Aliasing: y and final_state must not overlap any input.  The decode state
 * is updated in place.
 */
#ifndef SSD_GB300_H
#define SSD_GB300_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SSD_OK = 0,
    SSD_ERR_INVALID_ARG = 1,   /* null pointer, size <= 0, H % G != 0, misaligned pointer */
    SSD_ERR_UNSUPPORTED = 2,   /* a valid shape the requested kernel does not handle */
    SSD_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
    SSD_ERR_TIMEOUT = 4,       /* a bounded device-side wait ran out (read via ssd_last_device_error) */
    SSD_ERR_WORKSPACE = 5      /* workspace pointer null or smaller than ssd_scan_workspace_bytes() */
} ssd_status;

typedef enum { SSD_F32 = 0, SSD_BF16 = 1, SSD_FP8_E4M3 = 2 } ssd_dtype;

/* Which kernels ssd_scan_fwd_algo uses.  AUTO takes the tensor-core path when
 * the shape allows it and the SIMT path otherwise; both run on the GPU. */
typedef enum {
    SSD_ALGO_AUTO = 0,
    SSD_ALGO_SIMT = 1,      /* exact-fp32 FFMA chunked scan, any shape */
    SSD_ALGO_TCGEN05 = 2    /* tcgen05/TMEM/TMA chunked scan: bf16 inputs, headdim 64,
                               dstate 128 */
} ssd_algo;

/* Bytes of device workspace ssd_scan_fwd / ssd_scan_fwd_algo need for this
 * shape on the CURRENT device (the segment plan depends on its SM count), for
 * either input dtype (fp32 inputs need none; the figure is that of bf16
 * inputs): the segment states and decays of the tensor-core path.  Returns 0
 * when the shape needs none, and (size_t)-1 for invalid sizes. */
size_t ssd_scan_workspace_bytes(int batch, int seqlen, int nheads, int headdim,
                                int dstate, int ngroups, int chunk);

/* The exact workspace of a call with this input dtype and, when
 * with_dt_transform != 0, a dt transform (ssd_scan_fwd_dt, ssd_scan_fwd_fused):
 * on the tensor-core path a transform adds batch x seqlen x nheads floats for
 * the transformed step sizes.  SSD_FP8_E4M3 adds the bfloat16 copies of x, B
 * and C (2 bytes per value, each copy rounded up to 256 bytes) in front of
 * the workspace of the bf16 call.  (size_t)-1 for invalid sizes. */
size_t ssd_scan_fused_workspace_bytes(int batch, int seqlen, int nheads, int headdim,
                                      int dstate, int ngroups, int chunk,
                                      ssd_dtype in_dtype, int with_dt_transform);

/* Number of kernel launches ssd_scan_fwd enqueues for this shape on the
 * current device (for launch accounting and CUDA-graph planning); -1 for
 * invalid sizes.  A dt transform on the tensor-core path adds one (the
 * elementwise pass that transforms every dt once), and so do fp8 inputs (the
 * widening of x, B and C). */
int ssd_scan_kernel_launches(int batch, int seqlen, int nheads, int headdim,
                             int dstate, int ngroups, int chunk,
                             ssd_dtype in_dtype);

/* Prefill: the chunked SSD scan over a whole sequence (section III.A of the
 * CGLA page: Step-1 intra-chunk dual form, chunk states, Step-3 inter-chunk
 * recurrence, plus the off-diagonal output and the D skip).
 *
 *   x, B, C     in_dtype device arrays (layouts above; SSD_FP8_E4M3 as
 *               described there, with its workspace from
 *               ssd_scan_fused_workspace_bytes).
 *   dt, A       float.  D: float [nheads] or NULL (no skip term).
 *   chunk       the chunk length Q: one of 16, 32, 64, 128, 256, validated
 *               and otherwise UNUSED.  The result does not depend on Q (the
 *               chunked form is an exact re-association of the recurrence);
 *               the kernels tile the sequence in their own block sizes (128
 *               tokens on the tensor-core path, 64 on the SIMT path).
 *   dt          any sign is accepted.  dt >= 0 (a time step) is the intended
 *               use; with dt < 0 the recurrence grows instead of decaying,
 *               and the tensor-core path stays exact only while that growth
 *               inside one 128-token tile is below about e^60 (its mask
 *               factors are fp32); the SIMT path has no such limit.
 *   init_state  float [batch][nheads][headdim][dstate] or NULL (zeros).
 *   y           in_dtype output (bfloat16 for fp8 inputs).  final_state:
 *               float output or NULL.
 *   workspace   device scratch of at least ssd_scan_workspace_bytes() bytes
 *               (may be NULL when that is 0), 256-byte aligned; its contents
 *               need no initialisation.
 * Requirements: all sizes > 0, nheads % ngroups == 0, dstate % 4 == 0,
 * dstate <= 256, base pointers 16-byte aligned.  seqlen may be any length
 * (the last block is ragged). */
ssd_status ssd_scan_fwd(const void *x, const float *dt, const float *A,
                        const void *B, const void *C, const float *D,
                        ssd_dtype in_dtype, int batch, int seqlen, int nheads,
                        int headdim, int dstate, int ngroups, int chunk,
                        const float *init_state, void *y, float *final_state,
                        void *workspace, size_t workspace_bytes,
                        cudaStream_t stream);

/* Same as ssd_scan_fwd with an explicit kernel choice.  SSD_ALGO_TCGEN05
 * returns SSD_ERR_UNSUPPORTED for shapes it does not handle. */
ssd_status ssd_scan_fwd_algo(ssd_algo algo, const void *x, const float *dt,
                             const float *A, const void *B, const void *C,
                             const float *D, ssd_dtype in_dtype, int batch,
                             int seqlen, int nheads, int headdim, int dstate,
                             int ngroups, int chunk, const float *init_state,
                             void *y, float *final_state, void *workspace,
                             size_t workspace_bytes, cudaStream_t stream);

/* Optional transform of the raw step size, applied to every dt the kernels
 * read (the pages take the step Delta from the input projection, CGLA
 * section III.A, without spelling out how it is made positive; this is the
 * usual bias + softplus parameterisation).  The fp32 and decode kernels apply
 * it where they read dt; the tensor-core path transforms every dt once, in an
 * elementwise pass into the workspace, before its kernels run:
 *
 *   dt <- min(max(sp(dt_raw + dt_bias[h]), dt_min), dt_max)
 *   sp(u) = log(1 + e^u) when softplus != 0, else sp(u) = u.
 *
 * dt_bias: float [nheads] device array or NULL (no bias).  dt_min <= dt_max
 * (NaN rejected); use -INFINITY / INFINITY for no clamp.  The sign rule of
 * ssd_scan_fwd applies to the transformed dt (softplus, or dt_min >= 0, makes
 * it a non-negative time step).  The caller owns dt_bias; it is read during
 * the call's kernels. */
typedef struct ssd_dt_transform {
    const float *dt_bias;
    int softplus;
    float dt_min, dt_max;
} ssd_dt_transform;

/* ssd_scan_fwd_algo with a dt transform (NULL = identity: exactly
 * ssd_scan_fwd_algo).  Returns SSD_ERR_INVALID_ARG when dt_min > dt_max or
 * either is NaN.  With a transform the workspace is
 * ssd_scan_fused_workspace_bytes(..., in_dtype, 1). */
ssd_status ssd_scan_fwd_dt(ssd_algo algo, const void *x, const float *dt,
                           const float *A, const void *B, const void *C,
                           const float *D, const ssd_dt_transform *dt_transform,
                           ssd_dtype in_dtype, int batch, int seqlen, int nheads,
                           int headdim, int dstate, int ngroups, int chunk,
                           const float *init_state, void *y, float *final_state,
                           void *workspace, size_t workspace_bytes,
                           cudaStream_t stream);

/* Packed variable-length sequences: the scan of ssd_scan_fwd_dt run on each
 * of nseq independent sequences laid end to end on one token axis (each
 * sequence is its own recurrence with its own initial and final state, as
 * the pages define the scan per sequence; the packing is this library's
 * layout, not the pages').  Sequence s is tokens cu[s] .. cu[s+1]-1 of
 * T = cu[nseq] tokens:
 *   x, y   in_dtype [T][nheads][headdim];  dt float [T][nheads];
 *   B, C   in_dtype [T][ngroups][dstate];
 *   init_state, final_state  float [nseq][nheads][headdim][dstate] or NULL.
 *   cu_seqlens_host  int [nseq + 1] HOST array: cu[0] = 0, non-decreasing.
 *                    Empty sequences are allowed (final = initial state, or
 *                    zeros); with T = 0 the token arrays may be NULL.  It
 *                    sizes the grid and the workspace.
 *   cu_seqlens_dev   the same nseq + 1 values in a DEVICE int array, read by
 *                    the kernels; the two copies must agree (not checked).
 *   z      in_dtype [T][nheads][headdim] (bfloat16 for fp8 inputs) or
 *          NULL: the output gate of ssd_scan_fwd_fused.
 * Other arguments and requirements as ssd_scan_fwd_dt.  The workspace is
 * sized by ssd_scan_varlen_workspace_bytes() for the same offsets.
 * Returns SSD_ERR_INVALID_ARG for offsets that do not start at 0 or decrease. */
ssd_status ssd_scan_fwd_varlen(ssd_algo algo, const void *x, const float *dt,
                               const float *A, const void *B, const void *C,
                               const float *D, const ssd_dt_transform *dt_transform,
                               const void *z, ssd_dtype in_dtype, int nseq,
                               const int *cu_seqlens_host,
                               const int *cu_seqlens_dev, int nheads, int headdim,
                               int dstate, int ngroups, int chunk,
                               const float *init_state, void *y,
                               float *final_state, void *workspace,
                               size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes and kernel launches of ssd_scan_fwd_varlen for these
 * offsets on the current device ((size_t)-1 / -1 for invalid arguments).  The
 * workspace figure covers a call with a dt transform (total tokens x nheads
 * floats for the transformed step sizes on the tensor-core path); a call
 * without one uses that much less of it. */
size_t ssd_scan_varlen_workspace_bytes(int nseq, const int *cu_seqlens_host,
                                       int nheads, int headdim, int dstate,
                                       int ngroups, int chunk, ssd_dtype in_dtype);
int ssd_scan_varlen_kernel_launches(int nseq, const int *cu_seqlens_host,
                                    int nheads, int headdim, int dstate,
                                    int ngroups, int chunk, ssd_dtype in_dtype);

/* Output gate of the layer step after the scan, fused into the kernels that
 * write y (the fusion of neighbouring layer steps into the scan that the
 * compiler-first SSD page and the Mambalaya cascade describe; the gate's
 * form is the usual Mamba-2 one, not spelled out on the pages):
 *
 *   y <- y * silu(z),   silu(z) = z / (1 + e^-z),
 *
 * applied after the D skip, before y is rounded to its dtype.  z: a device
 * array of y's dtype and layout, 16-byte aligned, or NULL (no gate).  The
 * normalisation that may follow the gate in a layer is not fused (it reduces
 * over all heads of a token).  Everything else as ssd_scan_fwd_dt. */
ssd_status ssd_scan_fwd_fused(ssd_algo algo, const void *x, const float *dt,
                              const float *A, const void *B, const void *C,
                              const float *D, const ssd_dt_transform *dt_transform,
                              const void *z, ssd_dtype in_dtype, int batch,
                              int seqlen, int nheads, int headdim, int dstate,
                              int ngroups, int chunk, const float *init_state,
                              void *y, float *final_state, void *workspace,
                              size_t workspace_bytes, cudaStream_t stream);

/* Profiling hook (process-wide, not for concurrent callers): while both
 * events are non-NULL, every following ssd_scan_fwd / ssd_scan_fwd_algo
 * records `before` immediately before and `after` immediately after the
 * kernel that writes y, on the call's stream, so cudaEventElapsedTime gives
 * that kernel's device time.  Works inside stream capture (the records become
 * graph nodes).  Pass NULL, NULL to stop.  Always returns SSD_OK. */
ssd_status ssd_scan_profile_events(cudaEvent_t before, cudaEvent_t after);

/* Size of the scratch array built into the library for ssd_scan_fwd_static. */
#define SSD_STATIC_SCRATCH_BYTES (64u << 20)

/* ssd_scan_fwd for callers that cannot allocate device memory (the pages
 * have no counterpart: this exists for callers whose memory is fixed at
 * start-up, such as an engine plugin handed only its inputs and outputs, or a
 * runtime that forbids device allocation after initialisation).  Same
 * arguments and results as ssd_scan_fwd without the workspace: the scratch is
 * a fixed array of SSD_STATIC_SCRATCH_BYTES inside the library, held on every
 * GPU that loads the library until the process exits.  Allocates nothing.
 *   - Returns SSD_ERR_WORKSPACE when the shape needs more scratch than
 *     SSD_STATIC_SCRATCH_BYTES (ssd_scan_workspace_bytes() tells how much).
 *     The 2.7B-shaped 65536-token layer (80 heads, 23 MB of bf16 segment
 *     states on a 152-SM GB300) fits.
 *   - The first call on each device looks up the scratch address for that
 *     device; make that first call before any stream capture.
 *   - All calls share the one scratch array: calls whose work overlaps on the
 *     GPU (unordered streams) race.  No scratch contents need clearing. */
ssd_status ssd_scan_fwd_static(const void *x, const float *dt, const float *A,
                               const void *B, const void *C, const float *D,
                               ssd_dtype in_dtype, int batch, int seqlen,
                               int nheads, int headdim, int dstate,
                               int ngroups, int chunk,
                               const float *init_state, void *y,
                               float *final_state, cudaStream_t stream);

/* Decode: one token of the recurrence for every (batch, head), the O(1)
 * cached step of the compiler-first SSD page.
 *   state  float [batch][nheads][headdim][dstate], read and updated IN PLACE.
 *   x      in_dtype [batch][nheads][headdim];  dt float [batch][nheads];
 *   B, C   in_dtype [batch][ngroups][dstate];  A, D float [nheads] (D may be NULL).
 *   y      in_dtype [batch][nheads][headdim], computed from the updated state.
 * A stack of layers can be updated in one call by treating (layer, head) as
 * the head index and giving every layer its own group (ngroups = layers).
 * Requirements: sizes > 0, nheads % ngroups == 0, dstate a power of two in
 * [4, 256], 16-byte aligned state / B / C. */
ssd_status ssd_state_update(float *state, const void *x, const float *dt,
                            const float *A, const void *B, const void *C,
                            const float *D, ssd_dtype in_dtype, int batch,
                            int nheads, int headdim, int dstate, int ngroups,
                            void *y, cudaStream_t stream);

/* ssd_state_update with a dt transform (see ssd_dt_transform; NULL =
 * identity). */
ssd_status ssd_state_update_dt(float *state, const void *x, const float *dt,
                               const float *A, const void *B, const void *C,
                               const float *D, const ssd_dt_transform *dt_transform,
                               ssd_dtype in_dtype, int batch, int nheads,
                               int headdim, int dstate, int ngroups, void *y,
                               cudaStream_t stream);

/* ssd_state_update_dt with the output gate of ssd_scan_fwd_fused and a
 * choice of state storage.
 *   state        [batch][nheads][headdim][dstate] of state_dtype, in place.
 *                SSD_BF16 stores the state as bfloat16 (half the bytes of
 *                the HBM-bound update): each step reads it, updates it in
 *                fp32 and writes it rounded to nearest even; y is computed
 *                from the fp32 update before that rounding.  The pages name
 *                reduced precision as future work (CGLA sections IV and VI)
 *                without fixing a format; this is the plainest one.  bf16
 *                states need in_dtype SSD_BF16 (else SSD_ERR_UNSUPPORTED).
 *   z            in_dtype [batch][nheads][headdim] (y's layout), 16-byte
 *                aligned, or NULL: the output gate y <- y * silu(z). */
ssd_status ssd_state_update_fused(void *state, ssd_dtype state_dtype, const void *x,
                                  const float *dt, const float *A, const void *B,
                                  const void *C, const float *D,
                                  const ssd_dt_transform *dt_transform, const void *z,
                                  ssd_dtype in_dtype, int batch, int nheads, int headdim,
                                  int dstate, int ngroups, void *y, cudaStream_t stream);

/* Decode of `ntokens` consecutive tokens per (batch, head) in one call: the
 * on-device multi-step loop of the O(1) cached decode (compiler-first SSD
 * page, abstract).  Equivalent to ntokens calls of ssd_state_update_fused in
 * token order, except that a bf16 state is rounded once, when it is written
 * back after the last token, not after every token (the state stays fp32 on
 * chip in between).  Each state is read once and written once per call, so
 * its HBM traffic per token falls by ntokens.
 *   state        [batch][nheads][headdim][dstate] of state_dtype, in place.
 *   x, y, z      in_dtype [batch][ntokens][nheads][headdim] (z may be NULL).
 *   dt           float [batch][ntokens][nheads].
 *   B, C         in_dtype [batch][ntokens][ngroups][dstate].
 *   A, D, dt_transform as ssd_state_update_fused.
 * The token arrays have the layouts of ssd_scan_fwd with seqlen = ntokens.
 * Requirements: those of ssd_state_update_fused, ntokens > 0, and headdim at
 * most 512 for dstate 4 to 16, 8192 / dstate for dstate 32 to 128 (256, 128,
 * 64) and 64 for dstate 256, else SSD_ERR_UNSUPPORTED. */
ssd_status ssd_state_update_multi(void *state, ssd_dtype state_dtype, const void *x,
                                  const float *dt, const float *A, const void *B,
                                  const void *C, const float *D,
                                  const ssd_dt_transform *dt_transform, const void *z,
                                  ssd_dtype in_dtype, int batch, int ntokens, int nheads,
                                  int headdim, int dstate, int ngroups, void *y,
                                  cudaStream_t stream);

/* Widens n E4M3 values (the fp8 encoding described at the top) to bfloat16,
 * exactly: the conversion every fp8 prefill call runs on x, B and C, exported
 * for callers that keep fp8 copies of other tensors.  NaN codes give a
 * bfloat16 NaN.  src: n bytes, dst: n bfloat16 values, both device pointers,
 * 16-byte aligned, not overlapping.  n == 0 enqueues nothing.  Returns
 * SSD_ERR_INVALID_ARG for a null or misaligned pointer (n > 0). */
ssd_status ssd_fp8_e4m3_to_bf16(const void *src, void *dst, size_t n, cudaStream_t stream);

/* One long sequence split over GPUs by tokens (GPU r holds a contiguous
 * range of its tokens): the exchange step.  Step-3 of the recurrence at the
 * granularity of a range (CGLA section III.A: the state is carried
 * sequentially, with the input-dependent diagonal decay):
 *     H_in[0] = init,   H_in[r+1] = exp(a_r) H_in[r] + F_r,
 * with a_r the range's log-decay and F_r the state the range reaches from a
 * zero state (its ssd_scan_fwd with init_state = NULL).  Each GPU scans its
 * range from zero for F_r, the pairs (a_r, F_r) are gathered from every GPU,
 * each chains them to its own H_in and scans its range again from H_in for
 * y; the last range's final state is the sequence's.  The pages do not build
 * this split (their runs are on one device); the all-gather is the caller's
 * (torch.distributed in the Python package).
 *
 * ssd_range_log_decay: log_decay[b][h] = A[h] * sum over the range's tokens
 * of dt[b][t][h] (after the dt transform, when one is given, as the scan
 * applies it), summed in double precision.  dt [batch][seqlen][nheads],
 * A [nheads], log_decay [batch][nheads]: float device arrays.
 * SSD_ERR_INVALID_ARG for null pointers, sizes <= 0 or an invalid transform. */
ssd_status ssd_range_log_decay(const float *dt, const float *A,
                               const ssd_dt_transform *dt_transform, int batch, int seqlen,
                               int nheads, float *log_decay, cudaStream_t stream);

/* ssd_chain_states: entering[r] = H_in[r] for r = 0 .. nranges-1 from the
 * ranges' contributions contrib[r] = F_r and log-decays log_decay[r] = a_r,
 * starting from init (zeros when NULL).  contrib, entering
 * [nranges][batch][nheads][headdim][dstate]; log_decay
 * [nranges][batch][nheads]; init [batch][nheads][headdim][dstate]: float
 * device arrays; entering must not overlap the inputs.  SSD_ERR_INVALID_ARG
 * for null required pointers or sizes <= 0. */
ssd_status ssd_chain_states(const float *contrib, const float *log_decay, const float *init,
                            int nranges, int batch, int nheads, int headdim, int dstate,
                            float *entering, cudaStream_t stream);

/* Human-readable name of a status code (static storage). */
const char *ssd_status_string(ssd_status s);

/* Reads and clears the device error word on the current device
 * (synchronises the device).  SSD_OK when no kernel reported a fault. */
ssd_status ssd_last_device_error(void);

/* Test hook for the bounded device-side waits (the pages have no
 * counterpart).  Every later launch of the tensor-core scan reads the
 * setting; it is process-wide and not synchronised with calls in flight on
 * other host threads.
 *   fault          SSD_FAULT_NONE: normal operation.  SSD_FAULT_WITHHOLD_SIGNAL:
 *                  in the CTAs of each sequence's first segment, the barrier
 *                  that signals "decay factors ready" waits for one arrival
 *                  more than the warp computing them gives, so the first wait
 *                  for it runs out; the CTA then lets its issued copies and
 *                  tensor-core products complete, frees its tensor memory and
 *                  exits, and the device error word reads SSD_ERR_TIMEOUT.
 *                  The outputs of that call are undefined.
 *   wait_limit_ns  limit of every bounded wait in those kernels; 0 restores
 *                  the default (2 s).
 * Returns SSD_ERR_INVALID_ARG for an unknown fault. */
typedef enum { SSD_FAULT_NONE = 0, SSD_FAULT_WITHHOLD_SIGNAL = 1 } ssd_fault;
ssd_status ssd_debug_inject_fault(ssd_fault fault, unsigned long long wait_limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* SSD_GB300_H */
