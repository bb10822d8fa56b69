// Decode: one token of the SSD recurrence for every (batch, head), the O(1)
// cached step of "Compiler-First State Space Duality and Portable O(1)
// Autoregressive Caching" (abstract); the per-head transition is the
// input-dependent diagonal of the CGLA kernel page, section III.A.
//
//   h[p][n] <- exp(dt*A_h) * h[p][n] + dt * B[n] * x[p]
//   y[p]     = sum_n C[n] * h[p][n] + D_h * x[p]
//
// The update is HBM-bound (0.75 flop per byte): every state byte is read once
// and written once.  One CTA owns one (batch, head) state of P x N floats, or
// a run of its rows when there are fewer states than two per SM (rows are
// independent: y[p] reads row p alone); a row p is spread over TPR threads
// holding VPT float4 each, so a warp reads and writes whole 128-byte lines.
// All of a thread's row loads are issued before any arithmetic to keep
// enough bytes in flight, and the state uses streaming (evict-first) loads
// and stores because it is touched once per call.  y reduces C . h across
// the TPR threads of a row with shuffles.
//
// Both single-token kernels are launched with programmatic stream
// serialization: a call's grid may be scheduled while the previous kernel in
// the stream still runs, waits for it (griddepcontrol.wait) before touching
// memory, and releases the next launch at once.  Per-layer calls of a small
// batch are launch-bound, and this hides most of a launch per call (timed on
// 64 per-layer calls a token: 355 -> 274 us at batch 1 with the row split,
// 1046 -> 1005 us at batch 16).  The streaming kernel, and the multi-token
// kernel below, take it only for calls of at most 64 states per SM.
#include <algorithm>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace {

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel in the stream runs; it calls griddepcontrol.wait
// before touching memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

constexpr int kThreads = 256;
constexpr int kBatchRows = 8;   // rows each thread has in flight at once

template <typename T, typename S, int VPT, bool kFuse>
__global__ void __launch_bounds__(kThreads)
ssd_decode_kernel(S *__restrict__ state, const T *__restrict__ x,
                  const float *__restrict__ dt, const float *__restrict__ A,
                  const T *__restrict__ Bm, const T *__restrict__ Cm,
                  const float *__restrict__ D, T *__restrict__ y, int H, int P,
                  int N, int G, int rpc, const SsdFuse fuse) {
    const int bh = blockIdx.x;             // b * H + h
    // rows p0 .. p1-1 of the state: all of them, or a part when the states
    // alone would leave SMs idle
    const int p0 = blockIdx.y * rpc, p1 = min(P, p0 + rpc);
    ssdptx::griddep_wait();
    ssdptx::griddep_launch_dependents();
    const int b = bh / H, h = bh - b * H;
    const int g = h / (H / G);
    const int tpr = N / (4 * VPT);         // threads per row, power of two <= 32
    const int rpp = kThreads / tpr;        // rows per pass
    const int lane_n = threadIdx.x % tpr;
    const int r0 = threadIdx.x / tpr;

    const float dtv = ssd_dt<kFuse>(fuse, dt[bh], ssd_dt_bias<kFuse>(fuse, h));
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
    S *st = state + (size_t)bh * P * N;
    const T *xr = x + (size_t)bh * P;
    T *yr = y + (size_t)bh * P;

    // the loop bound is the same for every thread so the row shuffles below
    // always see full warps
    for (int pb0 = p0; pb0 < p1; pb0 += kBatchRows * rpp) {
        const int pb = pb0 + r0;
        float4 s[kBatchRows][VPT];
        float xv[kBatchRows];
#pragma unroll
        for (int i = 0; i < kBatchRows; ++i) {
            const int p = pb + i * rpp;
            if (p < p1) {
                xv[i] = ssd_ld(xr + p);
#pragma unroll
                for (int v = 0; v < VPT; ++v)
                    s[i][v] = ssd_ld4_cs(st + (size_t)p * N + 4 * (lane_n + v * tpr));
            }
        }
#pragma unroll
        for (int i = 0; i < kBatchRows; ++i) {
            const int p = pb + i * rpp;
            float acc = 0.0f;
            if (p < p1) {
                const float dx = dtv * xv[i];
#pragma unroll
                for (int v = 0; v < VPT; ++v) {
                    float4 q = s[i][v];
                    q.x = fmaf(decay, q.x, dx * Bv[v].x);
                    q.y = fmaf(decay, q.y, dx * Bv[v].y);
                    q.z = fmaf(decay, q.z, dx * Bv[v].z);
                    q.w = fmaf(decay, q.w, dx * Bv[v].w);
                    ssd_st4_cs(st + (size_t)p * N + 4 * (lane_n + v * tpr), q);
                    acc = fmaf(Cv[v].x, q.x, acc);
                    acc = fmaf(Cv[v].y, q.y, acc);
                    acc = fmaf(Cv[v].z, q.z, acc);
                    acc = fmaf(Cv[v].w, q.w, acc);
                }
            }
            // reduce over the tpr threads of this row (aligned power-of-two group)
            for (int off = tpr >> 1; off > 0; off >>= 1)
                acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (p < p1 && lane_n == 0)
                ssd_st(yr + p, ssd_gate<kFuse, T>(fuse, acc + Dh * xv[i], (size_t)bh * P + p));
        }
    }
}

// Streaming variant for large stacks: a persistent CTA per SM walks its
// (batch, head) states through a ring of shared-memory stages.  Each stage
// receives, by bulk copies, one fp32 state (32 KB at P 64, N 128) or two
// consecutive bf16 states, their x rows and their groups' B and C rows, so no
// global-memory latency sits between the update of one state and the next;
// the copy engine keeps several states in flight without occupying registers.
// The states are updated in place in shared memory and written back by one
// bulk store per stage.
constexpr int kStreamThreads = 512;
constexpr int kStreamRows = 4;          // rows each thread updates per pass
constexpr uint32_t kStreamRing = 229376;   // ring capacity in bytes
constexpr uint64_t kStreamWaitNs = 2000000000ull;

struct StreamLayout {
    uint32_t state_bytes, x_bytes, bc_bytes, stage_bytes;
};

// A stage holds `per` consecutive states, then their x rows, then each
// one's B and C rows.
__host__ __device__ inline StreamLayout stream_layout(int P, int N, int es, int ss, int per) {
    StreamLayout l;
    l.state_bytes = (uint32_t)P * N * (uint32_t)ss;
    l.x_bytes = (uint32_t)P * es;
    l.bc_bytes = (uint32_t)N * es;
    const uint32_t raw = (uint32_t)per * (l.state_bytes + l.x_bytes + 2 * l.bc_bytes);
    l.stage_bytes = (raw + 127u) & ~127u;
    return l;
}
// states per ring stage: two with bf16 states (a 32 KB stage, as one fp32 state)
template <typename S>
__host__ __device__ constexpr int stream_per_stage() { return sizeof(S) < 4 ? 2 : 1; }

template <typename T, typename S, int N, bool kFuse>
__global__ void __launch_bounds__(kStreamThreads + 32, 1)
ssd_decode_stream_kernel(S *__restrict__ state, const T *__restrict__ x,
                         const float *__restrict__ dt, const float *__restrict__ A,
                         const T *__restrict__ Bm, const T *__restrict__ Cm,
                         const float *__restrict__ D, T *__restrict__ y, int batch, int H, int P,
                         int G, int stages, unsigned int *err, const SsdFuse fuse) {
    constexpr int VPT = N > 128 ? 2 : 1;
    using namespace ssdptx;
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int U = stream_per_stage<S>();
    const StreamLayout L = stream_layout(P, N, (int)sizeof(T), (int)sizeof(S), U);
    const long units = (long)batch * H;
    const long items = (units + U - 1) / U;   // stage loads of U consecutive states
    const int tid = threadIdx.x;
    // barriers: full[stages] (bulk loads landed), done[stages] (update finished)
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)stages * L.stage_bytes);
    uint64_t *done = full + stages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(done + stages);
    const uint32_t sbase = smem_u32(smem);
    constexpr int kComputeWarps = kStreamThreads / 32;
    // bf16 states halve the bytes per state, so the per-state work becomes the
    // limit: a ring stage then holds two consecutive states (one 32 KB bulk
    // copy each way, as one fp32 state), and four groups of compute warps take
    // alternate stages (timed at batch 16: 0.405 ms a token against 0.487 with
    // one state per stage, 0.55 with one per stage and two groups fewer)
    constexpr int kGroups = sizeof(S) < 4 ? 4 : 1;
    if (tid == 0) {
        for (int i = 0; i < stages; ++i) {
            mbar_init(smem_u32(full + i), 1);
            mbar_init(smem_u32(done + i), kComputeWarps / kGroups);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    griddep_wait();
    griddep_launch_dependents();
    const long nk = blockIdx.x < items ? (items - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    // first state and state count of this CTA's k-th stage load
    auto unit_of = [&](long k) { return ((long)blockIdx.x + k * (long)gridDim.x) * U; };
    auto count_of = [&](long k) { return (int)min((long)U, units - unit_of(k)); };

    if (tid >= kStreamThreads) {
        // ---- copy warp: loads run stages-1 units ahead; each updated state is
        //      written back as soon as its compute warps are done with it
        if (tid == kStreamThreads) {
            const uint64_t evict_first = l2_evict_first_policy();   // states: touched once
            auto issue_load = [&](long k) {
                const int st = (int)(k % stages);
                const long u0 = unit_of(k);
                const int cnt = count_of(k);
                const uint32_t dst = sbase + st * L.stage_bytes;
                const uint32_t bar = smem_u32(full + st);
                mbar_arrive_expect_tx(bar, cnt * (L.state_bytes + L.x_bytes + 2 * L.bc_bytes));
                bulk_load_evict_first(dst, state + (size_t)u0 * P * N, cnt * L.state_bytes, bar,
                                      evict_first);
                bulk_load(dst + U * L.state_bytes, x + (size_t)u0 * P, cnt * L.x_bytes, bar);
                for (int i = 0; i < cnt; ++i) {
                    const long u = u0 + i;
                    const int b = (int)(u / H), h = (int)(u - (long)b * H);
                    const size_t grow = ((size_t)b * G + h / (H / G)) * N;
                    const uint32_t bc = dst + U * (L.state_bytes + L.x_bytes) + i * 2 * L.bc_bytes;
                    bulk_load(bc, Bm + grow, L.bc_bytes, bar);
                    bulk_load(bc + L.bc_bytes, Cm + grow, L.bc_bytes, bar);
                }
            };
            for (long k = 0; k < nk && k < stages - 1; ++k) issue_load(k);
            for (long k = 0; k < nk; ++k) {
                const int st = (int)(k % stages);
                if (!mbar_wait<true>(smem_u32(done + st), (uint32_t)((k / stages) & 1), kStreamWaitNs)) {
                    *abort_flag = 1;
                    ssd_report(err, SSD_DEVERR_TIMEOUT);
                    break;
                }
                bulk_store_evict_first(state + (size_t)unit_of(k) * P * N,
                                       sbase + st * L.stage_bytes, count_of(k) * L.state_bytes,
                                       evict_first);
                bulk_commit();
                if (k + stages - 1 < nk) {
                    // its stage last held unit k-1, whose store must be done reading
                    bulk_wait_read<1>();
                    issue_load(k + stages - 1);
                }
            }
            bulk_wait_all();
        }
    } else {
        // ---- compute warps
        // tpr (threads per row) and N are powers of two: rows and offsets by
        // shifts; a thread's rows advance by kGroupThreads / tpr per step
        constexpr int kGroupThreads = kStreamThreads / kGroups;
        const int grp = tid / kGroupThreads, gtid = tid - grp * kGroupThreads;
        constexpr int tpr = N / (4 * VPT);
        constexpr int tsh = tpr >= 32 ? 5 : tpr >= 16 ? 4 : tpr >= 8 ? 3 : tpr >= 4 ? 2 : tpr >= 2 ? 1 : 0;
        constexpr int nsh = N >= 256 ? 8 : N >= 128 ? 7 : N >= 64 ? 6 : N >= 32 ? 5 : N >= 16 ? 4 : N >= 8 ? 3 : 2;
        const int lane_n = gtid & (tpr - 1);
        const int total = P * tpr;
        const int row0 = gtid >> tsh, row_step = kGroupThreads >> tsh;
        // the next unit's dt, A and D are loaded one unit ahead, so no global
        // load latency sits between two units' updates (dt raw; transformed at use)
        // one state of a stage: its update and readout (S, x, B, C in the stage)
        auto update = [&](S *sm, const T *xs, const T *Bs, const T *Cs, float dtv, float decay,
                          float Dh, long u) {
            float4 Bv[VPT], Cv[VPT];
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const int n0 = 4 * (lane_n + v * tpr);
                Bv[v] = ssd_ld4(Bs + n0);
                Cv[v] = ssd_ld4(Cs + n0);
            }
            // kStreamRows independent rows per thread per pass: all shared-memory
            // reads first, then the updates, then the interleaved row reductions
            for (int e0 = 0; e0 < total; e0 += kGroupThreads * kStreamRows) {
                const int pbase = (e0 >> tsh) + row0;   // row of this thread's i = 0
                float4 q[kStreamRows][VPT];
                float xv[kStreamRows], acc[kStreamRows];
#pragma unroll
                for (int i = 0; i < kStreamRows; ++i) {
                    const int p = pbase + i * row_step;
                    acc[i] = 0.0f;
                    xv[i] = 0.0f;
                    if (p < P) {
                        xv[i] = ssd_ld(xs + p);
#pragma unroll
                        for (int v = 0; v < VPT; ++v)
                            q[i][v] = ssd_ld4(sm + (p << nsh) + 4 * (lane_n + v * tpr));
                    }
                }
#pragma unroll
                for (int i = 0; i < kStreamRows; ++i) {
                    const int p = pbase + i * row_step;
                    if (p < P) {
                        const float dx = dtv * xv[i];
#pragma unroll
                        for (int v = 0; v < VPT; ++v) {
                            float4 w = q[i][v];
                            w.x = fmaf(decay, w.x, dx * Bv[v].x);
                            w.y = fmaf(decay, w.y, dx * Bv[v].y);
                            w.z = fmaf(decay, w.z, dx * Bv[v].z);
                            w.w = fmaf(decay, w.w, dx * Bv[v].w);
                            ssd_st4(sm + (p << nsh) + 4 * (lane_n + v * tpr), w);
                            acc[i] = fmaf(Cv[v].x, w.x, acc[i]);
                            acc[i] = fmaf(Cv[v].y, w.y, acc[i]);
                            acc[i] = fmaf(Cv[v].z, w.z, acc[i]);
                            acc[i] = fmaf(Cv[v].w, w.w, acc[i]);
                        }
                    }
                }
                // reduce over the tpr threads of each row.  fp32 states (HBM-bound):
                // a butterfly per row.  bf16 states (half the bytes, so the
                // per-state work is the limit): at exchange k (offset tpr >> (k+1))
                // a thread keeps one half of its remaining rows and adds its
                // partner's partials of them; once one row is left, plain
                // butterflies finish the sum (all resolved at compile time).
                // Timed on the 64-layer stack: the exchange form is 14% faster
                // with bf16 states and 1-4% slower with fp32 states.
                int base = 0;
                if constexpr (sizeof(S) >= 4) {
#pragma unroll
                    for (int off = tpr >> 1; off > 0; off >>= 1) {
#pragma unroll
                        for (int i = 0; i < kStreamRows; ++i)
                            acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], off);
                    }
                    if (lane_n == 0) {
#pragma unroll
                        for (int i = 0; i < kStreamRows; ++i) {
                            const int p = pbase + i * row_step;
                            if (p < P)
                                ssd_st(y + (size_t)u * P + p,
                                       ssd_gate<kFuse, T>(fuse, acc[i] + Dh * xv[i], (size_t)u * P + p));
                        }
                    }
                } else {
#pragma unroll
                for (int k = 0; k < 5; ++k) {
                    constexpr int kHalf0 = kStreamRows / 2;
                    const int o = tpr >> (k + 1);
                    if (o > 0 && k < 2) {
                        const int half = kHalf0 >> k;
                        const bool up = (lane_n & o) != 0;
#pragma unroll
                        for (int j = 0; j < kHalf0; ++j) {
                            if (j < half) {
                                const float send = up ? acc[j] : acc[j + half];
                                const float keep = up ? acc[j + half] : acc[j];
                                acc[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                                xv[j] = up ? xv[j + half] : xv[j];
                            }
                        }
                        if (up) base += half;
                    } else if (o > 0) {
                        acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], o);
                    }
                }
                constexpr int left = tpr >= 4 ? 1 : (tpr == 2 ? 2 : kStreamRows);
                constexpr int low = tpr > 4 ? tpr / 4 - 1 : 0;
                if ((lane_n & low) == 0) {
#pragma unroll
                    for (int j = 0; j < left; ++j) {
                        const int p = pbase + (base + j) * row_step;
                        if (p < P)
                            ssd_st(y + (size_t)u * P + p,
                                   ssd_gate<kFuse, T>(fuse, acc[j] + Dh * xv[j], (size_t)u * P + p));
                    }
                }
                }
            }
        };
        if constexpr (U == 1) {
            // the next state's dt, A and D are loaded one state ahead, so no
            // global load latency sits between two states' updates
            float dt_next = 0.f, A_next = 0.f, D_next = 0.f;
            if (grp < nk) {
                const int h0 = (int)(unit_of(grp) % H);
                dt_next = dt[unit_of(grp)];
                A_next = A[h0];
                D_next = D ? D[h0] : 0.0f;
            }
            for (long k = grp; k < nk; k += kGroups) {
                const int st = (int)(k % stages);
                const long u = unit_of(k);
                const int h = (int)(u % H);
                const float dtv = ssd_dt<kFuse>(fuse, dt_next, ssd_dt_bias<kFuse>(fuse, h));
                const float Ah = A_next, Dh = D_next;
                if (k + kGroups < nk) {
                    const long un = unit_of(k + kGroups);
                    const int hn = (int)(un % H);
                    dt_next = dt[un];
                    A_next = A[hn];
                    D_next = D ? D[hn] : 0.0f;
                }
                const float decay = expf(dtv * Ah);
                bool ok = !*abort_flag &&
                          mbar_wait<true>(smem_u32(full + st), (uint32_t)((k / stages) & 1), kStreamWaitNs);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) {
                    *abort_flag = 1;
                    ssd_report(err, SSD_DEVERR_TIMEOUT);
                    break;
                }
                uint8_t *stage = smem + (size_t)st * L.stage_bytes;
                S *sm = reinterpret_cast<S *>(stage);
                const T *xs = reinterpret_cast<const T *>(stage + L.state_bytes);
                const T *Bs = reinterpret_cast<const T *>(stage + L.state_bytes + L.x_bytes);
                const T *Cs = Bs + N;
                update(sm, xs, Bs, Cs, dtv, decay, Dh, u);
                fence_proxy_async_smem();
                __syncwarp();
                if ((tid & 31) == 0) mbar_arrive(smem_u32(done + st));
            }
        } else {
        float dt_next[U], A_next[U], D_next[U];
        auto load_next = [&](long k) {
#pragma unroll
            for (int i = 0; i < U; ++i) {
                dt_next[i] = A_next[i] = D_next[i] = 0.f;
                if (k < nk && i < count_of(k)) {
                    const long un = unit_of(k) + i;
                    const int hn = (int)(un % H);
                    dt_next[i] = dt[un];
                    A_next[i] = A[hn];
                    D_next[i] = D ? D[hn] : 0.0f;
                }
            }
        };
        load_next(grp);
        for (long k = grp; k < nk; k += kGroups) {
            const int st = (int)(k % stages);
            const int cnt = count_of(k);
            float dtc[U], Ac[U], Dc[U];
#pragma unroll
            for (int i = 0; i < U; ++i) {
                dtc[i] = dt_next[i];
                Ac[i] = A_next[i];
                Dc[i] = D_next[i];
            }
            load_next(k + kGroups);
            bool ok = !*abort_flag &&
                      mbar_wait<true>(smem_u32(full + st), (uint32_t)((k / stages) & 1), kStreamWaitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                *abort_flag = 1;
                ssd_report(err, SSD_DEVERR_TIMEOUT);
                break;
            }
            uint8_t *stage = smem + (size_t)st * L.stage_bytes;
#pragma unroll
            for (int i = 0; i < U; ++i) {
            if (i >= cnt) break;
            const long u = unit_of(k) + i;
            const int h = (int)(u % H);
            const float dtv = ssd_dt<kFuse>(fuse, dtc[i], ssd_dt_bias<kFuse>(fuse, h));
            const float Ah = Ac[i], Dh = Dc[i];
            const float decay = expf(dtv * Ah);
            S *sm = reinterpret_cast<S *>(stage + i * L.state_bytes);
            const T *xs = reinterpret_cast<const T *>(stage + U * L.state_bytes + i * L.x_bytes);
            const T *Bs = reinterpret_cast<const T *>(stage + U * (L.state_bytes + L.x_bytes) +
                                                      i * 2 * L.bc_bytes);
            const T *Cs = Bs + N;
            update(sm, xs, Bs, Cs, dtv, decay, Dh, u);
            }   // states of the stage
            fence_proxy_async_smem();
            __syncwarp();
            if ((tid & 31) == 0) mbar_arrive(smem_u32(done + st));
        }
        }
    }
    __syncthreads();
}

template <typename T, typename S, bool kFuse>
cudaError_t launch_t(S *state, const void *x, const float *dt, const float *A,
                     const void *B, const void *C, const float *D, void *y, int batch,
                     int H, int P, int N, int G, int num_sms, unsigned int *err,
                     const SsdFuse &fuse, cudaStream_t stream) {
    const size_t units = (size_t)batch * H;
    const StreamLayout lay = stream_layout(P, N, (int)sizeof(T), (int)sizeof(S),
                                           stream_per_stage<S>());
    const int stages = (int)std::min<size_t>(8, kStreamRing / lay.stage_bytes);
    // the streaming ring pays off once every SM has several states to walk;
    // its bulk copies need 16-byte multiples for the state, x, B and C rows
    if (num_sms > 0 && stages >= 3 && units >= (size_t)num_sms * 4 && lay.x_bytes % 16 == 0 &&
        lay.bc_bytes % 16 == 0 && lay.state_bytes % 16 == 0) {
        const size_t smem = (size_t)stages * lay.stage_bytes + 16 * stages + 16;
        // programmatic launch hides a launch only where that is worth it: a
        // short call (its griddepcontrol instructions are no-ops otherwise);
        // on stacks of hundreds of states per SM it cost ~1 %
        const bool pdl = units <= (size_t)num_sms * 64;
        cudaError_t e;
#define SSD_STREAM_N(NN)                                                                   \
    case NN:                                                                               \
        e = cudaFuncSetAttribute(ssd_decode_stream_kernel<T, S, NN, kFuse>,               \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);   \
        if (e != cudaSuccess) return e;                                                    \
        if (pdl) {                                                                         \
            e = launch_pdl(ssd_decode_stream_kernel<T, S, NN, kFuse>, dim3(num_sms),         \
                           dim3(kStreamThreads + 32), smem, stream, state, (const T *)x, dt, \
                           A, (const T *)B, (const T *)C, D, (T *)y, batch, H, P, G, stages, \
                           err, fuse);                                                     \
            if (e != cudaSuccess) return e;                                                \
        } else {                                                                           \
            ssd_decode_stream_kernel<T, S, NN, kFuse><<<num_sms, kStreamThreads + 32, smem,  \
                                                       stream>>>(                          \
                state, (const T *)x, dt, A, (const T *)B, (const T *)C, D, (T *)y, batch, H, \
                P, G, stages, err, fuse);                                                  \
        }                                                                                  \
        break
        switch (N) {
            SSD_STREAM_N(4);
            SSD_STREAM_N(8);
            SSD_STREAM_N(16);
            SSD_STREAM_N(32);
            SSD_STREAM_N(64);
            SSD_STREAM_N(128);
            SSD_STREAM_N(256);
            default:
                return cudaErrorInvalidValue;   // dstate is checked by the caller
        }
#undef SSD_STREAM_N
        return cudaGetLastError();
    }
    // too few states for two CTAs per SM: split each state's rows over CTAs
    // (rows are independent: y[p] reads row p alone), at least one row per thread
    const int rpp = kThreads / (N <= 128 ? N / 4 : N / 8);
    int nsplit = 1;
    if (num_sms > 0 && units < (size_t)num_sms * 2)
        nsplit = (int)std::min<size_t>(((size_t)num_sms * 2 + units - 1) / units,
                                       (size_t)((P + rpp - 1) / rpp));
    const int rpc = (P + nsplit - 1) / nsplit;
    const dim3 grid((unsigned)units, (unsigned)((P + rpc - 1) / rpc));
    if (N <= 128)
        return launch_pdl(ssd_decode_kernel<T, S, 1, kFuse>, grid, dim3(kThreads), 0, stream,
                          state, (const T *)x, dt, A, (const T *)B, (const T *)C, D, (T *)y, H, P,
                          N, G, rpc, fuse);
    return launch_pdl(ssd_decode_kernel<T, S, 2, kFuse>, grid, dim3(kThreads), 0, stream, state,
                      (const T *)x, dt, A, (const T *)B, (const T *)C, D, (T *)y, H, P, N, G, rpc,
                      fuse);
}

// ------------------------------------------------------------ multi-token
// T consecutive tokens per (batch, head) in one launch: the on-device loop of
// the O(1) cached decode (compiler-first SSD page, abstract).  Each CTA reads
// its P x N state once into registers, applies the tokens in order -- for
// each, the update of every state element and the readout y_t from the
// updated state -- and writes the state back once, so state traffic per token
// falls by T.
//
// The registers hold a scaled state hs = h / sigma, sigma the product of the
// decays since the last rescale, so a token's update is one fused
// multiply-add per element: hs += (dt x / sigma) B.  The readout is
// y = sigma (C . hs) + D x.  The true state is restored (hs *= sigma) at the
// end of every group of staged tokens and before any token that would take
// sigma beyond e^-40 or e^40, so the scaled values stay well inside fp32.
//
// The tokens' x, B and C (and z when gated) are staged in shared memory
// kMultiTok at a time as fp32, with dt x / sigma laid out so that a thread's
// kMultiRows rows of one token are one vector.  A state row of N elements is
// spread over tpr threads (VPT float4 each); a thread keeps rows r0, r0 + rpp,
// ...  The per-row sums C . hs reduce over the tpr threads of a row by
// exchanging halves of the row set, then plain butterflies, and go to shared
// memory; once the group's tokens are applied, one vectorised pass forms
// y = sigma (C . hs) + D x (times silu(z) when gated) and stores it.
constexpr int kMultiTok = 16;      // tokens staged in shared memory at a time
constexpr int kMultiRows = 4;      // state rows a thread keeps in registers (2 or 4)
constexpr int kLogMultiRows = kMultiRows == 4 ? 2 : 1;
constexpr float kMultiRenorm = 40.f;

// threads per CTA and float4 per thread of a row for a state width
__host__ __device__ constexpr int multi_threads(int N) {
    return (N > 128 ? 256 : 128) * (4 / kMultiRows);
}
// CTAs per SM the register budget is set for
__host__ __device__ constexpr int multi_ctas(int N) {
    return (kMultiRows == 4 ? 512 : 768) / multi_threads(N) > 0
               ? (kMultiRows == 4 ? 512 : 768) / multi_threads(N)
               : 1;
}
__host__ __device__ constexpr int multi_vpt(int N) { return N >= 16 ? 4 : N / 4; }
// most state rows (headdim) one CTA holds for a state width
__host__ __device__ constexpr int multi_rows(int N) {
    return kMultiRows * (multi_threads(N) / (N / (4 * multi_vpt(N))));
}
// floats of staged token data: x, the row sums (then y) and z when gated per
// row, dt x / sigma for every row slot, B and C, and four per-token scalars
__host__ __device__ inline size_t multi_smem_floats(int P, int N, bool gated) {
    return (size_t)kMultiTok * ((gated ? 3 : 2) * P + multi_rows(N) + 2 * N + 4);
}

// V consecutive elements (16 bytes or fewer, aligned to their size) as fp32
// in shared memory.
template <int V>
__device__ __forceinline__ void multi_ld_vec(const float *g, float *s) {
    static_assert(V == 4, "fp32 rows load four at a time");
    *reinterpret_cast<float4 *>(s) = *reinterpret_cast<const float4 *>(g);
}
template <int V>
__device__ __forceinline__ void multi_ld_vec(const __nv_bfloat16 *g, float *s) {
    static_assert(V == 4 || V == 8, "bf16 rows load four or eight at a time");
    if constexpr (V == 8) {
        const uint4 u = *reinterpret_cast<const uint4 *>(g);
        *reinterpret_cast<float4 *>(s) =
            make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                        __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
        *reinterpret_cast<float4 *>(s + 4) =
            make_float4(__uint_as_float(u.z << 16), __uint_as_float(u.z & 0xffff0000u),
                        __uint_as_float(u.w << 16), __uint_as_float(u.w & 0xffff0000u));
    } else {
        *reinterpret_cast<float4 *>(s) = ssd_ld4(g);
    }
}
// V consecutive outputs from fp32 values.
template <int V>
__device__ __forceinline__ void multi_st_vec(float *g, const float *v) {
    static_assert(V == 4, "fp32 rows store four at a time");
    *reinterpret_cast<float4 *>(g) = make_float4(v[0], v[1], v[2], v[3]);
}
template <int V>
__device__ __forceinline__ void multi_st_vec(__nv_bfloat16 *g, const float *v) {
    static_assert(V == 8, "bf16 rows store eight at a time");
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
        w[k] = *reinterpret_cast<const uint32_t *>(&b);
    }
    *reinterpret_cast<uint4 *>(g) = make_uint4(w[0], w[1], w[2], w[3]);
}

template <typename T, typename S, int N, bool kFuse>
__global__ void __launch_bounds__(multi_threads(N), multi_ctas(N))
ssd_decode_multi_kernel(S *__restrict__ state, const T *__restrict__ x,
                        const float *__restrict__ dt, const float *__restrict__ A,
                        const T *__restrict__ Bm, const T *__restrict__ Cm,
                        const float *__restrict__ D, T *__restrict__ y, int ntok, int H, int P,
                        int G, const SsdFuse fuse) {
    using namespace ssdptx;
    extern __shared__ float msm[];
    constexpr int NT = multi_threads(N);
    constexpr int VPT = multi_vpt(N);
    constexpr int tpr = N / (4 * VPT);     // threads per row: a power of two <= 16
    constexpr int rpp = NT / tpr;          // rows per pass
    constexpr int PM = multi_rows(N);      // row slots: kMultiRows per thread of a row
    static_assert(kMultiRows == 2 || kMultiRows == 4, "a thread's dt x / sigma of one token is one vector");
    constexpr int VV = 16 / (int)sizeof(T);          // elements of one 16-byte vector
    const int bh = blockIdx.x;             // b * H + h
    const int b = bh / H, h = bh - b * H;
    const int g = h / (H / G);
    const int lane_n = threadIdx.x & (tpr - 1);
    const int r0 = threadIdx.x / tpr;
    griddep_wait();                        // no-ops unless launched programmatically
    griddep_launch_dependents();
    const float Ah = A[h];
    const float Dh = D ? D[h] : 0.0f;
    const float bias = ssd_dt_bias<kFuse>(fuse, h);
    const bool gated = kFuse && fuse.z != nullptr;
    const bool xvec = P % VV == 0;         // x, y, z rows in 16-byte vectors
    float *xs = msm;                         // [kMultiTok][P]  x
    float *ys = xs + kMultiTok * P;          // [kMultiTok][P]  C . hs, per row
    float *us = ys + kMultiTok * P;          // [kMultiTok][rpp][kMultiRows]  dt x / sigma
    float *Bs = us + kMultiTok * PM;         // [kMultiTok][N]
    float *Cs = Bs + kMultiTok * N;          // [kMultiTok][N]
    float *sig = Cs + kMultiTok * N;         // [kMultiTok]: sigma after the token
    float *pre = sig + kMultiTok;            // [kMultiTok]: rescale before the token (1 = none)
    float *dsz = pre + kMultiTok;            // [kMultiTok]: step size
    float *inv = dsz + kMultiTok;            // [kMultiTok]: 1 / sigma
    float *zs = inv + kMultiTok;             // [kMultiTok][P] when gated

    S *st = state + (size_t)bh * P * N;
    float4 s[kMultiRows][VPT];
#pragma unroll
    for (int i = 0; i < kMultiRows; ++i) {
        const int p = r0 + i * rpp;
#pragma unroll
        for (int v = 0; v < VPT; ++v)
            s[i][v] = p < P ? ssd_ld4_cs(st + (size_t)p * N + 4 * (lane_n + v * tpr))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    auto rescale = [&](float f) {
        const float2 f2 = make_float2(f, f);
#pragma unroll
        for (int i = 0; i < kMultiRows; ++i)
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const float2 lo = fmul2(make_float2(s[i][v].x, s[i][v].y), f2);
                const float2 hi = fmul2(make_float2(s[i][v].z, s[i][v].w), f2);
                s[i][v] = make_float4(lo.x, lo.y, hi.x, hi.y);
            }
    };

    for (int t0 = 0; t0 < ntok; t0 += kMultiTok) {
        const int nt = min(kMultiTok, ntok - t0);
        __syncthreads();                     // the previous tokens' staging is consumed
        const size_t row0 = (size_t)b * ntok + t0;   // token row of the [b][T] axis
        if (threadIdx.x < nt)
            dsz[threadIdx.x] = ssd_dt<kFuse>(fuse, dt[(row0 + threadIdx.x) * H + h], bias);
        // B and C four elements at a time; x in 16-byte vectors only when
        // every thread gets one (fewer, wider loads on fewer warps measured
        // slower for short groups)
        for (int e = threadIdx.x * 4; e < nt * N; e += NT * 4) {
            const int t = e / N, n = e - t * N;
            const size_t o = ((row0 + t) * G + g) * N + n;
            multi_ld_vec<4>(Bm + o, Bs + e);
            multi_ld_vec<4>(Cm + o, Cs + e);
        }
        if (xvec && nt * P >= NT * VV) {
            for (int e = threadIdx.x * VV; e < nt * P; e += NT * VV) {
                const int t = e / P;
                const size_t o = ((row0 + t) * H + h) * P + (e - t * P);
                multi_ld_vec<VV>(x + o, xs + e);
                if (gated) multi_ld_vec<VV>(static_cast<const T *>(fuse.z) + o, zs + e);
            }
        } else {
            for (int e = threadIdx.x; e < nt * P; e += NT) {
                const int t = e / P;
                const size_t o = ((row0 + t) * H + h) * P + (e - t * P);
                xs[e] = ssd_ld(x + o);
                if (gated) zs[e] = ssd_ld(static_cast<const T *>(fuse.z) + o);
            }
        }
        __syncthreads();
        // per-token factors: log sigma accumulates dt A.  A token that would
        // take it past +-kMultiRenorm first restores the state (pre = the
        // sigma so far) and restarts sigma at its own decay; a token whose own
        // decay is that large is applied to the restored state directly (pre =
        // sigma so far times it), and sigma restarts at 1.  When no token of
        // the group needs either, the first warp forms the factors from a
        // prefix sum in one step; otherwise one thread walks the tokens.
        bool walk = false;
        if (threadIdx.x < 32) {
            const int ln = threadIdx.x;
            const float l = ln < nt ? dsz[ln] * Ah : 0.f;
            float L = l;
#pragma unroll
            for (int o = 1; o < kMultiTok; o <<= 1) {
                const float v = __shfl_up_sync(0xffffffffu, L, o);
                if (ln >= o) L += v;
            }
            const bool big = ln < nt && (fabsf(l) > kMultiRenorm || fabsf(L) > kMultiRenorm);
            walk = __any_sync(0xffffffffu, big);
            if (!walk && ln < nt) {
                pre[ln] = 1.f;
                sig[ln] = expf(L);
                inv[ln] = expf(-L);
            }
        }
        if (walk && threadIdx.x == 0) {
            float ls = 0.f;
            for (int t = 0; t < nt; ++t) {
                const float l = dsz[t] * Ah;
                float rs = 1.f;
                if (fabsf(l) > kMultiRenorm) {
                    rs = expf(ls + l);
                    ls = 0.f;
                } else if (fabsf(ls + l) > kMultiRenorm) {
                    rs = expf(ls);
                    ls = l;
                } else {
                    ls += l;
                }
                pre[t] = rs;
                sig[t] = expf(ls);
                inv[t] = expf(-ls);
            }
        }
        __syncthreads();
        // dt x / sigma by row slot: slot r * kMultiRows + i is row r + i * rpp
        // (zero past the last row)
        for (int e = threadIdx.x; e < nt * PM; e += NT) {
            const int t = e / PM, k = e - t * PM;
            const int p = k / kMultiRows + (k % kMultiRows) * rpp;
            us[e] = p < P ? (dsz[t] * xs[t * P + p]) * inv[t] : 0.f;
        }
        __syncthreads();

        for (int t = 0; t < nt; ++t) {
            const float rs = pre[t];
            if (rs != 1.f) rescale(rs);       // uniform: every thread reads the same slot
            // update hs += u B and the row's partial readout C . hs (packed
            // pairs), one float4 of B and C at a time for all rows
            float2 u2[kMultiRows];
            if constexpr (kMultiRows == 4) {
                const float4 u4 = *reinterpret_cast<const float4 *>(us + t * PM + kMultiRows * r0);
                u2[0] = make_float2(u4.x, u4.x);
                u2[1] = make_float2(u4.y, u4.y);
                u2[kMultiRows - 2] = make_float2(u4.z, u4.z);
                u2[kMultiRows - 1] = make_float2(u4.w, u4.w);
            } else {
                const float2 uv = *reinterpret_cast<const float2 *>(us + t * PM + kMultiRows * r0);
                u2[0] = make_float2(uv.x, uv.x);
                u2[kMultiRows - 1] = make_float2(uv.y, uv.y);
            }
            float2 a2[kMultiRows];
#pragma unroll
            for (int i = 0; i < kMultiRows; ++i) a2[i] = make_float2(0.f, 0.f);
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const float4 Bv = *reinterpret_cast<const float4 *>(Bs + t * N + 4 * (lane_n + v * tpr));
                const float4 Cv = *reinterpret_cast<const float4 *>(Cs + t * N + 4 * (lane_n + v * tpr));
                const float2 b01 = make_float2(Bv.x, Bv.y), b23 = make_float2(Bv.z, Bv.w);
                const float2 c01 = make_float2(Cv.x, Cv.y), c23 = make_float2(Cv.z, Cv.w);
#pragma unroll
                for (int i = 0; i < kMultiRows; ++i) {
                    const float2 q01 = ffma2(u2[i], b01, make_float2(s[i][v].x, s[i][v].y));
                    const float2 q23 = ffma2(u2[i], b23, make_float2(s[i][v].z, s[i][v].w));
                    s[i][v] = make_float4(q01.x, q01.y, q23.x, q23.y);
                    a2[i] = ffma2(c01, q01, a2[i]);
                    a2[i] = ffma2(c23, q23, a2[i]);
                }
            }
            float acc[kMultiRows];
#pragma unroll
            for (int i = 0; i < kMultiRows; ++i) acc[i] = a2[i].x + a2[i].y;
            // reduce over the tpr threads of each row: at exchange k (offset
            // tpr >> (k+1)) a thread keeps one half of its remaining rows and
            // adds its partner's partials of them; once one row is left, plain
            // butterflies finish the sum
            // (all of it resolved at compile time from tpr)
            int base = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                constexpr int kHalf0 = kMultiRows / 2;
                const int o = tpr >> (k + 1);
                if (o > 0 && k < kLogMultiRows) {
                    const int half = kHalf0 >> k;
                    const bool up = (lane_n & o) != 0;
#pragma unroll
                    for (int j = 0; j < kHalf0; ++j) {
                        if (j < half) {
                            const float send = up ? acc[j] : acc[j + half];
                            const float keep = up ? acc[j + half] : acc[j];
                            acc[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                        }
                    }
                    if (up) base += half;
                } else if (o > 0) {
                    acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], o);
                }
            }
            // rows this thread now holds: base + j for j < left; the lowest
            // thread of each set of equal holders records them
            constexpr int kLogTpr = tpr >= 16 ? 4 : (tpr >= 8 ? 3 : (tpr >= 4 ? 2 : (tpr >= 2 ? 1 : 0)));
            constexpr int rounds = kLogTpr < kLogMultiRows ? kLogTpr : kLogMultiRows;
            constexpr int left = kMultiRows >> rounds;
            constexpr int low = (1 << (kLogTpr - rounds)) - 1;
            if ((lane_n & low) == 0) {
#pragma unroll
                for (int j = 0; j < kMultiRows; ++j) {
                    const int p = r0 + (base + j) * rpp;
                    if (j < left && p < P) ys[t * P + p] = acc[j];
                }
            }
        }
        rescale(sig[nt - 1]);                 // the true state again
        if (t0 + nt >= ntok) {                // last group: the state goes out first
#pragma unroll
            for (int i = 0; i < kMultiRows; ++i) {
                const int p = r0 + i * rpp;
                if (p < P) {
#pragma unroll
                    for (int v = 0; v < VPT; ++v)
                        ssd_st4_cs(st + (size_t)p * N + 4 * (lane_n + v * tpr), s[i][v]);
                }
            }
        }
        __syncthreads();                      // every row sum of the group recorded
        // y = sigma (C . hs) + D x, gated: times silu(z)
        if (xvec) {
            for (int e = threadIdx.x * VV; e < nt * P; e += NT * VV) {
                const int t = e / P;
                const float sg = sig[t];
                float v[VV];
#pragma unroll
                for (int k = 0; k < VV; k += 4) {
                    const float4 yy = *reinterpret_cast<const float4 *>(ys + e + k);
                    const float4 xx = *reinterpret_cast<const float4 *>(xs + e + k);
                    v[k] = sg * yy.x + Dh * xx.x;
                    v[k + 1] = sg * yy.y + Dh * xx.y;
                    v[k + 2] = sg * yy.z + Dh * xx.z;
                    v[k + 3] = sg * yy.w + Dh * xx.w;
                    if (gated) {
                        const float4 zz = *reinterpret_cast<const float4 *>(zs + e + k);
                        v[k] *= ssd_silu(zz.x);
                        v[k + 1] *= ssd_silu(zz.y);
                        v[k + 2] *= ssd_silu(zz.z);
                        v[k + 3] *= ssd_silu(zz.w);
                    }
                }
                multi_st_vec<VV>(y + ((row0 + t) * H + h) * P + (e - t * P), v);
            }
        } else {
            for (int e = threadIdx.x; e < nt * P; e += NT) {
                const int t = e / P;
                float v = sig[t] * ys[e] + Dh * xs[e];
                if (gated) v *= ssd_silu(zs[e]);
                ssd_st(y + ((row0 + t) * H + h) * P + (e - t * P), v);
            }
        }
    }
}

template <typename T, typename S, int N, bool kFuse>
cudaError_t launch_multi_k(S *state, const void *x, const float *dt, const float *A,
                           const void *B, const void *C, const float *D, void *y, int batch,
                           int ntok, int H, int P, int G, int num_sms, const SsdFuse &fuse,
                           cudaStream_t stream) {
    const size_t smem = multi_smem_floats(P, N, kFuse && fuse.z != nullptr) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(ssd_decode_multi_kernel<T, S, N, kFuse>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const size_t units = (size_t)batch * H;
    // programmatic launch for short calls only, as for the streaming kernel
    // (at batch 1 it took 3 % off a 64-layer call of 4 tokens; long calls
    // lost 0.4 %)
    if (num_sms > 0 && units <= (size_t)num_sms * 64)
        return launch_pdl(ssd_decode_multi_kernel<T, S, N, kFuse>, dim3((unsigned)units),
                          dim3(multi_threads(N)), smem, stream, state, (const T *)x, dt, A,
                          (const T *)B, (const T *)C, D, (T *)y, ntok, H, P, G, fuse);
    ssd_decode_multi_kernel<T, S, N, kFuse><<<(unsigned)units, multi_threads(N), smem, stream>>>(
        state, (const T *)x, dt, A, (const T *)B, (const T *)C, D, (T *)y, ntok, H, P, G, fuse);
    return cudaGetLastError();
}

template <typename T, typename S, bool kFuse>
cudaError_t launch_multi_t(S *state, const void *x, const float *dt, const float *A,
                           const void *B, const void *C, const float *D, void *y, int batch,
                           int ntok, int H, int P, int N, int G, int num_sms, const SsdFuse &fuse,
                           cudaStream_t stream) {
#define SSD_MULTI_N(NN)                                                                    \
    case NN:                                                                               \
        return launch_multi_k<T, S, NN, kFuse>(state, x, dt, A, B, C, D, y, batch, ntok, H, P, \
                                               G, num_sms, fuse, stream)
    switch (N) {
        SSD_MULTI_N(4);
        SSD_MULTI_N(8);
        SSD_MULTI_N(16);
        SSD_MULTI_N(32);
        SSD_MULTI_N(64);
        SSD_MULTI_N(128);
        SSD_MULTI_N(256);
        default:
            return cudaErrorInvalidValue;   // dstate is checked by the caller
    }
#undef SSD_MULTI_N
}

}  // namespace

cudaError_t ssd_launch_decode(void *state, bool bf16_state, const void *x, const float *dt,
                              const float *A, const void *B, const void *C,
                              const float *D, void *y, bool bf16, int batch,
                              int H, int P, int N, int G, int num_sms, unsigned int *err,
                              const SsdFuse &fuse, cudaStream_t stream) {
    const bool fused = ssd_fuse_active(fuse);
    using bf = __nv_bfloat16;
    if (bf16_state) {   // bf16 inputs only (checked by the caller)
        bf *st = static_cast<bf *>(state);
        return fused ? launch_t<bf, bf, true>(st, x, dt, A, B, C, D, y, batch, H, P, N, G,
                                              num_sms, err, fuse, stream)
                     : launch_t<bf, bf, false>(st, x, dt, A, B, C, D, y, batch, H, P, N, G,
                                               num_sms, err, fuse, stream);
    }
    float *st = static_cast<float *>(state);
    if (bf16)
        return fused ? launch_t<bf, float, true>(st, x, dt, A, B, C, D, y, batch, H, P, N, G,
                                                 num_sms, err, fuse, stream)
                     : launch_t<bf, float, false>(st, x, dt, A, B, C, D, y, batch, H, P, N, G,
                                                  num_sms, err, fuse, stream);
    return fused ? launch_t<float, float, true>(st, x, dt, A, B, C, D, y, batch, H, P, N, G,
                                                num_sms, err, fuse, stream)
                 : launch_t<float, float, false>(st, x, dt, A, B, C, D, y, batch, H, P, N, G,
                                                 num_sms, err, fuse, stream);
}

int ssd_decode_multi_max_headdim(int N) {
    if (N < 4 || N > 256 || (N & (N - 1)) != 0) return 0;
    return multi_rows(N);
}

cudaError_t ssd_launch_decode_multi(void *state, bool bf16_state, const void *x, const float *dt,
                                    const float *A, const void *B, const void *C,
                                    const float *D, void *y, bool bf16, int batch, int ntok,
                                    int H, int P, int N, int G, int num_sms, const SsdFuse &fuse,
                                    cudaStream_t stream) {
    const bool fused = ssd_fuse_active(fuse);
    using bf = __nv_bfloat16;
    if (bf16_state) {   // bf16 inputs only (checked by the caller)
        bf *st = static_cast<bf *>(state);
        return fused ? launch_multi_t<bf, bf, true>(st, x, dt, A, B, C, D, y, batch, ntok, H, P,
                                                    N, G, num_sms, fuse, stream)
                     : launch_multi_t<bf, bf, false>(st, x, dt, A, B, C, D, y, batch, ntok, H, P,
                                                     N, G, num_sms, fuse, stream);
    }
    float *st = static_cast<float *>(state);
    if (bf16)
        return fused ? launch_multi_t<bf, float, true>(st, x, dt, A, B, C, D, y, batch, ntok, H,
                                                       P, N, G, num_sms, fuse, stream)
                     : launch_multi_t<bf, float, false>(st, x, dt, A, B, C, D, y, batch, ntok, H,
                                                        P, N, G, num_sms, fuse, stream);
    return fused ? launch_multi_t<float, float, true>(st, x, dt, A, B, C, D, y, batch, ntok, H, P,
                                                      N, G, num_sms, fuse, stream)
                 : launch_multi_t<float, float, false>(st, x, dt, A, B, C, D, y, batch, ntok, H,
                                                       P, N, G, num_sms, fuse, stream);
}
