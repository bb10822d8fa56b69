// Tensor-core chunked SSD scan for sm_103a (tcgen05 + TMEM + TMA).
//
// The chunk steps follow "Mamba-Family State-Space Model Kernels on a
// Programmable CGLA", section III.A: Step-1 inside a chunk is GEMM1 (C.B^T,
// reduction over the state size N) -> Hadamard decay mask -> GEMM2
// (reduction over the chunk); Step-3 carries the N x P state across chunks.
// Section IV.B of the same page names the boundary between the mask and
// GEMM2 as the overhead that fusion should remove, and the Mambalaya page
// (Figures 4-5: RI and RSb fusion) fuses Einsums that share an iteration
// space or drop a rank.  Here every step of a 128-token tile stays on chip:
//
//   G     = C . B^T                (tcgen05, smem x smem -> TMEM fp32)
//   M     = G o exp(a_t - a_s) dt_s, s <= t
//                                  (TMEM -> registers -> TMEM as bf16, in place)
//   Yd    = M . X                  (tcgen05 with A read from TMEM)
//   Yo    = C . H_prev^T           (off-diagonal term from the entering state)
//   H    <- exp(a_end) H + B^T . (w o X),  w_s = exp(a_end - a_s) dt_s
//   y     = Yd + exp(a_t) Yo + D x (epilogue, bf16 store)
//
// Exponents are differences of the chunk-local cumsum a, taken inside 32-token
// blocks (the mask factors) or from a tile's start or end: with dt >= 0 and
// A <= 0 none is positive.  dt enters every factor as a multiplier, so its
// sign is not assumed; a negative dt makes the factors grow, and they stay
// finite while that growth inside a tile stays below about e^60.
//
// Parallelism over the sequence: a segment is a run of consecutive tiles
// handled by one CTA with the state carried in TMEM.  When a sequence has more
// than one segment, a first kernel computes each segment's own state
// contribution F (tiles walked backwards so the decay to the segment end is a
// running sum; four heads per CTA for the segments that fill whole waves, two
// for the rest, in a second launch), a small kernel chains them into every
// segment's entering state, and the scan kernel starts each segment from it.  Heads that share a
// group (ngroups divides nheads) are paired in one CTA so C.B^T is computed
// once for both.
//
// Warp roles of the scan kernel (640 threads): warp 1 allocates TMEM and issues
// C.B^T, the state update, the off-diagonal product and the second head's
// masked product; warps 2-17 (four warpgroups) build the masks, keep the state
// and run the epilogue; warp 18 issues the first head's masked product and the
// y stores; warps 0 and 19 are the TMA producer and the factor warp (each
// tile's cumsum of dt A and its exponentials, computed ahead of use), in the
// order the launch picks (template parameter kFacLow).  The segment kernel: warp 0 loads, warp 1 issues,
// warps 2-9 scale X, warp 10 computes the token weights.  Every wait is on an
// mbarrier with a time limit; a wait that runs out sets the device error word
// and the CTA fast-forwards to its exit without further loads or stores.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

using namespace ssdptx;

namespace {

constexpr int kTile = 128;                 // tokens per tile
constexpr int kP = 64;                     // headdim handled by this path
constexpr int kN = 128;                    // dstate handled by this path
constexpr int kXWarps = 16;                // scan kernel: transform/epilogue warps
// scan kernel: producer, MMA issuer A, 16 transform warps, MMA issuer B and a
// factor warp: 20 warps, 5 per SM sub-partition, which keeps the register cap
// at 96 (a 21st warp would lower it to 80).  One thread issues a tcgen05.mma
// only every ~70-100 cycles, longer than an M = 128, N <= 128 instruction
// takes to execute, so two issuing warps feed the tensor core from two
// instruction streams.
constexpr int kThreads = 64 + 32 * kXWarps + 64;
// Warp w runs on SM sub-partition w % 4, and the transform warps' sub-partition
// is fixed by their TMEM lane quarter (warp % 4): quarter 3 has the most mask
// work, quarter 0 the least.  The producer and the factor warp take warps 0 and
// 3 + kXWarps in an order chosen per launch (kFacLow): the factor warp
// on the light sub-partition pays on long segments, the producer there on short
// ones (its first loads are then the critical path).
constexpr int kIssuerA = 1;                // first MMA issuer (also allocates TMEM)
constexpr int kIssuerB = 2 + kXWarps;      // second MMA issuer
constexpr int kSpareWarpLo = 0, kSpareWarpHi = 3 + kXWarps;   // producer / factor warp
constexpr int kLongSegTiles = 24;          // from this many tiles per segment on
constexpr int kSegXWarps = 8;              // segment kernel: X scaling warps
constexpr int kSegFacWarp = 2 + kSegXWarps;  // segment kernel: token weight warp
constexpr int kSegThreads = 64 + 32 * kSegXWarps + 32;
// segment kernel: B + X stages (4 heads per CTA: 96 KB stages, two fit)
constexpr int seg_stages(int hg) { return hg == 4 ? 2 : 3; }
// Largest decay (in log units) across one 32-token block for which the mask's
// diagonal block uses the factored form (its R_t factor stays below e^60).
constexpr float kMaxBlockDecay = 60.f;

constexpr uint32_t kBlk = 16384;           // 128 rows x 128 bytes, 128B-swizzled
constexpr uint32_t kCBytes = 2 * kBlk;     // C tile: 128 tokens x 128 n
constexpr uint32_t kBBytes = 2 * kBlk;     // B tile
constexpr uint32_t kXBytes = kBlk;         // X tile: 128 tokens x 64 p
constexpr uint32_t kHbBytes = 16384;       // bf16 entering state, 128 n rows x 64 p
constexpr uint32_t kCtrl = 3072;           // barriers and per-tile scalars

// TMEM columns of the scan kernel
constexpr uint32_t kColG = 0;              // G, then M for both heads in place
constexpr uint32_t kColYd = 128;           // + 64 h : intra-chunk output
constexpr uint32_t kColYo = 256;           // + 64 h : off-diagonal output
constexpr uint32_t kColH = 384;            // + 64 h : carried state (lane = n, column = p)

constexpr uint32_t kIdG = idesc_bf16_f32(128, 128, false, false);   // C . B^T
constexpr uint32_t kIdOff = idesc_bf16_f32(128, 64, false, true);   // C . Hb (Hb rows = n)
constexpr uint32_t kIdS = idesc_bf16_f32(128, 64, true, true);      // B^T . Xt
constexpr uint32_t kIdY = idesc_bf16_f32(128, 64, false, true);     // M(TMEM) . X

// control-region offsets (bytes)
constexpr uint32_t kOffTslot = 192;       // (barriers occupy bytes 0 .. 159)
constexpr uint32_t kOffAbort = 196;
constexpr uint32_t kOffLast = 200;        // int[3]: last tile of X, B, C loads issued
// scan kernel factor slot, written by the factor warp for one tile at a time
constexpr uint32_t kOffAch = 256;         // float[2][4]: a at the end of each 32-token block
constexpr uint32_t kOffAt = 512;          // float[2][128]: a_t, chunk-local inclusive cumsum of dt A
constexpr uint32_t kOffV = 1536;          // float[2][128]: exp(a_end(32-block of s) - a_s) dt_s

struct TcArgs {
    const float *dt, *A, *D, *init;
    // [b][nseg-1][H][P][N] bf16: segment contributions, then entering states
    // (fp32 in TMEM and in the chaining arithmetic, rounded to bf16 in HBM)
    __nv_bfloat16 *ws_state;
    float *ws_decay;       // [b][nseg-1][H]: segment total decay
    __nv_bfloat16 *y;
    float *fin;
    unsigned int *err;
    int L, H, G, tiles, seg_tiles, nseg;
    SsdFuse fuse;             // transform of the raw step size
    // packed sequences (cu != nullptr): tokens cu[s] .. cu[s+1]-1 of the
    // flattened token axis form sequence s; item0 / fslot0 [nseq + 1] are the
    // prefix sums of each sequence's segments and of its segments but the last
    const int *cu;
    const int *item0, *fslot0;
    int nseq;
    uint64_t wait_ns;         // limit of every bounded wait (ns)
    int fault;                // host-set fault injection (SSD_FAULT_*), 0 = none
    int sigma0;               // batched segment kernel: segment of grid row y = 0
};

// Where one CTA's segment lies: its sequence, the sequence's first row in the
// flattened token axis, its length, tiles and segments, the segment's index,
// and the workspace slot of the sequence's first segment contribution.
struct SegWork {
    size_t grow0;
    int seq, len, tiles, nseg, sigma, fslot;
};

// The segment of CTA (item, z): batched sequences are z with `item` the
// segment; packed ones are found by binary search of the prefix tables (over
// all segments, or over all but each sequence's last when `nonlast`).
template <bool kPacked>
__device__ __forceinline__ SegWork seg_work(const TcArgs &a, int item, int z, bool nonlast) {
    SegWork w;
    if (!kPacked) {
        w.seq = z;
        w.grow0 = (size_t)z * a.L;
        w.len = a.L;
        w.tiles = a.tiles;
        w.nseg = a.nseg;
        w.sigma = item;
        w.fslot = z * (a.nseg - 1);
        return w;
    }
    const int *pre = nonlast ? a.fslot0 : a.item0;
    int lo = 0, hi = a.nseq;                  // the last s with pre[s] <= item
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pre[mid] <= item) lo = mid;
        else hi = mid;
    }
    w.seq = lo;
    w.grow0 = (size_t)a.cu[lo];
    w.len = a.cu[lo + 1] - a.cu[lo];
    w.tiles = (w.len + kTile - 1) / kTile;
    w.nseg = (w.tiles + a.seg_tiles - 1) / a.seg_tiles;
    w.sigma = item - pre[lo];
    w.fslot = a.fslot0[lo];
    return w;
}

// The step-size transform of a layer (bias, softplus, clamp) applied once to
// every dt of the call, into the workspace, before the tensor-core kernels
// read it.  Elementwise and HBM-bound: a round trip of 8 bytes per (token,
// head), about 1% of a scan's traffic, where carrying the transform inside
// the single warps that make the per-token factors put it on their critical
// path (the segment kernel ran 45% slower).
__global__ void __launch_bounds__(256)
ssd_dt_prepass_kernel(const float *__restrict__ dt, float *__restrict__ out, size_t n, int H,
                      const SsdFuse f) {
    for (size_t i = (size_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (size_t)gridDim.x * 256)
        out[i] = ssd_dt<true>(f, dt[i], ssd_dt_bias<true>(f, (int)(i % (size_t)H)));
}

// Prefix tables of packed sequences for the kernels above: item0[s] = segments
// of sequences before s, fslot0[s] = their segments but each one's last.  One
// block walks the sequences 1024 at a time.  An empty sequence has no segment
// (no CTA visits it), so this kernel also gives it its final state: the
// initial one (zeros without init), `hpn` = heads x P x N floats.
__global__ void __launch_bounds__(1024)
ssd_varlen_plan_kernel(const int *__restrict__ cu, int nseq, int seg_tiles, int *item0,
                       int *fslot0, const float *__restrict__ init, float *__restrict__ fin,
                       int hpn) {
    __shared__ int wsum[2][32];
    __shared__ int carry[2];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) carry[0] = carry[1] = 0;
    __syncthreads();
    for (int base = 0; base < nseq; base += 1024) {
        const int s = base + tid;
        int n = 0;
        if (s < nseq) {
            const int tiles = (cu[s + 1] - cu[s] + kTile - 1) / kTile;
            n = (tiles + seg_tiles - 1) / seg_tiles;
        }
        int v[2] = {n, n > 0 ? n - 1 : 0};
        int incl[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            incl[k] = v[k];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, incl[k], off);
                if (lane >= off) incl[k] += o;
            }
            if (lane == 31) wsum[k][warp] = incl[k];
        }
        __syncthreads();
        if (warp == 0) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                int t = wsum[k][lane];
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int o = __shfl_up_sync(0xffffffffu, t, off);
                    if (lane >= off) t += o;
                }
                wsum[k][lane] = t;        // inclusive over warps
            }
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int before = carry[k] + (warp > 0 ? wsum[k][warp - 1] : 0) + incl[k] - v[k];
            if (s < nseq) (k == 0 ? item0 : fslot0)[s] = before;
        }
        __syncthreads();
        if (tid == 0) {
            carry[0] += wsum[0][31];
            carry[1] += wsum[1][31];
        }
        __syncthreads();
    }
    if (tid == 0) {
        item0[nseq] = carry[0];
        fslot0[nseq] = carry[1];
    }
    if (!fin) return;
    for (int s = 0; s < nseq; ++s) {
        if (cu[s + 1] != cu[s]) continue;
        const size_t o = (size_t)s * hpn;
        for (int i = tid; i < hpn; i += 1024) fin[o + i] = init ? init[o + i] : 0.f;
    }
}

// A bounded wait on an mbarrier phase.  After any wait of the CTA has run out
// (abort_flag set) every later wait returns false at once.  The producers and
// the MMA issuers then stop issuing; the transform warps run out their loops
// without waiting (their tensor-memory loads and stores are synchronous and
// stay inside the CTA's own allocation, and they store no y by TMA); the CTA
// drains what it has in flight at its exit and frees its tensor memory.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                         unsigned int *err, uint64_t limit_ns) {
    if (*abort_flag) return false;
    if (mbar_wait(bar, parity, limit_ns)) return true;
    *abort_flag = 1;
    ssd_report(err, SSD_DEVERR_TIMEOUT);
    return false;
}

// Warp-uniform wait (every lane polls; the warp proceeds only if all saw it).
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity,
                                              volatile int *abort_flag, unsigned int *err,
                                              uint64_t limit_ns) {
    const bool ok = wait_bar(bar, parity, abort_flag, err, limit_ns);
    return __all_sync(0xffffffffu, ok);
}

// Drain wait: for the CTA's own copies or tensor-core work to complete before
// it frees tensor memory and exits.  Unlike wait_bar it does not give up when
// another wait has run out (that work completes regardless of the other
// warps); it is bounded all the same, and records a timeout if it runs out.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          unsigned int *err, uint64_t limit_ns) {
    if (mbar_wait(bar, parity, limit_ns)) return;
    *abort_flag = 1;
    ssd_report(err, SSD_DEVERR_TIMEOUT);
}

// Byte offset of element (row, col) in a 128-byte-swizzled tile whose rows are
// 64 bf16 wide (row r of an 8-row, 1024-byte atom; 16-byte chunk c lands at
// c ^ (r % 8)).
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t col) {
    return (row >> 3) * 1024u + (row & 7u) * 128u + ((((col >> 3) ^ row) & 7u) << 4) +
           (col & 7u) * 2u;
}

__device__ __forceinline__ uint4 scale_bf16x8(uint4 v, float w) {
    const uint32_t in[4] = {v.x, v.y, v.z, v.w};
    const uint64_t w2 = pack_f32x2(w, w);
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        out[i] = pack_bf16x2_from_f32x2(mul_f32x2(
            pack_f32x2(__uint_as_float(in[i] << 16), __uint_as_float(in[i] & 0xffff0000u)), w2));
    return make_uint4(out[0], out[1], out[2], out[3]);
}
// The same with w rounded to bf16 first and bf16x2 multiplies (four instructions
// instead of about twenty, for an extra relative error of at most 2^-9 from w).
__device__ __forceinline__ uint4 scale_bf16x8_bf(uint4 v, float w) {
    const uint32_t w2 = pack_bf16x2(w, w);
    return make_uint4(mul_bf16x2(v.x, w2), mul_bf16x2(v.y, w2), mul_bf16x2(v.z, w2),
                      mul_bf16x2(v.w, w2));
}

// ============================================================ scan kernel
// Shared memory (HG heads per CTA): two stages of {C tile, X tile per head},
// one B tile, the bf16 entering states of all heads (Hb) and the w o X
// operands of all heads (Xt).  Merging the heads' off-diagonal and
// state-update products into one N = 64 * HG instruction stream halves their
// instruction count: the tensor core spends about the same time on an
// M = 128 instruction with N = 64 as with N = 128.
template <int HG>
struct ScanLayout {
    static constexpr uint32_t kStage = kCBytes + HG * kXBytes;      // C + X of each head
    static constexpr uint32_t kOffB = 2 * kStage;
    static constexpr uint32_t kOffHb = kOffB + kBBytes;
    static constexpr uint32_t kOffXt = kOffHb + HG * kXBytes;
    static constexpr uint32_t kBytes = kOffXt + HG * kXBytes;
};

template <int HG, bool kFacLow, bool kGate, bool kPacked>
__global__ void __launch_bounds__(kThreads, 1)
ssd_tc_scan_kernel(const __grid_constant__ CUtensorMap mapC,
                   const __grid_constant__ CUtensorMap mapB,
                   const __grid_constant__ CUtensorMap mapX,
                   const __grid_constant__ CUtensorMap mapY,
                   const __grid_constant__ CUtensorMap mapZ, const TcArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    using Lay = ScanLayout<HG>;
    constexpr uint32_t kStage = Lay::kStage;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h0 = blockIdx.x * HG;
    const SegWork w = seg_work<kPacked>(a, blockIdx.y, blockIdx.z, false);
    // batched: from the grid and the kernel parameters at each use (nothing
    // held in registers across the kernel); packed: from the prefix tables
    auto w_seq = [&]() -> int { return kPacked ? w.seq : (int)blockIdx.z; };
    auto w_grow0 = [&]() -> size_t { return kPacked ? w.grow0 : (size_t)blockIdx.z * a.L; };
    auto w_len = [&]() -> int { return kPacked ? w.len : a.L; };
    auto w_tiles = [&]() -> int { return kPacked ? w.tiles : a.tiles; };
    auto w_nseg = [&]() -> int { return kPacked ? w.nseg : a.nseg; };
    auto w_sigma = [&]() -> int { return kPacked ? w.sigma : (int)blockIdx.y; };
    auto w_fslot = [&]() -> int { return kPacked ? w.fslot : (int)blockIdx.z * (a.nseg - 1); };
    const int sigma = w_sigma();
    const int g = h0 / (a.H / a.G);
    const int k0 = sigma * a.seg_tiles;
    const int k1 = min(w_tiles(), k0 + a.seg_tiles);
    const int ntile = k1 - k0;
    // TMA coordinates of the sequence's token t: row trow + t of batch tb
    const int trow = kPacked ? (int)w_grow0() : 0;
    const int tb = kPacked ? 0 : w_seq();
    // a packed sequence's partial last tile is written row by row, not by a
    // TMA store (whose box would run into the next sequence)
    auto partial = [&](int it) { return kPacked && (k0 + it + 1) * kTile > w_len(); };

    const uint32_t sbase = smem_u32(smem);
    if ((sbase & 1023u) != 0u) {
        if (threadIdx.x == 0) ssd_report(a.err, SSD_DEVERR_SMEM_ALIGN);
        return;
    }
    // barriers: 0,1 fullC[stage]; 2,3 emptyC[stage]; 4 fullB; 5 emptyB;
    //           6 g_full; 7 m_ready; 8 hx_ready; 9 hx_free; 10 y_full;
    //           11 y_done (Yd / Yo read, y staged over C); 12 g_free (the masks
    //           in TMEM have been consumed); 13 fac_ready (factor slot written);
    //           14,15 fullX[stage]; 16,17 emptyX[stage]; 18, 19 drain of issuer
    //           A's / issuer B's tensor-core work before the CTA exits
    auto bar = [&](int i) { return sbase + 8u * (uint32_t)i; };
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + kOffTslot);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffAbort);
    float *ach_s = reinterpret_cast<float *>(smem + kOffAch);
    float *at_s = reinterpret_cast<float *>(smem + kOffAt);
    float *v_s = reinterpret_cast<float *>(smem + kOffV);
    const uint32_t tiles_base = sbase + kCtrl;
    const uint32_t b_base = tiles_base + Lay::kOffB;
    const uint32_t hb_base = tiles_base + Lay::kOffHb;
    const uint32_t xt_base = tiles_base + Lay::kOffXt;
    uint8_t *tiles_ptr = smem + kCtrl;
    uint8_t *hb_ptr = tiles_ptr + Lay::kOffHb;
    uint8_t *xt_ptr = tiles_ptr + Lay::kOffXt;

    if (threadIdx.x == 0) {
        mbar_init(bar(0), 1);
        mbar_init(bar(1), 1);
        // a C tile (which holds the tile's y once the epilogue is done) is free
        // once the tile's off-diagonal product is done and the y store has read
        // it; an X tile once the masked product and the epilogue's skip term
        // (every transform warp) have read it
        mbar_init(bar(2), 2);
        mbar_init(bar(3), 2);
        mbar_init(bar(14), 1);
        mbar_init(bar(15), 1);
        mbar_init(bar(16), HG + kXWarps);
        mbar_init(bar(17), HG + kXWarps);
        mbar_init(bar(4), 1);
        mbar_init(bar(5), 1);
        mbar_init(bar(6), 1);
        mbar_init(bar(7), kXWarps);
        mbar_init(bar(8), kXWarps);
        mbar_init(bar(9), 1);
        mbar_init(bar(10), 2);
        mbar_init(bar(11), kXWarps);
        mbar_init(bar(12), HG);                // one commit per masked-product issuer
        // fault injection (host-set, tests only): in the first segment the
        // factors-ready barrier waits for a second arrival that never comes,
        // so the transform warps' first wait for the factors runs out
        mbar_init(bar(13), (a.fault == kSsdFaultWithholdSignal && sigma == 0) ? 2 : 1);
        mbar_init(bar(18), 1);
        mbar_init(bar(19), 1);
        int *last = reinterpret_cast<int *>(smem + kOffLast);
        last[0] = last[1] = last[2] = -1;
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tslot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    constexpr int fac_warp = kFacLow ? kSpareWarpLo : kSpareWarpHi;
    constexpr int producer_warp = kFacLow ? kSpareWarpHi : kSpareWarpLo;
    if (warp == producer_warp) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&mapC);
            tma_prefetch_desc(&mapB);
            tma_prefetch_desc(&mapX);
            // the last tile whose X, B and C loads were issued, for the drain
            int lastX = -1, lastB = -1, lastC = -1;
            for (int it = 0; it < ntile; ++it) {
                const int stage = it & 1;
                const int t0 = (k0 + it) * kTile;
                // Loads go out in the order their buffers free up: X (read last by
                // the epilogue two tiles ago), B (by the previous state update),
                // then C (by the y store two tiles ago).
                const uint32_t stg = tiles_base + stage * kStage;
                // X of this tile
                if (it >= 2 && !wait_bar(bar(16 + stage), ((it >> 1) - 1) & 1, abort_flag, a.err, a.wait_ns))
                    break;
                lastX = it;
                mbar_arrive_expect_tx(bar(14 + stage), HG * kXBytes);
#pragma unroll
                for (int h = 0; h < HG; ++h)
                    tma_load_4d(stg + kCBytes + h * kXBytes, &mapX, bar(14 + stage), 0, h0 + h,
                                trow + t0, tb);
                if constexpr (kGate) {
                    // the gate's z tile into L2: the epilogue reads it about two
                    // tiles from now (rows past a packed sequence's end are
                    // fetched but never read)
#pragma unroll
                    for (int h = 0; h < HG; ++h) tma_prefetch_l2_4d(&mapZ, 0, h0 + h, trow + t0, tb);
                }
                // B of this tile (single buffer: free once the previous tile's state
                // update has read it)
                if (it >= 1 && !wait_bar(bar(5), (it - 1) & 1, abort_flag, a.err, a.wait_ns)) break;
                lastB = it;
                mbar_arrive_expect_tx(bar(4), kBBytes);
                tma_load_4d(b_base, &mapB, bar(4), 0, g, trow + t0, tb);
                tma_load_4d(b_base + kBlk, &mapB, bar(4), 64, g, trow + t0, tb);
                // C of this tile (stage last used two tiles ago)
                if (it >= 2 && !wait_bar(bar(2 + stage), ((it >> 1) - 1) & 1, abort_flag, a.err, a.wait_ns))
                    break;
                lastC = it;
                mbar_arrive_expect_tx(bar(stage), kCBytes);
                tma_load_4d(stg, &mapC, bar(stage), 0, g, trow + t0, tb);
                tma_load_4d(stg + kBlk, &mapC, bar(stage), 64, g, trow + t0, tb);
            }
            // for the drain at exit after a wait ran out
            int *last = reinterpret_cast<int *>(smem + kOffLast);
            last[0] = lastX;
            last[1] = lastB;
            last[2] = lastC;
        }
    } else if (warp == kIssuerA) {
        // ------------------------------------------------------ MMA issuer
        // Descriptors are built once; a K step only adds its byte offset / 16 to
        // the start-address field.
        if (lane == 0) {
            constexpr uint32_t kIdOffAll = idesc_bf16_f32(128, 64 * HG, false, true);
            constexpr uint32_t kIdSAll = idesc_bf16_f32(128, 64 * HG, true, true);
            const uint64_t cK0 = smem_desc(tiles_base, 16, 1024, kSwizzle128B);
            const uint64_t bK = smem_desc(b_base, 16, 1024, kSwizzle128B);
            const uint64_t bMN = smem_desc(b_base, kBlk, 1024, kSwizzle128B);
            const uint64_t hbD = smem_desc(hb_base, kXBytes, 1024, kSwizzle128B);
            const uint64_t xtD = smem_desc(xt_base, kXBytes, 1024, kSwizzle128B);
            const uint64_t xlastD = smem_desc(tiles_base + kCBytes + (HG - 1) * kXBytes, kBlk, 1024,
                                              kSwizzle128B);
            for (int it = 0; it < ntile; ++it) {
                const int stage = it & 1;
                const uint64_t so = stage ? (uint64_t)(kStage >> 4) : 0ull;
                const uint64_t cK = cK0 + so;
                if (!wait_bar(bar(stage), (it >> 1) & 1, abort_flag, a.err, a.wait_ns)) break;
                if (!wait_bar(bar(4), it & 1, abort_flag, a.err, a.wait_ns)) break;
                // the previous tile's masks (in the G columns) must have been read
                if (it > 0 && !wait_bar(bar(12), (it - 1) & 1, abort_flag, a.err, a.wait_ns)) break;
                tc_fence_after();
                // G = C . B^T  (M = 128 tokens t, N = 128 tokens s, K = 128 n)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ko = ((kk >> 2) * kBlk + (kk & 3) * 32) >> 4;
                    mma_ss(tmem + kColG, cK + ko, bK + ko, kIdG, kk > 0);
                }
                mma_commit(bar(6));
                // all heads' state update: H += B^T . Xt (chunk state onto the decayed
                // state), then the off-diagonal term Yo = C . Hb from the entering state
                if (!wait_bar(bar(8), it & 1, abort_flag, a.err, a.wait_ns)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss(tmem + kColH, bMN + (uint64_t)(kk * 128), xtD + (uint64_t)(kk * 128),
                           kIdSAll, 1);
                mma_commit(bar(5));                     // B may be reloaded
                if (it > 0 && !wait_bar(bar(11), (it - 1) & 1, abort_flag, a.err, a.wait_ns)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ko = ((kk >> 2) * kBlk + (kk & 3) * 32) >> 4;
                    mma_ss(tmem + kColYo, cK + ko, hbD + (uint64_t)(kk * 128), kIdOffAll, kk > 0);
                }
                mma_commit(bar(9));                     // Hb / Xt free, H updated
                mma_commit(bar(2 + stage));
                if (HG == 2) {
                    // the second head's masked product, split off issuer B's stream
                    if (!wait_bar(bar(14 + stage), (it >> 1) & 1, abort_flag, a.err, a.wait_ns)) break;
                    if (!wait_bar(bar(7), it & 1, abort_flag, a.err, a.wait_ns)) break;
                    tc_fence_after();
                    const uint64_t xD = xlastD + (stage ? (uint64_t)(kStage >> 4) : 0ull);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t acol = kColG + 32 * (kk >> 1) + 16 * (HG - 1) + 8 * (kk & 1);
                        mma_ts(tmem + kColYd + 64 * (HG - 1), tmem + acol, xD + (uint64_t)(kk * 128),
                               kIdY, kk > 0);
                    }
                    mma_commit(bar(12));
                    mma_commit(bar(16 + stage));
                }
                mma_commit(bar(10));
            }
        }
    } else if (warp == kIssuerB) {
        // ------------------------------------------------ MMA issuer B
        // Intra-chunk output Yd_0 = M_0 . X_0 once the masks are in TMEM.  It
        // also sends out each tile's y (staged over its C tile by the epilogue)
        // by TMA as soon as the epilogue is done, and releases that C buffer
        // once the store has read it.
        if (lane == 0) {
            const uint64_t x00 = smem_desc(tiles_base + kCBytes, kBlk, 1024, kSwizzle128B);
            auto store_y = [&](int k) {
                const uint32_t ys = tiles_base + (k & 1) * kStage;
                if (!partial(k)) {
#pragma unroll
                    for (int h = 0; h < HG; ++h)
                        tma_store_4d(&mapY, ys + h * kBlk, 0, h0 + h, trow + (k0 + k) * kTile, tb);
                }
                bulk_commit();
            };
            int it = 0;
            for (; it < ntile; ++it) {
                const int stage = it & 1;
                const uint64_t xD = x00 + (stage ? (uint64_t)(kStage >> 4) : 0ull);
                if (it > 0) {
                    // tile it-1's y is staged and its Yd read: store it, reuse Yd
                    if (!wait_bar(bar(11), (it - 1) & 1, abort_flag, a.err, a.wait_ns)) break;
                    store_y(it - 1);
                }
                if (!wait_bar(bar(14 + stage), (it >> 1) & 1, abort_flag, a.err, a.wait_ns)) break;
                if (!wait_bar(bar(7), it & 1, abort_flag, a.err, a.wait_ns)) break;
                if (it > 0) {
                    bulk_wait_read<0>();
                    mbar_arrive(bar(2 + (stage ^ 1)));       // tile it-1's C buffer
                }
                tc_fence_after();
                // head 0 (issuer A takes the second head of a pair)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t acol = kColG + 32 * (kk >> 1) + 8 * (kk & 1);
                    mma_ts(tmem + kColYd, tmem + acol, xD + (uint64_t)(kk * 128), kIdY, kk > 0);
                }
                mma_commit(bar(12));
                mma_commit(bar(16 + stage));
                mma_commit(bar(10));
            }
            if (it == ntile && ntile > 0 &&
                wait_bar(bar(11), (ntile - 1) & 1, abort_flag, a.err, a.wait_ns))
                store_y(ntile - 1);
            bulk_wait_all();                                 // y stores complete before exit
        }
    } else if (warp == fac_warp) {
        // ------------------------------------------------------ decay factors
        // Lane l owns tokens 4l .. 4l+3 of a tile.  The factors of tile k are
        // computed in registers ahead of time and written to the slot (a_t, the
        // block ends, v_s) once every mask of tile k-1 is built: the masks are
        // the last readers of the previous tile's v_s.
        float Af[HG], dn[HG][4];
        float fa[HG][4], fv[HG][4], fe[HG][4];
#pragma unroll
        for (int h = 0; h < HG; ++h) Af[h] = a.A[h0 + h];
        auto load_dt4 = [&](int it) {
            const int tok0 = (k0 + it) * kTile + 4 * lane;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int tok = tok0 + i;
#pragma unroll
                for (int h = 0; h < HG; ++h)
                    dn[h][i] = tok < w_len() ? a.dt[(w_grow0() + tok) * a.H + h0 + h] : 0.f;
            }
        };
        // chunk-local inclusive cumsum a_t of dt A, the 32-block ends a_e(j) and
        // v_s = exp(a_e(block of s) - a_s) dt_s, from the raw dt values in dn
        // (tile it); the transform is applied here, not at the load, so the
        // loads stay in flight until the values are needed
        auto factors = [&](int it) {
            const int tok0 = (k0 + it) * kTile + 4 * lane;
#pragma unroll
            for (int h = 0; h < HG; ++h)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    dn[h][i] = tok0 + i < w_len() ? dn[h][i] : 0.f;
#pragma unroll
            for (int h = 0; h < HG; ++h) {
                float c[4];
                c[0] = dn[h][0] * Af[h];
#pragma unroll
                for (int i = 1; i < 4; ++i) c[i] = c[i - 1] + dn[h][i] * Af[h];
                float incl = c[3];
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float o = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl += o;
                }
                float excl = __shfl_up_sync(0xffffffffu, incl, 1);
                if (lane == 0) excl = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) fa[h][i] = excl + c[i];
#pragma unroll
                for (int j = 0; j < 4; ++j) fe[h][j] = __shfl_sync(0xffffffffu, fa[h][3], 8 * j + 7);
                const int jb = lane >> 3;
                const float ae = jb == 0 ? fe[h][0] : (jb == 1 ? fe[h][1] : (jb == 2 ? fe[h][2] : fe[h][3]));
#pragma unroll
                for (int i = 0; i < 4; ++i) fv[h][i] = __expf(ae - fa[h][i]) * dn[h][i];
            }
        };
        auto publish = [&]() {
#pragma unroll
            for (int h = 0; h < HG; ++h) {
                *reinterpret_cast<float4 *>(at_s + h * kTile + 4 * lane) =
                    make_float4(fa[h][0], fa[h][1], fa[h][2], fa[h][3]);
                *reinterpret_cast<float4 *>(v_s + h * kTile + 4 * lane) =
                    make_float4(fv[h][0], fv[h][1], fv[h][2], fv[h][3]);
            }
            if (lane < 4 * HG) {
                float e = 0.f;       // fe[lane / 4][lane % 4] by selects
#pragma unroll
                for (int h = 0; h < HG; ++h)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (lane == 4 * h + j) e = fe[h][j];
                ach_s[lane] = e;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(13));
        };
        if (ntile > 0) {
            load_dt4(0);
            factors(0);
            publish();
            if (ntile > 1) load_dt4(1);
        }
        for (int it = 0; it + 1 < ntile; ++it) {
            factors(it + 1);                                 // tile it + 1
            if (it + 2 < ntile) load_dt4(it + 2);            // in flight meanwhile
            wait_bar_warp(bar(7), it & 1, abort_flag, a.err, a.wait_ns);
            publish();
        }
    } else {
        // ------------------------------------------- transform / epilogue
        // 16 warps = 4 warpgroups.  Thread `row` owns TMEM lane row: token t
        // for the G / M / Y accumulators, state index n for H.
        const int tw = warp - 2;
        const int wg = tw >> 2;               // warpgroup 0..3
        const int q = warp & 3;               // TMEM lane quarter
        const int row = 32 * q + lane;
        const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
        float Dh[HG];
#pragma unroll
        for (int h = 0; h < HG; ++h) Dh[h] = a.D ? a.D[h0 + h] : 0.f;
        // this thread's token: dt_t (this tile's and, in flight, the next
        // tile's), a_t, the tile's 32-block ends a_e(j) and the state weight
        // w_t = exp(a_end - a_t) dt_t
        float at[HG], ach[HG][4], wt[HG];
        auto load_factors = [&](int it) {
            wait_bar_warp(bar(13), it & 1, abort_flag, a.err, a.wait_ns);
#pragma unroll
            for (int h = 0; h < HG; ++h) {
                const float4 e = *reinterpret_cast<const float4 *>(ach_s + 4 * h);
                ach[h][0] = e.x;
                ach[h][1] = e.y;
                ach[h][2] = e.z;
                ach[h][3] = e.w;
                at[h] = at_s[h * kTile + row];
                const float aq = q == 0 ? e.x : (q == 1 ? e.y : (q == 2 ? e.z : e.w));
                wt[h] = v_s[h * kTile + row] * __expf(e.w - aq);
            }
        };

        // ---- all heads of tile it: entering state -> bf16 operand (MN-major rows n),
        //      state scaled by the tile decay, and Xt = w o X
        auto prep_tile = [&](int it) {
            const uint8_t *stg_ptr = tiles_ptr + (it & 1) * kStage;
            if (it > 0) wait_bar_warp(bar(9), (it - 1) & 1, abort_flag, a.err, a.wait_ns);
            tc_fence_after();
            if (it == 0 && sigma > 0) griddep_wait();   // entering states of later segments
#pragma unroll
            for (int h = 0; h < HG; ++h) {
                const float de = __expf(ach[h][3]);
                const uint32_t colH = kColH + 64 * h + 16 * wg;
                uint32_t r[16];
                if (it == 0 && sigma == 0) {
                    const float *src =
                        a.init ? a.init + ((size_t)w_seq() * a.H + h0 + h) * kP * kN : nullptr;
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        r[j] = __float_as_uint(src ? src[(size_t)(16 * wg + j) * kN + row] : 0.f);
                } else if (it == 0) {
                    const __nv_bfloat16 *src =
                        a.ws_state + ((size_t)(w_fslot() + sigma - 1) * a.H + h0 + h) * kP * kN;
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        r[j] = __float_as_uint(__bfloat162float(src[(size_t)(16 * wg + j) * kN + row]));
                } else {
                    tmem_ld16(tq + colH, r);
                    tmem_ld_wait();
                }
                uint32_t pk[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    pk[e] = pack_bf16x2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
                uint8_t *hb = hb_ptr + h * kXBytes;
                *reinterpret_cast<uint4 *>(hb + sw128(row, 16 * wg)) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
                *reinterpret_cast<uint4 *>(hb + sw128(row, 16 * wg + 8)) =
                    make_uint4(pk[4], pk[5], pk[6], pk[7]);
                const uint64_t de2 = pack_f32x2(de, de);
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                    const uint64_t v = mul_f32x2(pack_f32x2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), de2);
                    r[j] = (uint32_t)v;
                    r[j + 1] = (uint32_t)(v >> 32);
                }
                tmem_st16(tq + colH, r);
            }
            // the X tile is needed only now: its landing overlaps the state half
            wait_bar_warp(bar(14 + (it & 1)), (it >> 1) & 1, abort_flag, a.err, a.wait_ns);
#pragma unroll
            for (int h = 0; h < HG; ++h) {
                const uint8_t *xs = stg_ptr + kCBytes + h * kXBytes;
                uint8_t *xt = xt_ptr + h * kXBytes;
#pragma unroll
                for (int c = 2 * wg; c < 2 * wg + 2; ++c) {
                    const uint32_t off = sw128(row, 8 * c);
                    *reinterpret_cast<uint4 *>(xt + off) =
                        scale_bf16x8(*reinterpret_cast<const uint4 *>(xs + off), wt[h]);
                }
            }
            fence_proxy_async_smem();
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(8));
        };

        // Software pipeline: the next tile's state prep runs while the tensor core
        // finishes this tile, then this tile's epilogue.  A wait that fails (one
        // of the CTA's waits ran out) ends the loop.
        if (ntile > 0) {
            load_factors(0);
            prep_tile(0);
        }
        for (int it = 0; it < ntile; ++it) {
            const int t0 = (k0 + it) * kTile;
            const int stage = it & 1;
            const uint8_t *stg_ptr = tiles_ptr + stage * kStage;

            // ---- mask for the 32-token column block j = wg, all heads:
            //      M = G o exp(a_t - a_s) dt_s (s <= t).
            //      exp(a_t - a_s) dt_s = R_t v_s with R_t = exp(a_t - a_e(j)) and
            //      v_s = exp(a_e(j) - a_s) dt_s, e(j) the block's last token: left of
            //      the diagonal both factors are <= 1; on the diagonal block R_t is
            //      >= 1 but bounded by the block's own decay, and a block whose decay
            //      exceeds kMaxBlockDecay falls back to one exponential per element.
            wait_bar_warp(bar(6), it & 1, abort_flag, a.err, a.wait_ns);
            tc_fence_after();
            {
                const int j = wg;
                uint32_t gr[32];
                tmem_ld32(tq + kColG + 32 * j, gr);
                tmem_ld_wait();
#pragma unroll
                for (int hh = 0; hh < HG; ++hh) {
                    const float aej = j == 0 ? ach[hh][0] : (j == 1 ? ach[hh][1] : (j == 2 ? ach[hh][2] : ach[hh][3]));
                    const float abj = j == 0 ? 0.f : (j == 1 ? ach[hh][0] : (j == 2 ? ach[hh][1] : ach[hh][2]));
                    uint32_t mr[16];
                    if (q < j) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) mr[e] = 0u;
                    } else if (q == j && abj - aej > kMaxBlockDecay) {
                        const float *ah = at_s + hh * kTile + 32 * j;
                        const int tb = t0 + 32 * j;
                        auto lw = [&](int s) {
                            const int tok = tb + s;
                            const float d =
                                tok < w_len()
                                    ? a.dt[(w_grow0() + tok) * a.H + h0 + hh]
                                    : 0.f;
                            return __expf(at[hh] - ah[s]) * d;
                        };
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int s0 = 2 * e;
                            const float m0 = s0 <= lane ? __uint_as_float(gr[2 * e]) * lw(s0) : 0.f;
                            const float m1 = s0 + 1 <= lane ? __uint_as_float(gr[2 * e + 1]) * lw(s0 + 1) : 0.f;
                            mr[e] = pack_bf16x2(m0, m1);
                        }
                    } else {
                        const float R = __expf(at[hh] - aej);
                        const uint64_t rr = pack_f32x2(R, R);
                        const float4 *vh = reinterpret_cast<const float4 *>(v_s + hh * kTile + 32 * j);
#pragma unroll
                        for (int e4 = 0; e4 < 8; ++e4) {
                            const float4 v = vh[e4];
                            const uint64_t g01 = pack_f32x2(__uint_as_float(gr[4 * e4]), __uint_as_float(gr[4 * e4 + 1]));
                            const uint64_t g23 = pack_f32x2(__uint_as_float(gr[4 * e4 + 2]), __uint_as_float(gr[4 * e4 + 3]));
                            const uint64_t m01 = mul_f32x2(mul_f32x2(g01, pack_f32x2(v.x, v.y)), rr);
                            const uint64_t m23 = mul_f32x2(mul_f32x2(g23, pack_f32x2(v.z, v.w)), rr);
                            mr[2 * e4] = pack_bf16x2_from_f32x2(m01);
                            mr[2 * e4 + 1] = pack_bf16x2_from_f32x2(m23);
                        }
                        if (q == j) {
                            // causal cut inside the diagonal block: keep s <= t (= lane)
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const int s0 = 2 * e;
                                const uint32_t keep = s0 + 1 <= lane ? 0xffffffffu : (s0 <= lane ? 0x0000ffffu : 0u);
                                mr[e] &= keep;
                            }
                        }
                    }
                    tmem_st16(tq + kColG + 32 * j + 16 * hh, mr);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(7));

            // exp(a_t) of this tile for its epilogue, before the next tile's factors
            float e_at_t[HG];
#pragma unroll
            for (int h = 0; h < HG; ++h) e_at_t[h] = __expf(at[h]);
            // (head, 32-column range) of this warpgroup: HG = 2 -> head wg & 1,
            // columns 32 (wg >> 1) ..; HG = 1 -> head 0, columns 16 wg ..
            const int hh = HG == 2 ? (wg & 1) : 0;
            const int p0 = HG == 2 ? 32 * (wg >> 1) : 16 * wg;
            constexpr int np = HG == 2 ? 32 : 16;
            // the output gate's z for this thread's token and columns, loaded
            // (from L2, where the producer prefetched it) before the next
            // tile's state prep, which hides their latency (loaded just before
            // the wait for the products, the gated long layer took 913 us
            // against 727); rows past the sequence's end read nothing
            uint4 zv[np / 8];
            bool gated = false;
            if constexpr (kGate) {
                if (a.fuse.z && t0 + row < w_len()) {
                    gated = true;
                    const __nv_bfloat16 *zrow = static_cast<const __nv_bfloat16 *>(a.fuse.z) +
                                                ((w_grow0() + t0 + row) * a.H + h0 + hh) * kP + p0;
#pragma unroll
                    for (int q = 0; q < np / 8; ++q) zv[q] = *reinterpret_cast<const uint4 *>(zrow + 8 * q);
                }
            }
            if (it + 1 < ntile) {
                load_factors(it + 1);
                prep_tile(it + 1);
            }

            // ---- epilogue: y = Yd + exp(a_t) Yo + D x, staged as bf16 in this
            //      stage's C blocks (free once the tile's off-diagonal product is
            //      done; head h in block h) for issuer B's TMA stores
            wait_bar_warp(bar(10), it & 1, abort_flag, a.err, a.wait_ns);
            tc_fence_after();
            {
                // selects, not dynamic indexing (which would move the arrays to local memory)
                const float e_at = (HG == 2 && hh == 1) ? e_at_t[HG - 1] : e_at_t[0];
                const float dsk = (HG == 2 && hh == 1) ? Dh[HG - 1] : Dh[0];
                const uint64_t ea2 = pack_f32x2(e_at, e_at), dsk2 = pack_f32x2(dsk, dsk);
                const uint8_t *xs = tiles_ptr + stage * kStage + kCBytes + hh * kXBytes;
                uint8_t *ybuf = tiles_ptr + stage * kStage + hh * kBlk;
                const bool direct = partial(it);
#pragma unroll
                for (int c16 = 0; c16 < np; c16 += 16) {
                    const int pc = p0 + c16;
                    uint32_t yd[16], yo[16];
                    tmem_ld16(tq + kColYd + 64 * hh + pc, yd);
                    tmem_ld16(tq + kColYo + 64 * hh + pc, yo);
                    tmem_ld_wait();
                    uint32_t pk[8];
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        // D x for these 8 columns from the X tile in the stage
                        const uint4 xv = *reinterpret_cast<const uint4 *>(xs + sw128(row, pc + 8 * half));
                        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i = 8 * half + 2 * e;
                            const uint64_t x01 = pack_f32x2(__uint_as_float(xw[e] << 16),
                                                            __uint_as_float(xw[e] & 0xffff0000u));
                            const uint64_t y01 = fma_f32x2(
                                ea2, pack_f32x2(__uint_as_float(yo[i]), __uint_as_float(yo[i + 1])),
                                pack_f32x2(__uint_as_float(yd[i]), __uint_as_float(yd[i + 1])));
                            uint64_t v01 = fma_f32x2(dsk2, x01, y01);
                            if constexpr (kGate) {
                                if (gated) {
                                    // silu(z) = h + h tanh(h), h = z / 2 (sigmoid(z) =
                                    // (1 + tanh(z/2)) / 2): one hardware tanh per
                                    // element; its 2^-11 error is below the bf16 output's
                                    const uint4 zq = zv[c16 / 8 + half];
                                    const uint32_t zw = e == 0 ? zq.x : e == 1 ? zq.y : e == 2 ? zq.z : zq.w;
                                    const uint64_t h01 = mul_f32x2(
                                        pack_f32x2(__uint_as_float(zw << 16), __uint_as_float(zw & 0xffff0000u)),
                                        pack_f32x2(0.5f, 0.5f));
                                    const uint64_t t01 = pack_f32x2(tanh_approx(__uint_as_float((uint32_t)h01)),
                                                                    tanh_approx(__uint_as_float((uint32_t)(h01 >> 32))));
                                    v01 = mul_f32x2(v01, fma_f32x2(h01, t01, h01));
                                }
                            }
                            pk[4 * half + e] = pack_bf16x2_from_f32x2(v01);
                        }
                    }
                    if (!direct) {
                        *reinterpret_cast<uint4 *>(ybuf + sw128(row, pc)) =
                            make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        *reinterpret_cast<uint4 *>(ybuf + sw128(row, pc + 8)) =
                            make_uint4(pk[4], pk[5], pk[6], pk[7]);
                    } else if (t0 + row < w_len()) {
                        __nv_bfloat16 *yr = a.y + ((w_grow0() + t0 + row) * a.H + h0 + hh) * kP + pc;
                        *reinterpret_cast<uint4 *>(yr) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        *reinterpret_cast<uint4 *>(yr + 8) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar(11));          // y staged, Yd / Yo read
                mbar_arrive(bar(16 + stage));  // this tile's X read
            }
        }
        // ---- final state of the sequence (all MMAs completed: y_full of the last tile)
        if (sigma == w_nseg() - 1 && a.fin && ntile > 0 && !*abort_flag) {
            tc_fence_after();
#pragma unroll 1
            for (int h = 0; h < HG; ++h) {
                uint32_t r[16];
                tmem_ld16(tq + kColH + 64 * h + 16 * wg, r);
                tmem_ld_wait();
                float *dst = a.fin + ((size_t)w_seq() * a.H + h0 + h) * kP * kN;
#pragma unroll
                for (int j = 0; j < 16; ++j) dst[(size_t)(16 * wg + j) * kN + row] = __uint_as_float(r[j]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        // A wait ran out: before TMEM is freed and the CTA exits, every product
        // either issuer issued is complete (each commits once more, on barrier
        // 18 or 19, and waits) and every load the producer issued has landed
        // (its consumers may never have waited for it).  Loads go out tile by
        // tile, so the last two tiles of X and C (one per stage) and the last
        // of B hold the only phases that can still be pending.
        if (lane == 0 && (warp == kIssuerA || warp == kIssuerB)) {
            const int b2 = warp == kIssuerA ? 18 : 19;
            mma_commit(bar(b2));
            drain_bar(bar(b2), 0, abort_flag, a.err, a.wait_ns);
        }
        if (threadIdx.x == 0) {
            const int *last = reinterpret_cast<const int *>(smem + kOffLast);
            const int lastX = last[0], lastB = last[1], lastC = last[2];
            for (int k = lastX; k >= 0 && k >= lastX - 1; --k)
                drain_bar(bar(14 + (k & 1)), (k >> 1) & 1, abort_flag, a.err, a.wait_ns);
            for (int k = lastC; k >= 0 && k >= lastC - 1; --k)
                drain_bar(bar(k & 1), (k >> 1) & 1, abort_flag, a.err, a.wait_ns);
            if (lastB >= 0) drain_bar(bar(4), lastB & 1, abort_flag, a.err, a.wait_ns);
        }
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ============================================= segment contribution kernel
// F_sigma = sum over the segment's tokens of exp(a_end(segment) - a_s) dt_s
//           x_s B_s^T, with tiles visited last to first so the decay from a
// tile's end to the segment's end is a running sum of tile totals.  HG heads
// of one group (1, 2 or 4) share each B tile.
//
// Warp roles: warp 0 issues TMA loads (B and X of a tile per stage), warp 1
// issues F += B^T . (w o X) for all heads of the CTA at once, warps 2-9 scale
// each X tile in place by its token weights, and warp 10 computes the weights
// w_s = exp(decay from s to the segment end) dt_s of each tile into a ring
// with one slot per stage.
template <int HG, bool kPacked>
__global__ void __launch_bounds__(kSegThreads, 1)
ssd_tc_segment_kernel(const __grid_constant__ CUtensorMap mapB,
                      const __grid_constant__ CUtensorMap mapX, const TcArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int kStages = seg_stages(HG);
    constexpr uint32_t kStage = kBBytes + HG * kXBytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h0 = blockIdx.x * HG;
    const SegWork w = seg_work<kPacked>(a, blockIdx.y, blockIdx.z, true);
    // batched: from the grid and the kernel parameters at each use (nothing
    // held in registers across the kernel); packed: from the prefix tables
    auto w_seq = [&]() -> int { return kPacked ? w.seq : (int)blockIdx.z; };
    auto w_grow0 = [&]() -> size_t { return kPacked ? w.grow0 : (size_t)blockIdx.z * a.L; };
    auto w_len = [&]() -> int { return kPacked ? w.len : a.L; };
    auto w_tiles = [&]() -> int { return kPacked ? w.tiles : a.tiles; };
    auto w_nseg = [&]() -> int { return kPacked ? w.nseg : a.nseg; };
    auto w_sigma = [&]() -> int { return kPacked ? w.sigma : (int)blockIdx.y + a.sigma0; };
    auto w_fslot = [&]() -> int { return kPacked ? w.fslot : (int)blockIdx.z * (a.nseg - 1); };
    const int sigma = w_sigma();                    // < the sequence's last segment
    const int g = h0 / (a.H / a.G);
    const int k0 = sigma * a.seg_tiles;
    const int k1 = min(w_tiles(), k0 + a.seg_tiles);
    const int ntile = k1 - k0;
    const int trow = kPacked ? (int)w_grow0() : 0;    // TMA row / batch of token 0
    const int tb = kPacked ? 0 : w_seq();

    const uint32_t sbase = smem_u32(smem);
    if ((sbase & 1023u) != 0u) {
        if (threadIdx.x == 0) ssd_report(a.err, SSD_DEVERR_SMEM_ALIGN);
        return;
    }
    // barriers: 0..2 full[stage] (B, X landed); 3..5 empty[stage] (MMA done);
    //           6..8 xt_ready[stage] (X scaled); 9..11 w_ready[stage]; 12 done
    auto bar = [&](int i) { return sbase + 8u * (uint32_t)i; };
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + kOffTslot);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffAbort);
    const uint32_t tiles_base = sbase + kCtrl;
    uint8_t *tiles_ptr = smem + kCtrl;
    float *w_ring = reinterpret_cast<float *>(tiles_ptr + kStages * kStage);   // [stage][HG][128]
    constexpr uint32_t kCols = 64 * HG;        // F of every head (lane n, column p)
    griddep_launch_dependents();

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(bar(i), 1);
            mbar_init(bar(3 + i), 1);
            mbar_init(bar(6 + i), kSegXWarps);
            mbar_init(bar(9 + i), 1);
        }
        mbar_init(bar(12), 1);
        *reinterpret_cast<int *>(smem + kOffLast) = 0;
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tslot), kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&mapB);
            tma_prefetch_desc(&mapX);
            int issued = 0;
            for (int it = 0; it < ntile; ++it) {
                const int stage = it % kStages;
                if (it >= kStages &&
                    !wait_bar(bar(3 + stage), ((it / kStages) - 1) & 1, abort_flag, a.err, a.wait_ns))
                    break;
                issued = it + 1;
                const uint32_t stg = tiles_base + stage * kStage;
                const int t0 = (k1 - 1 - it) * kTile;
                mbar_arrive_expect_tx(bar(stage), kStage);
                tma_load_4d(stg, &mapB, bar(stage), 0, g, trow + t0, tb);
                tma_load_4d(stg + kBlk, &mapB, bar(stage), 64, g, trow + t0, tb);
#pragma unroll
                for (int h = 0; h < HG; ++h)
                    tma_load_4d(stg + kBBytes + h * kXBytes, &mapX, bar(stage), 0, h0 + h,
                                trow + t0, tb);
            }
            *reinterpret_cast<int *>(smem + kOffLast) = issued;   // for the drain at exit
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdSAll = idesc_bf16_f32(128, 64 * HG, true, true);
            const uint64_t bD = smem_desc(tiles_base, kBlk, 1024, kSwizzle128B);
            const uint64_t xD = smem_desc(tiles_base + kBBytes, kXBytes, 1024, kSwizzle128B);
            for (int it = 0; it < ntile; ++it) {
                const int stage = it % kStages;
                const uint64_t so = (uint64_t)((stage * kStage) >> 4);
                if (!wait_bar(bar(6 + stage), (it / kStages) & 1, abort_flag, a.err, a.wait_ns)) break;
                tc_fence_after();
                // all heads at once: F += B^T . [w o X_0 | w o X_1]  (N = 64 * HG)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss(tmem, bD + so + (uint64_t)(kk * 128), xD + so + (uint64_t)(kk * 128),
                           kIdSAll, (it > 0 || kk > 0) ? 1u : 0u);
                mma_commit(bar(3 + stage));
            }
            mma_commit(bar(12));
        }
    } else if (warp == kSegFacWarp) {
        // ------------------------------------------------- token weights
        // Lane l owns tokens 4l .. 4l+3 of a tile: w_s = exp(suffix of dt A from
        // s to the segment end) dt_s; suf carries the totals of the tiles done.
        // dt is loaded three tiles ahead (a tile takes about a microsecond here,
        // less than a loaded memory system's latency).
        float Af[HG], suf[HG], d0[HG][4], d1[HG][4], d2[HG][4];
#pragma unroll
        for (int h = 0; h < HG; ++h) {
            Af[h] = a.A[h0 + h];
            suf[h] = 0.f;
        }
        auto load_dt4 = [&](int it, float (&dn)[HG][4]) {
            const int tok0 = (k1 - 1 - it) * kTile + 4 * lane;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int tok = tok0 + i;
#pragma unroll
                for (int h = 0; h < HG; ++h)
                    dn[h][i] = (it < ntile && tok < w_len()) ? a.dt[(w_grow0() + tok) * a.H + h0 + h]
                                                           : 0.f;
            }
        };
        load_dt4(0, d0);
        load_dt4(1, d1);
        load_dt4(2, d2);
        for (int it = 0; it < ntile; ++it) {
            const int stage = it % kStages;
            float d[HG][4];
#pragma unroll
            for (int h = 0; h < HG; ++h)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    // the transform at use keeps the three tiles of loads in flight
                    const int tok = (k1 - 1 - it) * kTile + 4 * lane + i;
                    d[h][i] = tok < w_len() ? d0[h][i] : 0.f;
                    d0[h][i] = d1[h][i];
                    d1[h][i] = d2[h][i];
                }
            load_dt4(it + 3, d2);
            float wv[HG][4];
#pragma unroll
            for (int h = 0; h < HG; ++h) {
                float c[4];
                c[0] = d[h][0] * Af[h];
#pragma unroll
                for (int i = 1; i < 4; ++i) c[i] = c[i - 1] + d[h][i] * Af[h];
                float incl = c[3];
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float o = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl += o;
                }
                float excl = __shfl_up_sync(0xffffffffu, incl, 1);
                if (lane == 0) excl = 0.f;
                const float tot = __shfl_sync(0xffffffffu, incl, 31);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    wv[h][i] = __expf(suf[h] + tot - (excl + c[i])) * d[h][i];
                suf[h] += tot;
            }
            // the slot was last read by the scaling of tile it - kStages
            if (it >= kStages &&
                !wait_bar_warp(bar(6 + stage), ((it / kStages) - 1) & 1, abort_flag, a.err, a.wait_ns))
                break;
            float *slot = w_ring + stage * HG * kTile;
#pragma unroll
            for (int h = 0; h < HG; ++h)
                *reinterpret_cast<float4 *>(slot + h * kTile + 4 * lane) =
                    make_float4(wv[h][0], wv[h][1], wv[h][2], wv[h][3]);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(9 + stage));
        }
        if (lane == 0 && !*abort_flag) {
#pragma unroll
            for (int h = 0; h < HG; ++h)
                a.ws_decay[(size_t)(w_fslot() + sigma) * a.H + h0 + h] = __expf(suf[h]);
        }
    } else {
        // ------------------------------------------- X scaling, then F out
        const int tw = warp - 2;
        const int wg = tw >> 2;               // warpgroup 0..1: X columns 32 wg ..
        const int q = warp & 3;
        const int row = 32 * q + lane;
        const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
        for (int it = 0; it < ntile; ++it) {
            const int stage = it % kStages;
            uint8_t *stg_ptr = tiles_ptr + stage * kStage;
            if (!wait_bar_warp(bar(9 + stage), (it / kStages) & 1, abort_flag, a.err, a.wait_ns))
                break;                                                                  // weights
            if (!wait_bar_warp(bar(stage), (it / kStages) & 1, abort_flag, a.err, a.wait_ns))
                break;                                                                  // X landed
            const float *slot = w_ring + stage * HG * kTile;
#pragma unroll
            for (int h = 0; h < HG; ++h) {
                const float w = slot[h * kTile + row];
                uint8_t *xs = stg_ptr + kBBytes + h * kXBytes;
#pragma unroll
                for (int c = 4 * wg; c < 4 * wg + 4; ++c) {
                    const uint32_t off = sw128(row, 8 * c);
                    *reinterpret_cast<uint4 *>(xs + off) =
                        scale_bf16x8_bf(*reinterpret_cast<const uint4 *>(xs + off), w);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(6 + stage));
        }
        if (ntile > 0) wait_bar_warp(bar(12), 0, abort_flag, a.err, a.wait_ns);
        tc_fence_after();
        if (!*abort_flag) {
#pragma unroll 1
            for (int h = 0; h < HG; ++h) {
                uint32_t r[32];
                tmem_ld32(tq + 64 * h + 32 * wg, r);
                tmem_ld_wait();
                __nv_bfloat16 *dst = a.ws_state +
                                     ((size_t)(w_fslot() + sigma) * a.H + h0 + h) * kP * kN;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    dst[(size_t)(32 * wg + j) * kN + row] = __float2bfloat16_rn(__uint_as_float(r[j]));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        // A wait ran out: every issued load has landed (the last load of each
        // stage, tile issued - 1 - i, completes that stage's phases) and every
        // product is complete (the issuer's last commit, on barrier 12) before
        // TMEM is freed and the CTA exits.
        if (threadIdx.x == 0) {
            const int issued = *reinterpret_cast<const int *>(smem + kOffLast);
            for (int i = 0; i < kStages && i < issued; ++i) {
                const int it = issued - 1 - i;
                drain_bar(bar(it % kStages), (it / kStages) & 1, abort_flag, a.err, a.wait_ns);
            }
            drain_bar(bar(12), 0, abort_flag, a.err, a.wait_ns);
        }
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kCols);
    }
    // a second segment launch (the last segments, fewer heads per CTA) ends
    // only after the first: the chaining kernel waits for it alone (a no-op
    // for a launch with no programmatic predecessor)
    griddep_wait();
}

// ============================================ entering state of each segment
// Step-3 at segment granularity: H_in[s+1] = decay_s * H_in[s] + F_s, with
// H_in[0] = the sequence's initial state.  Overwrites slot s (F_s) with
// H_in[s+1].  A sequence's slots are nseg-1 consecutive ones from base
// (batched: sequence q has base q (nseg-1); packed: fslot0[q] .. fslot0[q+1]).
// The loads of up to kBatch segments are issued before their dependent FMA
// chain.  Timed: 20 a batch (one round trip for the long layer's 18
// contributions, 112 registers) takes 2 us off that call; 8 a batch (fewer
// registers) is 3 % faster for the 10 contributions of a 4096-token layer.
template <int kBatch>
__global__ void __launch_bounds__(256)
ssd_tc_segment_pass_kernel(__nv_bfloat16 *__restrict__ ws_state, const float *__restrict__ ws_decay,
                           const float *__restrict__ init, int nseqs, int H, int nseg,
                           const int *__restrict__ fslot0) {
    // let the scan kernel start right away: its first-segment CTAs need nothing
    // from here, the others wait for this grid before reading entering states
    griddep_launch_dependents();
    griddep_wait();                 // segment contributions are complete and visible
    const size_t per_head = (size_t)kP * kN / 4;
    const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const size_t total = (size_t)nseqs * H * per_head;
    if (idx >= total) return;
    const int q = (int)(idx / ((size_t)H * per_head));
    const size_t rem = idx - (size_t)q * H * per_head;
    const int h = (int)(rem / per_head);
    const size_t e = rem - (size_t)h * per_head;
    const int base = fslot0 ? fslot0[q] : q * (nseg - 1);
    const int count = fslot0 ? fslot0[q + 1] - base : nseg - 1;
    float4 hv = make_float4(0.f, 0.f, 0.f, 0.f);
    if (init) hv = reinterpret_cast<const float4 *>(init)[((size_t)q * H + h) * per_head + e];
    // four bf16 state elements per thread: contributions in, entering states out
    uint2 *st = reinterpret_cast<uint2 *>(ws_state);
    auto lo = [](uint32_t w) { return __uint_as_float(w << 16); };
    auto hi = [](uint32_t w) { return __uint_as_float(w & 0xffff0000u); };
    for (int s0 = 0; s0 < count; s0 += kBatch) {
        uint2 f[kBatch];
        float d[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            if (s0 + i < count) {
                const size_t slot = (size_t)(base + s0 + i) * H + h;
                f[i] = st[slot * per_head + e];
                d[i] = ws_decay[slot];
            }
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            if (s0 + i < count) {
                const size_t slot = (size_t)(base + s0 + i) * H + h;
                hv.x = fmaf(d[i], hv.x, lo(f[i].x));
                hv.y = fmaf(d[i], hv.y, hi(f[i].x));
                hv.z = fmaf(d[i], hv.z, lo(f[i].y));
                hv.w = fmaf(d[i], hv.w, hi(f[i].y));
                st[slot * per_head + e] = make_uint2(pack_bf16x2(hv.x, hv.y), pack_bf16x2(hv.z, hv.w));
            }
        }
    }
}

// ------------------------------------------------------------------ host
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

// 4-D bf16 map over [batch][L][d1][inner] with a box of 64 x 1 x 128 x 1,
// 128-byte swizzle; out-of-range tokens read as zero.
bool make_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t d1, uint64_t L,
              uint64_t batch) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[4] = {inner, d1, L, batch};
    cuuint64_t strides[3] = {inner * 2, inner * d1 * 2, inner * d1 * L * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)kTile, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int HG>
constexpr size_t scan_smem() {
    return kCtrl + (size_t)ScanLayout<HG>::kBytes;
}
template <int HG>
constexpr size_t seg_smem() {
    return kCtrl + seg_stages(HG) * ((size_t)(kBBytes + HG * kXBytes) + HG * kTile * sizeof(float));
}
static_assert(scan_smem<2>() <= 232448, "scan kernel shared memory exceeds 227 KB");
static_assert(seg_smem<2>() <= 232448, "segment kernel shared memory exceeds 227 KB");
static_assert(seg_smem<4>() <= 232448, "segment kernel shared memory exceeds 227 KB");

// Launch with programmatic stream serialization: the kernel may begin while
// the previous kernel in the stream finishes; it calls griddepcontrol.wait
// before touching that kernel's results.
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

// Segment contributions with SG heads per CTA: all of them, or (batched, with
// nsig > 0) segments args.sigma0 .. args.sigma0 + nsig - 1, launched after the
// previous kernel with programmatic stream serialization when `pdl`.
template <int SG, bool kPacked>
cudaError_t launch_segment(const SsdTcPlan &plan, const CUtensorMap &mB, const CUtensorMap &mX,
                           const TcArgs &args, int batch, int H, cudaStream_t stream,
                           int nsig = 0, bool pdl = false) {
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(ssd_tc_segment_kernel<SG, kPacked>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)seg_smem<SG>());
    });
    if (attr_err != cudaSuccess) return attr_err;
    dim3 g1(H / SG, plan.varlen ? plan.nslots : (nsig > 0 ? nsig : plan.nseg - 1),
            plan.varlen ? 1 : batch);
    if (pdl)
        return launch_pdl(ssd_tc_segment_kernel<SG, kPacked>, g1, dim3(kSegThreads),
                          seg_smem<SG>(), stream, mB, mX, args);
    ssd_tc_segment_kernel<SG, kPacked><<<g1, kSegThreads, seg_smem<SG>(), stream>>>(mB, mX, args);
    return cudaGetLastError();
}

template <int HG, bool kGate, bool kPacked>
cudaError_t launch_hg(const SsdTcPlan &plan, const CUtensorMap &mC, const CUtensorMap &mB,
                      const CUtensorMap &mX, const CUtensorMap &mY, const CUtensorMap &mZ,
                      const TcArgs &args, int batch, int H, SsdProfileEvents prof,
                      cudaStream_t stream) {
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(ssd_tc_scan_kernel<HG, false, kGate, kPacked>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)scan_smem<HG>());
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(ssd_tc_scan_kernel<HG, true, kGate, kPacked>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            (int)scan_smem<HG>());
    });
    if (attr_err != cudaSuccess) return attr_err;
    // factor warp on the light sub-partition for long segments, the producer
    // there for short ones (A/B timed on the 130M and 2.7B layers)
    auto kernel = plan.seg_tiles >= kLongSegTiles ? ssd_tc_scan_kernel<HG, true, kGate, kPacked>
                                                  : ssd_tc_scan_kernel<HG, false, kGate, kPacked>;
    if (plan.varlen) {
        ssd_varlen_plan_kernel<<<1, 1024, 0, stream>>>(
            args.cu, args.nseq, plan.seg_tiles, const_cast<int *>(args.item0),
            const_cast<int *>(args.fslot0), args.init, args.fin, H * kP * kN);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const bool chained = plan.nslots > 0;
    if (chained) {
        cudaError_t e;
        if (!plan.varlen && plan.seg_heads == 4 && plan.seg_split > 0) {
            // whole waves of four-head CTAs, then the remaining segments as
            // two-head CTAs, which fill the last wave with shorter work
            e = launch_segment<4, kPacked>(plan, mB, mX, args, batch, H, stream, plan.seg_split);
            if (e == cudaSuccess) {
                TcArgs rest = args;
                rest.sigma0 = plan.seg_split;
                e = launch_segment<2, kPacked>(plan, mB, mX, rest, batch, H, stream,
                                               plan.nseg - 1 - plan.seg_split, true);
            }
        } else {
            e = plan.seg_heads == 4
                    ? launch_segment<4, kPacked>(plan, mB, mX, args, batch, H, stream)
                    : launch_segment<HG, kPacked>(plan, mB, mX, args, batch, H, stream);
        }
        if (e != cudaSuccess) return e;
        const size_t total = (size_t)plan.nseqs * H * kP * kN / 4;
        auto pass = !plan.varlen && plan.nseg - 1 > 12 ? ssd_tc_segment_pass_kernel<20>
                                                       : ssd_tc_segment_pass_kernel<8>;
        e = launch_pdl(pass, dim3((unsigned)((total + 255) / 256)),
                       dim3(256), 0, stream, args.ws_state, args.ws_decay, args.init,
                       plan.nseqs, H, plan.nseg, plan.varlen ? args.fslot0 : nullptr);
        if (e != cudaSuccess) return e;
    }
    dim3 g2(H / HG, plan.varlen ? plan.items : plan.nseg, plan.varlen ? 1 : batch);
    if (prof.before && prof.after) {
        cudaError_t e = ssd_record_event(prof.before, stream);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e;
    if (chained) {
        // overlaps the scan kernel's prologue and first tile with the chaining kernel
        e = launch_pdl(kernel, g2, dim3(kThreads), scan_smem<HG>(), stream, mC, mB, mX, mY, mZ,
                       args);
    } else {
        kernel<<<g2, kThreads, scan_smem<HG>(), stream>>>(mC, mB, mX, mY, mZ, args);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess && prof.before && prof.after) e = ssd_record_event(prof.after, stream);
    return e;
}

}  // namespace

SsdTcPlan ssd_tc_plan(int batch, int L, int H, int P, int N, int G, int num_sms) {
    SsdTcPlan p{};
    p.launches = 1;
    p.supported = P == kP && N == kN && num_sms > 0 && batch > 0 && L > 0 && H > 0 && G > 0 &&
                  H % G == 0 && encoder() != nullptr;
    if (!p.supported) return p;
    p.heads_per_cta = ((H / G) % 2 == 0) ? 2 : 1;
    p.tiles = (L + kTile - 1) / kTile;
    const long units = (long)batch * (H / p.heads_per_cta);
    // Segments trade sequence parallelism against the extra pass over x that
    // the segment contributions cost: estimate per-SM time as waves x tiles
    // per segment, with that extra pass weighted 0.4 of a scan tile.
    double best = 1e300;
    int best_n = 1;
    const int max_n = p.tiles < 64 ? p.tiles : 64;
    for (int n = 1; n <= max_n; ++n) {
        const int seg = (p.tiles + n - 1) / n;
        const int nseg = (p.tiles + seg - 1) / seg;
        if (nseg != n) continue;
        const long ctas = units * nseg;
        const long waves = (ctas + num_sms - 1) / num_sms;
        const double cost = (double)waves * seg * (nseg > 1 ? 1.4 : 1.0);
        if (cost < best * 0.999) {
            best = cost;
            best_n = nseg;
        }
    }
    p.seg_tiles = (p.tiles + best_n - 1) / best_n;
    p.nseg = (p.tiles + p.seg_tiles - 1) / p.seg_tiles;
    // Four heads of a group share each B tile in the segment kernel, if that
    // grid still covers every SM.
    p.seg_heads = p.heads_per_cta;
    if ((H / G) % 4 == 0 && (long)batch * (H / 4) * (p.nseg - 1) >= num_sms) p.seg_heads = 4;
    // four-head segment CTAs for as many segments as fill whole waves, the
    // rest as two-head CTAs (a second launch) when that leaves a partial wave
    p.seg_split = 0;
    if (p.seg_heads == 4 && p.nseg > 2) {
        const long per = (long)batch * (H / 4);          // CTAs per segment
        const long total = per * (p.nseg - 1);
        const int split = (int)((total / num_sms) * num_sms / per);
        if (total % num_sms != 0 && split > 0 && split < p.nseg - 1) p.seg_split = split;
    }
    p.varlen = false;
    p.nseqs = batch;
    p.nslots = batch * (p.nseg - 1);
    p.items = batch * p.nseg;
    if (p.nseg > 1) {
        const size_t state = (size_t)batch * (p.nseg - 1) * H * kP * kN * sizeof(__nv_bfloat16);
        const size_t decay = (size_t)batch * (p.nseg - 1) * H * sizeof(float);
        p.workspace = ((state + 255) / 256) * 256 + ((decay + 255) / 256) * 256;
        p.launches = p.seg_split > 0 ? 4 : 3;
    }
    // room for the transformed step sizes (used only with a dt transform)
    p.dt_offset = p.workspace;
    p.workspace += (((size_t)batch * L * H * sizeof(float) + 255) / 256) * 256;
    return p;
}

SsdTcPlan ssd_tc_plan_varlen(int nseq, const int *cu, int H, int P, int N, int G, int num_sms) {
    SsdTcPlan p{};
    p.launches = 1;
    p.supported = P == kP && N == kN && num_sms > 0 && nseq > 0 && cu != nullptr && H > 0 &&
                  G > 0 && H % G == 0 && encoder() != nullptr;
    if (!p.supported) return p;
    int max_tiles = 0;
    for (int s = 0; s < nseq; ++s) {
        const int len = cu[s + 1] - cu[s];
        if (len < 0) {
            p.supported = false;
            return p;
        }
        max_tiles = max_tiles > (len + kTile - 1) / kTile ? max_tiles : (len + kTile - 1) / kTile;
    }
    if (max_tiles == 0) {   // no token at all: the SIMT path gives final = initial
        p.supported = false;
        return p;
    }
    p.varlen = true;
    p.nseqs = nseq;
    p.heads_per_cta = ((H / G) % 2 == 0) ? 2 : 1;
    p.tiles = max_tiles;
    const long units = H / p.heads_per_cta;
    // Cost of a segment length, in scan-tile times per SM: every CTA-tile
    // spread over the SMs, plus 0.4 of a tile for each tile the segment
    // kernel passes over again (all but each sequence's last segment), plus
    // 2.5 tiles per contribution slot (its state written, chained and read
    // back: 4 x 32 KB per head), plus half the longest item as the tail.
    // Timed on a 47-sequence, 65536-token packed batch of the 80-head layer,
    // where this picks no split (0.57 ms; 1-tile segments took 2.2 ms).
    auto segments = [&](int seg, long *items, long *slots, long *again) {
        *items = *slots = *again = 0;
        for (int s = 0; s < nseq; ++s) {
            const int tiles = (cu[s + 1] - cu[s] + kTile - 1) / kTile;
            const int n = (tiles + seg - 1) / seg;
            *items += n;
            *slots += n > 0 ? n - 1 : 0;   // an empty sequence has no segment
            *again += n > 0 ? (long)(n - 1) * seg : 0;
        }
    };
    long total_tiles = 0;
    for (int s = 0; s < nseq; ++s) total_tiles += (cu[s + 1] - cu[s] + kTile - 1) / kTile;
    static const int kCand[] = {1, 2, 3, 4, 6, 8, 12, 16, 24, 32, 48, 64, 96, 128, 192, 256};
    double best = 1e300;
    int best_seg = max_tiles;
    for (int i = -1; i < (int)(sizeof(kCand) / sizeof(kCand[0])); ++i) {
        const int seg = i < 0 ? max_tiles : kCand[i];
        if (seg > max_tiles) continue;
        long items, slots, again;
        segments(seg, &items, &slots, &again);
        const double cost = (double)units * (total_tiles + 0.4 * again + 2.5 * slots) / num_sms +
                            0.5 * seg;
        if (cost < best * 0.999) {
            best = cost;
            best_seg = seg;
        }
    }
    p.seg_tiles = best_seg;
    long items, slots, again;
    segments(best_seg, &items, &slots, &again);
    if (items > 65535) {   // grid y holds the work items
        p.supported = false;
        return p;
    }
    p.items = (int)items;
    p.nslots = (int)slots;
    p.nseg = 0;                    // per sequence
    p.seg_heads = p.heads_per_cta;
    if ((H / G) % 4 == 0 && (long)(H / 4) * slots >= num_sms) p.seg_heads = 4;
    const size_t state = (size_t)slots * H * kP * kN * sizeof(__nv_bfloat16);
    const size_t decay = (size_t)slots * H * sizeof(float);
    const size_t table = 2 * (size_t)(nseq + 1) * sizeof(int);
    p.workspace = ((state + 255) / 256) * 256 + ((decay + 255) / 256) * 256 +
                  ((table + 255) / 256) * 256;
    p.launches = slots > 0 ? 4 : 2;
    p.dt_offset = p.workspace;
    p.workspace += (((size_t)cu[nseq] * H * sizeof(float) + 255) / 256) * 256;
    return p;
}

cudaError_t ssd_launch_scan_tc(const SsdTcPlan &plan, const void *x, const float *dt,
                               const float *A, const void *B, const void *C, const float *D,
                               const float *init, void *y, float *fin, int batch, int L, int H,
                               int P, int N, int G, void *workspace, unsigned int *err,
                               const SsdFuse &fuse, SsdProfileEvents prof, cudaStream_t stream,
                               const int *cu_dev) {
    (void)P;
    (void)N;
    // packed sequences: one batch row of L = total tokens
    const int mrows = L, mbatch = plan.varlen ? 1 : batch;
    CUtensorMap mC, mB, mX, mY, mZ;
    if (!make_map(&mC, C, kN, G, mrows, mbatch) || !make_map(&mB, B, kN, G, mrows, mbatch) ||
        !make_map(&mX, x, kP, H, mrows, mbatch) || !make_map(&mY, y, kP, H, mrows, mbatch) ||
        !make_map(&mZ, fuse.z ? fuse.z : x, kP, H, mrows, mbatch))
        return cudaErrorInvalidValue;
    TcArgs args{};
    args.dt = dt;
    if (ssd_dt_transform_active(fuse)) {
        float *dt_eff = reinterpret_cast<float *>(static_cast<char *>(workspace) + plan.dt_offset);
        const size_t n = (size_t)(plan.varlen ? 1 : batch) * L * H;
        if (n > 0) {
            const size_t want = (n + 255) / 256;
            const unsigned grid = (unsigned)(want < 16u * 152u ? want : 16u * 152u);
            ssd_dt_prepass_kernel<<<grid, 256, 0, stream>>>(dt, dt_eff, n, H, fuse);
            const cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return e;
        }
        args.dt = dt_eff;
    }
    args.fuse = fuse;
    args.A = A;
    args.D = D;
    args.init = init;
    if (plan.nslots > 0 || plan.varlen) {
        const size_t state = (size_t)plan.nslots * H * kP * kN * sizeof(__nv_bfloat16);
        const size_t decay = (size_t)plan.nslots * H * sizeof(float);
        char *ws = static_cast<char *>(workspace);
        args.ws_state = reinterpret_cast<__nv_bfloat16 *>(ws);
        args.ws_decay = reinterpret_cast<float *>(ws + ((state + 255) / 256) * 256);
        if (plan.varlen) {
            int *table = reinterpret_cast<int *>(ws + ((state + 255) / 256) * 256 +
                                                 ((decay + 255) / 256) * 256);
            args.item0 = table;
            args.fslot0 = table + (batch + 1);
        }
    }
    args.cu = plan.varlen ? cu_dev : nullptr;
    args.nseq = plan.varlen ? batch : 0;
    args.y = static_cast<__nv_bfloat16 *>(y);
    args.fin = fin;
    args.err = err;
    const SsdDebug dbg = ssd_debug_config();
    args.wait_ns = dbg.wait_ns;
    args.fault = dbg.fault;
    args.L = L;
    args.H = H;
    args.G = G;
    args.tiles = plan.tiles;
    args.seg_tiles = plan.seg_tiles;
    args.nseg = plan.nseg;
    // one instantiation per (heads per CTA, output gate, packed layout): the
    // plain batched path carries neither the gate nor the packed bookkeeping
    // (registers it cannot spare)
    const bool fused = fuse.z != nullptr;
#define SSD_LAUNCH_HG(HG, X, PK) \
    launch_hg<HG, X, PK>(plan, mC, mB, mX, mY, mZ, args, batch, H, prof, stream)
    if (plan.varlen) {
        if (plan.heads_per_cta == 2) return fused ? SSD_LAUNCH_HG(2, true, true) : SSD_LAUNCH_HG(2, false, true);
        return fused ? SSD_LAUNCH_HG(1, true, true) : SSD_LAUNCH_HG(1, false, true);
    }
    if (plan.heads_per_cta == 2) return fused ? SSD_LAUNCH_HG(2, true, false) : SSD_LAUNCH_HG(2, false, false);
    return fused ? SSD_LAUNCH_HG(1, true, false) : SSD_LAUNCH_HG(1, false, false);
#undef SSD_LAUNCH_HG
}
