// Decode path of the hyper-connection read: a few tokens per call (up to 64 in one pass
// over the weights), latency-bound, with the 13 MB of bf16 weights every pass streams as
// its floor.
//
// Two kernels per pass (1-8 tokens; 9-16 as two passes of up to 8; 17-64 in one pass
// whose down kernel runs the tokens in chunks), chained by programmatic dependent
// launch so that each kernel's weight stream starts while the previous kernel on
// the stream is still running:
//
//  down_slice_kernel - the down projection split into 8 K slices (half a stream,
//      1280 columns) x 20 row blocks (16 of the 320 rows). The norm is folded in
//      ("#2488 sycl/A770: faster hyper-connection read on Arc A-series",
//      Summary, change 4): a slice stages R' * w_norm unscaled together with its
//      per-token sum of squares, and the reduce applies each stream's rs to that
//      stream's partial dots. The 8 slices of a row block form one thread-block
//      cluster: each pushes its partials into the shared memory of the CTA that
//      finishes those rows, one cluster barrier publishes them, and each CTA sums
//      its inbox in a fixed order (the page's change 1 does it with the last slice
//      to finish; a cluster needs no global counter), so the result is bitwise
//      repeatable.
//
//  up_mix_tc_kernel - the up projection of all the pass's tokens at once on the
//      tcgen05 tensor cores (W_up rows as A, lo as three bf16 terms as B, D in
//      TMEM), then the gate and the 4x4 mix in its epilogue ("#1370 prefill:
//      opt-in STRATA_HC_UPMIX=1 on CUDA ...", "What it does": the mix fused into
//      the up projection, writing mixed with its BF16 / FP16 images). The launcher
//      uses it for every T.
//
// Weights are requested before anything else, so a kernel's whole weight matrix is in
// flight at once: the down kernel loads its slice straight into registers with
// 16-byte streaming loads, the up kernel its 128 W_up rows into shared memory by TMA.
//
// A CUDA-core up kernel (a warp per 4 output columns, 8 lanes per column, an xor
// tree for the dots) came before the tcgen05 one; its measured times are given at
// the launcher below.
//
// decode_read_kernel is the same read as one kernel (the down kernel's body as its
// first phase, a global exchange of lo, an up phase on the CUDA cores); it is the
// HC_PATH_DECODE_ONE_KERNEL path and is described above it.
//
// Only the weight pointers carry __restrict__. A load through a const __restrict__
// pointer may be treated as invariant and moved above griddepcontrol.wait; the
// activations (R, P, lo, Rmix) are written by the kernels before these on the
// stream, so their loads must stay after the wait.
#include <cooperative_groups.h>

#include <atomic>

#include "hc_common.cuh"
#include "hc_internal.h"
#include "hc_tc.cuh"

namespace hc {

namespace {

constexpr int kDownThreads = 320;   // 10 warps: 2 row groups x 5 column groups
constexpr int kDownColGroups = 5;   // 5 x 256 columns = 1280

// Sum over the 32 lanes of eight per-lane values, one per row. On return the
// lanes whose bits (4,3,2) equal the row's index hold that row's full sum:
// row = (lane >> 2) & 7. Nine shuffles, fixed order.
__device__ __forceinline__ float warp_reduce_8rows(const float (&v)[8], int lane) {
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float send = b4 ? v[i] : v[i + 4];
        float keep = b4 ? v[i + 4] : v[i];
        a[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
    float b[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        float send = b3 ? a[i] : a[i + 2];
        float keep = b3 ? a[i + 2] : a[i];
        b[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    float send = b2 ? b[0] : b[1];
    float keep = b2 ? b[1] : b[0];
    float c = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    c += __shfl_xor_sync(0xffffffffu, c, 2);
    c += __shfl_xor_sync(0xffffffffu, c, 1);
    return c;
}

// T: tokens per chunk. The kernel reads its slice of W_down from HBM once and runs
// the call's ntok tokens (at most 64) through it in chunks of T (the last chunk may
// hold fewer). Each chunk stages its activations, takes the dot products and keeps
// the CTA's partial of each token in shared memory; one exchange in the cluster then
// finishes every token. kMulti = false: exactly one chunk (ntok == T). kMulti = true:
// several; after its dot products each chunk loads the CTA's 40 KB slice of W_down
// again for the next one, from L2, where the first load left it (holding the weights
// in registers across a chunk would spill at the two-CTAs-per-SM register budget).
// The staged activations live in dynamic shared memory: T x 5 KB.
constexpr int kMultiMaxT = 64;   // tokens of one multi-chunk pass at most

//
// The body is a device function shared with the one-kernel read (decode_read_kernel),
// which runs it as its first phase. Hooks: hk.before_wait() is called by every thread
// once the weight loads are issued, right before the dependency wait, hk.after_wait()
// right after it, and hk.store_lo(i, v) stores lo element i (token * 320 + row); the
// row-finishing stores are made by warp 0 alone when ntok <= 16. The staging area (T x
// 5 KB) starts `a_off` bytes into the dynamic shared memory (addressed from the extern
// array itself, so that the compiler keeps shared-memory loads and stores).
template <int T, bool kMulti, typename Hooks>
__device__ __forceinline__ void down_phase(const float* R, const float* P,
                                           const uint16_t* __restrict__ w_norm,
                                           const uint16_t* __restrict__ W_down, float eps,
                                           int ntok_run, int* status, int a_off, Hooks& hk) {
    namespace cg = cooperative_groups;
    constexpr int NT = kMulti ? kMultiMaxT : T;   // tokens the exchange holds at most
    const int sl = blockIdx.x;                 // K slice 0..7 == rank in the cluster
    const int rb = blockIdx.y;                 // row block 0..19 == the cluster
    const int s = sl >> 1;                     // stream of the slice
    const int c0 = (sl & 1) * kDownSliceCols;  // first column of the slice in the stream
    const int k0 = s * kWidth + c0;            // first column on the 10240 axis
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int rg = warp / kDownColGroups, cgp = warp % kDownColGroups;
    const int j0 = rb * kDownRowsPerCta + rg * 8;
    const int col = cgp * 256 + lane * 8;      // this lane's 8 columns within the slice
    const int ntok = kMulti ? ntok_run : T;

    // 1. weights first (layer parameters may be read before the previous kernel
    //    on the stream has finished): 8 rows x 8 columns, one 16-byte load per row
    uint4 wv[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const size_t wi = (size_t)(j0 + r) * kCols + k0 + col;
        wv[r] = HC_IN_RANGE(wi, 8, (size_t)kRank * kCols, status) ? ldg_stream_v4(W_down + wi)
                                                                  : make_uint4(0, 0, 0, 0);
    }
    const uint2 wn = HC_IN_RANGE(k0 + 4 * tid, 4, kCols, status)
                         ? *reinterpret_cast<const uint2*>(w_norm + k0 + 4 * tid)
                         : make_uint2(0, 0);
    // first half of a cluster barrier: the wait before the pushes of step 4 then
    // finds every CTA of the cluster started (their shared memory exists)
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    // the activations into L2 while the previous kernel finishes (read after the wait)
    if ((tid & 7) == 0) {   // one prefetch per 128-byte line
        for (int t = 0; t < ntok; ++t) {
            prefetch_l2(R + (size_t)t * kCols + k0 + 4 * tid);
            if (P != nullptr) prefetch_l2(P + (size_t)t * kCols + k0 + 4 * tid);
        }
    }
    hk.before_wait();
    pdl_launch_dependents();
    pdl_wait();
    hk.after_wait();

    // staged activations a = R' * w_norm of a chunk. Layout: a lane's 8 columns are
    // stored as two float4 runs, 128 floats apart, so that consecutive lanes read
    // consecutive 16-byte words.
    extern __shared__ __align__(16) uint8_t down_dyn[];
    auto a_s = reinterpret_cast<float4 (*)[kDownSliceCols / 4]>(down_dyn + a_off);
    __shared__ float red_ss[kDownThreads / 32][T];
    __shared__ float red[T][kDownColGroups][kDownRowsPerCta];
    __shared__ float part[NT][kDownRowsPerCta];    // this slice's partial of each token
    __shared__ float ss_p[NT];                     // this slice's sums of squares
    __shared__ float inbox[kDownSlices][NT][3];    // pushed by each slice: 2 partials, ss
    const float w0 = bf16_lo(wn.x), w1 = bf16_hi(wn.x), w2 = bf16_lo(wn.y), w3 = bf16_hi(wn.y);

#pragma unroll 1
    for (int tc0 = 0; tc0 < ntok; tc0 += T) {
        const int nt = ntok - tc0 < T ? ntok - tc0 : T;   // tokens of this chunk
        const float* Rc = R + (size_t)tc0 * kCols;
        const float* Pc = P != nullptr ? P + (size_t)tc0 * kCols : nullptr;

        // 2. activations and per-token sums of squares of R' (zero past the chunk's
        //    tokens)
        float4 xs[T];
        const size_t act_extent = (size_t)ntok * kCols;   // R and P from the pass's start
        (void)act_extent;
#pragma unroll
        for (int t = 0; t < T; ++t)
            xs[t] = t < nt && HC_IN_RANGE((size_t)(tc0 + t) * kCols + k0 + 4 * tid, 4, act_extent, status)
                        ? *reinterpret_cast<const float4*>(Rc + (size_t)t * kCols + k0 + 4 * tid)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
        if (Pc != nullptr) {
#pragma unroll
            for (int t = 0; t < T; ++t) {
                if (t >= nt) continue;
                if (!HC_IN_RANGE((size_t)(tc0 + t) * kCols + k0 + 4 * tid, 4, act_extent, status)) continue;
                const float4 p = *reinterpret_cast<const float4*>(Pc + (size_t)t * kCols + k0 + 4 * tid);
                xs[t].x += p.x; xs[t].y += p.y; xs[t].z += p.z; xs[t].w += p.w;
            }
        }
        {
            const int c = 4 * tid;                       // first of this thread's 4 columns
            const int scg = c >> 8, slane = (c & 255) >> 3, half = (c & 7) >> 2;
            const int slot = scg * 64 + half * 32 + slane;   // float4 index
            // all tokens' sums over the warp in one 8-row reduce-scatter: 9 shuffles for
            // any T instead of 5 per token (measured: T = 8 10.23 -> 9.81 us per read).
            // It pairs lanes at the same distances as a per-token xor butterfly, so each
            // token's sum has the same bits, and no token's tree depends on the others.
            float ssv[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) ssv[t] = 0.f;
#pragma unroll
            for (int t = 0; t < T; ++t) {
                const float4 x = xs[t];
                float ss = x.x * x.x;
                ss = fmaf(x.y, x.y, ss);
                ss = fmaf(x.z, x.z, ss);
                ss = fmaf(x.w, x.w, ss);
                a_s[t][slot] = make_float4(x.x * w0, x.y * w1, x.z * w2, x.w * w3);
                ssv[t] = ss;
            }
            const float ssum = warp_reduce_8rows(ssv, lane);
            const int tr = (lane >> 2) & 7;
            if ((lane & 3) == 0 && tr < T) red_ss[warp][tr] = ssum;
        }
        __syncthreads();
        if (tid < T && tid < nt) {
            float ss = 0.f;
#pragma unroll
            for (int w = 0; w < kDownThreads / 32; ++w) ss += red_ss[w][tid];
            ss_p[tc0 + tid] = ss;
        }

        // 3. partial dots of 8 rows over this lane's 8 columns, reduced over the warp
        float wf[8][8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            wf[r][0] = bf16_lo(wv[r].x); wf[r][1] = bf16_hi(wv[r].x);
            wf[r][2] = bf16_lo(wv[r].y); wf[r][3] = bf16_hi(wv[r].y);
            wf[r][4] = bf16_lo(wv[r].z); wf[r][5] = bf16_hi(wv[r].z);
            wf[r][6] = bf16_lo(wv[r].w); wf[r][7] = bf16_hi(wv[r].w);
        }
#pragma unroll
        for (int t = 0; t < T; ++t) {
            const float4 x0 = a_s[t][cgp * 64 + lane];
            const float4 x1 = a_s[t][cgp * 64 + 32 + lane];
            float acc[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                float v = wf[r][0] * x0.x;
                v = fmaf(wf[r][1], x0.y, v);
                v = fmaf(wf[r][2], x0.z, v);
                v = fmaf(wf[r][3], x0.w, v);
                v = fmaf(wf[r][4], x1.x, v);
                v = fmaf(wf[r][5], x1.y, v);
                v = fmaf(wf[r][6], x1.z, v);
                v = fmaf(wf[r][7], x1.w, v);
                acc[r] = v;
            }
            const float sum = warp_reduce_8rows(acc, lane);
            if ((lane & 3) == 0) red[t][cgp][rg * 8 + ((lane >> 2) & 7)] = sum;
        }
        if constexpr (kMulti) {
            // the next chunk's weights, from L2: issued here, where few registers are
            // live, so that they arrive while this chunk is summed and the next staged
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const size_t wi = (size_t)(j0 + r) * kCols + k0 + col;
                wv[r] = HC_IN_RANGE(wi, 8, (size_t)kRank * kCols, status)
                            ? *reinterpret_cast<const uint4*>(W_down + wi)
                            : make_uint4(0, 0, 0, 0);
            }
        }
        __syncthreads();
        // this slice's partial for each of its 16 rows: column groups summed in order
        if (tid < T * kDownRowsPerCta && tid / kDownRowsPerCta < nt) {
            const int t = tid / kDownRowsPerCta, j = tid % kDownRowsPerCta;
            float v = red[t][0][j];
#pragma unroll
            for (int g = 1; g < kDownColGroups; ++g) v += red[t][g][j];
            part[tc0 + t][j] = v;
        }
        // (the next chunk writes red and a_s only after the barrier that follows its
        // staging, which every thread reaches after these reads)
    }
    __syncthreads();

    // 4. the partials pushed into the shared memory of the CTA that finishes the row:
    //    CTA d finishes rows 2d and 2d+1 of the block and receives, from every slice
    //    r, those two partials and r's sums of squares, for every token. Remote stores
    //    need no round trip, and after the one cluster barrier that publishes them no
    //    CTA touches another's memory. The wait first: every CTA of the cluster has
    //    started.
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    cg::cluster_group cluster = cg::this_cluster();
    for (int i = tid; i < ntok * kDownRowsPerCta; i += kDownThreads) {
        const int t = i / kDownRowsPerCta, j = i % kDownRowsPerCta;
        *cluster.map_shared_rank(&inbox[sl][t][j & 1], j >> 1) = part[t][j];
    }
    for (int i = tid; i < ntok * kDownSlices; i += kDownThreads) {
        const int t = i / kDownSlices, d = i % kDownSlices;
        *cluster.map_shared_rank(&inbox[sl][t][2], d) = ss_p[t];
    }
    cluster.sync();

    // 5. CTA `sl` finishes rows 2*sl and 2*sl+1 of the block, summing the slices of
    //    each stream in order and applying that stream's rs
    for (int i = tid; i < ntok * 2; i += kDownThreads) {
        const int t = i >> 1, jj = i & 1;
        float v = 0.f;
#pragma unroll
        for (int st = 0; st < kStreams; ++st) {
            const float ss = inbox[2 * st][t][2] + inbox[2 * st + 1][t][2];
            const float rs = inv_rms(fmaf(ss, 1.0f / (float)kWidth, eps));
            const float d = inbox[2 * st][t][jj] + inbox[2 * st + 1][t][jj];
            v = fmaf(rs, d, v);
        }
        const size_t li = (size_t)t * kRank + rb * kDownRowsPerCta + 2 * sl + jj;
        if (HC_IN_RANGE(li, 1, (size_t)ntok * kRank, status)) hk.store_lo(li, v);
    }
}

// lo to global memory, nothing around the wait: the two-kernel read.
struct PlainLo {
    float* lo;
    __device__ __forceinline__ void before_wait() {}
    __device__ __forceinline__ void after_wait() {}
    __device__ __forceinline__ void store_lo(size_t i, float v) { lo[i] = v; }
};

template <int T, bool kMulti>
__global__ void __cluster_dims__(kDownSlices, 1, 1) __launch_bounds__(kDownThreads, 2)
down_slice_kernel(const float* R, const float* P, const uint16_t* __restrict__ w_norm,
                  const uint16_t* __restrict__ W_down, float* lo, float eps, int ntok_run,
                  int* status) {
    PlainLo hk{lo};
    down_phase<T, kMulti>(R, P, w_norm, W_down, eps, ntok_run, status, 0, hk);
}

// Dynamic shared memory of down_slice_kernel<T, ...>: the staged activations.
template <int T> constexpr int kDownDynSmem = T * kDownSliceCols * 4;

// ---------------------------------------------------------------------------
// up_mix_tc_kernel - the up projection of a decode read on the tcgen05 tensor cores:
// all of the call's tokens (up to 64) in one pass of MMAs instead of a loop over them.
// A CTA owns 32 output columns: A = their 128 W_up rows (4 streams x 32 columns,
// bf16 as stored, loaded by TMA before the dependency wait). B = lo of the tokens as
// three bf16 terms hi + mid + low (split3_bf16), the terms side by side as B rows
// term * T + t, so that one MMA takes all three: N = 3T rounded up to 16. D = 128 x N
// fp32 in TMEM; each bf16 product is exact in fp32 and each term accumulates 20 MMAs
// deep; the epilogue adds a token's three columns, smallest first. TMEM lane = row,
// so warp w holds stream w and lane l column l; the gate is applied there, the four
// streams of a column meet in shared memory, and the mix writes each output row with
// stores that are contiguous across the warp.
//
// TM is the largest token count of the instantiation: for TM <= 8 the kernel reads
// exactly TM tokens; TM = 16, 32 and 64 take any T in (TM / 2, TM] (and 16 any T in
// 9..16), given at run time.
// ---------------------------------------------------------------------------
constexpr int kTcCols = 32;                          // output columns per CTA
constexpr int kTcRows = kStreams * kTcCols;          // 128 W_up rows: MMA M
constexpr int kTcKB = 64;                            // K per 128-byte swizzle row
constexpr int kTcKBlocks = kRank / kTcKB;            // 5
constexpr int kTcABytes = kTcRows * kTcKB * 2;       // 16 KB per K block
constexpr int kTcThreads = 128;
constexpr int kWideMaxT = 64;                        // tokens of one decode pass at most
// MMA N: 3 terms x TM tokens, rounded up to 16 (32 for 6-8 tokens)
template <int TM> constexpr int kTcN = (3 * TM + 15) / 16 * 16;
// B rows reserved: 32 for every TM <= 8, so that those kernels keep one shared-memory
// footprint (and one CTA per SM) whatever their token count
template <int TM> constexpr int kTcBRows = TM <= 8 ? 32 : kTcN<TM>;
template <int TM> constexpr int kTcSmem = kTcKBlocks * kTcABytes + kTcKBlocks * kTcBRows<TM> * kTcKB * 2 + 1024;
// TMEM columns: a power of two, at least 32
template <int TM> constexpr int kTcTmemCols = kTcN<TM> <= 32 ? 32 : kTcN<TM> <= 64 ? 64 : kTcN<TM> <= 128 ? 128 : 256;
static_assert(kTcSmem<kWideMaxT> <= 227 * 1024 - 8 * 1024, "up kernel shared memory");

// A bounded wait on an mbarrier phase: false after 2 s, with the timeout recorded in
// the status word when there is one (the allocation-free entry has none; the kernel
// then writes NaN outputs).
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, int* status) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = tc::globaltimer();
    while (!tc::mbar_try_wait_suspend(bar, parity, tc::kSuspendHintNs)) {
        if (tc::globaltimer() - t0 > tc::kWaitLimitNs) {
            if (status != nullptr) atomicOr(status, kStatusTimeout);
            return false;
        }
    }
    return true;
}

// 8 consecutive fp32 columns of this thread's TMEM lane at three column offsets, one
// wait for all three.
__device__ __forceinline__ void tmem_ld8x3(uint32_t a0, uint32_t a1, uint32_t a2, float (&h)[8],
                                           float (&m)[8], float (&l)[8]) {
    uint32_t r[24];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%24];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%25];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16,%17,%18,%19,%20,%21,%22,%23}, [%26];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23])
        : "r"(a0), "r"(a1), "r"(a2)
        : "memory");
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        h[e] = __uint_as_float(r[e]);
        m[e] = __uint_as_float(r[8 + e]);
        l[e] = __uint_as_float(r[16 + e]);
    }
}

// lo of T tokens ([T][kRank] fp32, read through L2) as three bf16 terms in the B tiles
// of an up MMA: K-major, 128-byte swizzled, one tile of `b_stride` bytes per 64-wide
// K block, rows term * T + t. Rows past 3 T stay unwritten: they only feed D columns
// nobody reads. kBatch loads of each thread are in flight at once.
template <int kThreadsN, int kBatch>
__device__ __forceinline__ void stage_lo_terms(const float* lo, int T, uint8_t* sB, int b_stride,
                                               int tid, int* status) {
    const int quads = T * kRank / 4;                     // float4 granules of lo
    for (int base = 0; base < quads; base += kBatch * kThreadsN) {
        float4 xq[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int e = base + tid + i * kThreadsN;
            if (e < quads && HC_IN_RANGE(4 * (size_t)e, 4, (size_t)T * kRank, status))
                xq[i] = __ldcg(reinterpret_cast<const float4*>(lo) + e);
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int e = base + tid + i * kThreadsN;
            if (e >= quads) continue;
            const int t = e / (kRank / 4), k = 4 * (e % (kRank / 4));
            uint32_t h0, m0, l0, h1, m1, l1;
            split3_bf16(xq[i].x, xq[i].y, h0, m0, l0);
            split3_bf16(xq[i].z, xq[i].w, h1, m1, l1);
            uint8_t* b = sB + (k / kTcKB) * b_stride;
            const int kin = k % kTcKB;
            *reinterpret_cast<uint2*>(b + tc::sw128_offset(t, kin)) = make_uint2(h0, h1);
            *reinterpret_cast<uint2*>(b + tc::sw128_offset(T + t, kin)) = make_uint2(m0, m1);
            *reinterpret_cast<uint2*>(b + tc::sw128_offset(2 * T + t, kin)) = make_uint2(l0, l1);
        }
    }
}

template <int TM>
__global__ void __launch_bounds__(kTcThreads, 1)
up_mix_tc_kernel(const __grid_constant__ CUtensorMap tm_wu, const float* R, const float* P,
                 const float* lo, const float* Rmix, float* out_f32, uint16_t* out_bf16,
                 uint16_t* out_fp16, int* status, int t_run) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned: the 128-byte swizzle pattern repeats every 8 rows of 128 B
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr bool kSmall = TM <= 8;
    constexpr int kN = kTcN<TM>, kBBytes = kN * kTcKB * 2;
    constexpr int kBStride = kTcBRows<TM> * kTcKB * 2;  // bytes per K block of B
    const int T = kSmall ? TM : t_run;                  // tokens of this read
    uint8_t* sA = smem;                                  // [K block][128 rows][128 B]
    uint8_t* sB = smem + kTcKBlocks * kTcABytes;         // [K block][N rows][128 B]
    __shared__ __align__(8) uint64_t w_full, mma_done;
    __shared__ uint32_t tmem_slot;
    __shared__ __align__(16) float m_s[TM][16];
    // gated values of the tokens: static for a few tokens, else over the A tiles once
    // the MMAs have read them
    __shared__ float g_small[kSmall ? TM : 1][kStreams][kTcCols];
    float (*g_s)[kStreams][kTcCols] =
        kSmall ? g_small : reinterpret_cast<float (*)[kStreams][kTcCols]>(sA);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x * kTcCols + lane;           // this thread's output column
    (void)kBBytes;

    if (tid == 0) {
        tc::mbar_init(&w_full, 1);
        tc::mbar_init(&mma_done, 1);
        tc::fence_barrier_init();
    }
    if (warp == 0) tc::tmem_alloc(&tmem_slot, kTcTmemCols<TM>);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = tmem_slot;

    // 1. the CTA's W_up rows (layer parameters, read before the wait): per K block
    //    one 32-row box per stream
    if (tid == 0) {
        tc::mbar_arrive_expect_tx(&w_full, kTcKBlocks * kTcABytes);
#pragma unroll
        for (int kb = 0; kb < kTcKBlocks; ++kb)
#pragma unroll
            for (int s = 0; s < kStreams; ++s)
                tc::tma_load_2d(sA + kb * kTcABytes + s * (kTcABytes / kStreams), &tm_wu, kb * kTcKB,
                                s * kWidth + blockIdx.x * kTcCols, &w_full);
    }
    // this thread's residual (and pending write) into L2 while the down kernel runs:
    // a warp's 32 columns of a stream are one 128-byte line
    if (lane == 0) {
        for (int t = 0; t < T; ++t) {
            prefetch_l2(R + (size_t)t * kCols + warp * kWidth + c);
            if (P != nullptr) prefetch_l2(P + (size_t)t * kCols + warp * kWidth + c);
        }
    }
    pdl_launch_dependents();
    pdl_wait();

    // 2. lo of the tokens as three bf16 terms in the B tiles (K-major, 128-byte
    //    swizzled, rows term * T + t), R' of this thread's (stream, column), the mix
    float rp[TM];
    const size_t act_extent = (size_t)T * kCols;
    (void)act_extent;
#pragma unroll
    for (int t = 0; t < TM; ++t) {
        const size_t ri = (size_t)t * kCols + warp * kWidth + c;
        rp[t] = t < T && HC_IN_RANGE(ri, 1, act_extent, status) ? R[ri] : 0.f;
    }
    if (P != nullptr) {
#pragma unroll
        for (int t = 0; t < TM; ++t) {
            const size_t ri = (size_t)t * kCols + warp * kWidth + c;
            if (t < T && HC_IN_RANGE(ri, 1, act_extent, status)) rp[t] += P[ri];
        }
    }
    constexpr int kBatch = kSmall ? (TM * kRank / 4 + kTcThreads - 1) / kTcThreads : 10;
    stage_lo_terms<kTcThreads, kBatch>(lo, T, sB, kBStride, tid, status);
    for (int e = tid; e < T * 4; e += kTcThreads)
        if (HC_IN_RANGE(4 * (size_t)e, 4, (size_t)T * 16, status))
            reinterpret_cast<float4*>(&m_s[0][0])[e] = reinterpret_cast<const float4*>(Rmix)[e];
    tc::fence_proxy_async_smem();
    __syncthreads();

    // 3. the MMAs, issued by one thread once the weights have landed (20 MMAs of N <= 32
    //    take about 0.7 us to issue, whether A is read from shared memory or from TMEM
    //    and whether they accumulate into one D or five: a per-instruction cost)
    __shared__ int ok_s;
    if (tid == 0) {
        bool ok = tc_wait(&w_full, 0, status);
        if (!ok) ok = tc_wait(&w_full, 0, status);   // give the copies in flight one more limit
        if (ok) {
            tc::tc_fence_after();
            constexpr uint32_t idesc = tc::idesc_bf16_f32(kTcRows, kN);
#pragma unroll
            for (int kb = 0; kb < kTcKBlocks; ++kb)
#pragma unroll
                for (int kk = 0; kk < kTcKB / 16; ++kk)
                    tc::mma_f16(tmem, tc::desc_sw128(tc::smem_u32(sA + kb * kTcABytes) + kk * 32),
                                tc::desc_sw128(tc::smem_u32(sB + kb * kBStride) + kk * 32), idesc,
                                (kb | kk) != 0);
            tc::mma_commit(&mma_done);
        }
        ok_s = ok;
    }
    __syncthreads();
    const bool ok = ok_s && tc_wait(&mma_done, 0, status);

    // 4. gate in place (warp = stream, lane = column), the streams meet in shared
    //    memory (over the A tiles for many tokens: the MMAs have read them), then the
    //    mix and the three images
    if (ok) {
        tc::tc_fence_after();
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        if constexpr (kSmall) {
            float u[32];
            tc::tmem_ld32(lane_base, u);
#pragma unroll
            for (int t = 0; t < TM; ++t)
                g_s[t][warp][lane] = gate_value((u[2 * TM + t] + u[TM + t]) + u[t], rp[t]);
        } else {
#pragma unroll
            for (int g0 = 0; g0 < TM; g0 += 8) {
                if (g0 >= T) break;
                float h[8], m[8], l[8];
                tmem_ld8x3(lane_base + g0, lane_base + T + g0, lane_base + 2 * T + g0, h, m, l);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (g0 + e < T) g_s[g0 + e][warp][lane] = gate_value((l[e] + m[e]) + h[e], rp[g0 + e]);
            }
        }
    }
    tc::tc_fence_before();
    __syncthreads();
#pragma unroll(kSmall ? TM : 1)
    for (int t = 0; t < T; ++t) {
        // a CTA whose wait gave up writes NaN, so that even a caller without a status
        // word (the allocation-free entry) finds no stale values in its outputs
        const float m = ok ? mix_row(&m_s[t][warp * 4], g_s[t][0][lane], g_s[t][1][lane],
                                     g_s[t][2][lane], g_s[t][3][lane])
                           : __int_as_float(0x7fc00000);
        const size_t off = (size_t)t * kCols + warp * kWidth + c;
        if (!HC_IN_RANGE(off, 1, act_extent, status)) continue;
        out_f32[off] = m;
        out_bf16[off] = to_bf16_bits(m);
        out_fp16[off] = to_fp16_bits(m);
    }
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTcTmemCols<TM>);
    }
}

// ---------------------------------------------------------------------------
// decode_read_kernel - the whole read of up to 8 tokens as one kernel ("#2226
// STRATA_HC_PERSIST=1 (opt-in, HIP): the verifier's hyper-connection read as one
// persistent kernel", Summary: at 1-8 tokens the read is dominated by launches and
// global dependencies; one kernel whose blocks split the down projection by column
// slices, reduce, then run the up projection).
//
// The grid is the down kernel's: 20 clusters (row blocks) of 8 CTAs (K slices), two
// CTAs per SM, all resident at once (checked at set-up). Each CTA
//  1. issues its weight streams before the dependency wait: its W_down slice into
//     registers (the down phase) and, by bulk copy, the 64 W_up rows of its 16 output
//     columns (4 streams x 16 columns, bf16 as stored) into shared memory, one row
//     per copy into rows padded to 656 bytes (conflict-free 16-byte reads below);
//  2. reads the call count right after the wait (its latency hides behind the
//     staging), then runs the down phase (down_phase): its 2 finished rows of lo go
//     to global memory;
//  3. publishes them: one release-add on its row block's counter. Every CTA then
//     waits until all 20 row blocks' counters have reached 8 adds for this call, one
//     lane per counter, bounded by %globaltimer (the context's wait limit), and reads
//     lo through L2 into shared memory;
//  4. runs the up projection on the CUDA cores: thread (segment q, row r) takes the
//     dot of W_up row r with lo over K = 64q .. 64q+63 for every token (fp32 fused
//     multiply-adds, even and odd groups of four in two chains added at the end), and
//     the five segments are added in order;
//  5. gates, mixes and writes its 16 columns x 4 streams of every token.
//
// The tensor cores are not used here: a kernel that touches tensor memory runs one CTA
// per SM (measured with the occupancy API), too few for this grid, and at 1-8 tokens
// the up projection is 64 T x 320 multiply-adds per CTA.
//
// Measured, this read is slower than the two kernels (8.6-9.0 against 7.2 us at T = 4
// with P): a per-phase %globaltimer trace puts about 2 us between the last CTA's lo
// stores and the pollers seeing them, against about 0.9 us for the two kernels'
// hand-off through the end of the down grid; a tagged-word exchange (value and call
// tag in one 64-bit store, the pollers reading the table itself) took as long.
//
// Counters: sync[0..19] count the publishing CTAs of each row block over all calls
// (8 per call), sync[20] is the number of calls completed. Every CTA reads sync[20]
// after the dependency wait and before it publishes; CTA 0 adds one to it after its
// wait has seen every row block complete, when every CTA of the call has read it.
// The next call reads it after its own dependency wait, when this grid has finished.
// A wait that runs out records a timeout and the CTA writes NaN outputs;
// hc_read_status, which reports the timeout, zeroes the counters.
// ---------------------------------------------------------------------------
constexpr int kRdCols = kWidth / (kDownSlices * kDownRowBlocks);   // 16 output columns a CTA
constexpr int kRdRows = kStreams * kRdCols;                        // 64 W_up rows
constexpr int kRdRowBytes = kRank * 2 + 16;                        // padded row: 656 B
constexpr int kRdWBytes = kRdRows * kRdRowBytes;                   // 41 KB
constexpr int kRdSegs = kDownThreads / kRdRows;                    // 5 K segments of 64
constexpr int kRdSegLen = kRank / kRdSegs;                         // 64
template <int T> constexpr int kRdSmem = kRdWBytes + kDownDynSmem<T>;
static_assert(kRdSegs * kRdRows == kDownThreads && kRdSegLen % 8 == 0, "up mapping");
static_assert(2 * (kRdSmem<kDecodeMaxT> + 12 * 1024) <= 228 * 1024, "two CTAs per SM");
static_assert(kDownRowBlocks + 1 <= kSyncWords, "exchange counters");

__device__ __forceinline__ uint32_t ld_acquire_u32(const unsigned* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// The one-kernel read's hooks into the down phase: W_up rows requested before the
// wait, the call count read after it, lo stored to global memory.
struct CountedLo {
    const uint16_t* W_up;
    uint8_t* sW;
    uint64_t* w_full;
    int cbase;
    int* status;
    float* lo;
    const unsigned* calls;
    unsigned gen;
    __device__ __forceinline__ void before_wait() {
        if (threadIdx.x >= 32) return;
        const int lane = threadIdx.x;
        if (lane == 0) {
            tc::mbar_init(w_full, 1);
            tc::fence_barrier_init();
            tc::mbar_arrive_expect_tx(w_full, kRdRows * kRank * 2);
        }
        __syncwarp();
        // row r = stream * 16 + column; two row copies per lane
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = lane + 32 * h;
            const size_t wi = (size_t)((r / kRdCols) * kWidth + cbase + r % kRdCols) * kRank;
            const uint32_t dst = tc::smem_u32(sW + r * kRdRowBytes);
            const uint32_t bar = tc::smem_u32(w_full);
            if (HC_IN_RANGE(wi, kRank, (size_t)kCols * kRank, status)) {
                asm volatile(
                    "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                    "l"(W_up + wi), "r"((uint32_t)(kRank * 2)), "r"(bar)
                    : "memory");
            } else {
                // the copy is skipped: its bytes still count, so the wait ends
                asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(bar),
                             "r"((uint32_t)(kRank * 2))
                             : "memory");
            }
        }
    }
    __device__ __forceinline__ void after_wait() { gen = ld_acquire_u32(calls); }
    __device__ __forceinline__ void store_lo(size_t i, float v) { lo[i] = v; }
};

template <int T>
__global__ void __cluster_dims__(kDownSlices, 1, 1) __launch_bounds__(kDownThreads, 2)
decode_read_kernel(const float* R, const float* P, const uint16_t* __restrict__ w_norm,
                   const uint16_t* __restrict__ W_down, const uint16_t* __restrict__ W_up,
                   const float* Rmix, float* out_f32, uint16_t* out_bf16, uint16_t* out_fp16,
                   float* lo, unsigned* sync, float eps, int* status, uint64_t lo_wait_ns) {
    extern __shared__ __align__(16) uint8_t rd_dyn[];
    uint8_t* sW = rd_dyn;                                 // [64 rows][656 B]
    // staged activations of the down phase, then lo [T][320] and the segment partials
    float* lo_s = reinterpret_cast<float*>(rd_dyn + kRdWBytes);
    float* part_s = lo_s + T * kRank;                     // [T][5 segments][64 rows]
    __shared__ __align__(8) uint64_t w_full;
    __shared__ int ok_s;
    __shared__ __align__(16) float m_s[T][16];
    __shared__ float g_s[T][kStreams][kRdCols];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cid = blockIdx.y * kDownSlices + blockIdx.x;
    const int cbase = cid * kRdCols;                      // first output column of the CTA

    // 1-2. weights, call count, the down phase
    CountedLo hk{W_up, sW, &w_full, cbase, status, lo, &sync[kDownRowBlocks], 0u};
    down_phase<T, false>(R, P, w_norm, W_down, eps, T, status, kRdWBytes, hk);

    // R' of the gate elements (token t, W_up row r) and the mix, loaded while the other
    // clusters finish: element e = t * 64 + r, at most two per thread
    const size_t act_extent = (size_t)T * kCols;
    (void)act_extent;
    float rp[2] = {0.f, 0.f};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int e = tid + h * kDownThreads;
        if (e >= T * kRdRows) continue;
        const int t = e / kRdRows, r = e % kRdRows;
        const size_t ri = (size_t)t * kCols + (r / kRdCols) * kWidth + cbase + r % kRdCols;
        if (!HC_IN_RANGE(ri, 1, act_extent, status)) continue;
        rp[h] = R[ri];
        if (P != nullptr) rp[h] += P[ri];
    }
    for (int e = tid; e < T * 4; e += kDownThreads)
        if (HC_IN_RANGE(4 * (size_t)e, 4, (size_t)T * 16, status))
            reinterpret_cast<float4*>(&m_s[0][0])[e] = reinterpret_cast<const float4*>(Rmix)[e];

    // 3. publish this CTA's rows (stored by warp 0's lanes), wait for every row block
    if (warp == 0) {
        __syncwarp();
        if (lane == 0)
            asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&sync[blockIdx.y]) : "memory");
        bool ok = true;
        if (lane < kDownRowBlocks) {
            const unsigned target = (hk.gen + 1) * (unsigned)kDownSlices;
            if ((int)(ld_acquire_u32(&sync[lane]) - target) < 0) {
                const uint64_t t0 = tc::globaltimer();
                while ((int)(ld_acquire_u32(&sync[lane]) - target) < 0) {
                    if (tc::globaltimer() - t0 > lo_wait_ns) {
                        atomicOr(status, kStatusTimeout);
                        ok = false;
                        break;
                    }
                }
            }
        }
        ok = __all_sync(0xffffffffu, ok);
        if (lane == 0) {
            ok_s = ok;
            if (ok && cid == 0) sync[kDownRowBlocks] = hk.gen + 1;
        }
    }
    __syncthreads();
    //    lo into shared memory (over the staging area: its last reads were before the
    //    down phase's last barrier); then the W_up rows must have landed
    const bool lo_ok = ok_s;
    for (int e = tid; e < T * kRank / 4; e += kDownThreads) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (lo_ok && HC_IN_RANGE(4 * (size_t)e, 4, (size_t)T * kRank, status))
            v = __ldcg(reinterpret_cast<const float4*>(lo) + e);
        reinterpret_cast<float4*>(lo_s)[e] = v;
    }
    if (tid == 0) {
        // waited for even when lo is missing: no copy may still be in flight at exit
        bool w_ok = tc_wait(&w_full, 0, status);
        if (!w_ok) w_ok = tc_wait(&w_full, 0, status);
        ok_s = lo_ok && w_ok;
    }
    __syncthreads();
    const bool ok = ok_s;

    // 4. the dots: thread (q, r) over K = 64q .. 64q+63, all tokens
    {
        const int r = tid % kRdRows, q = tid / kRdRows;
        const uint4* wrow = reinterpret_cast<const uint4*>(sW + r * kRdRowBytes + q * kRdSegLen * 2);
        float acc0[T], acc1[T];
#pragma unroll
        for (int t = 0; t < T; ++t) acc0[t] = acc1[t] = 0.f;
#pragma unroll
        for (int i = 0; i < kRdSegLen / 8; ++i) {
            const uint4 w = wrow[i];
            const float wf[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                                 bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
#pragma unroll
            for (int t = 0; t < T; ++t) {
                const float4* l4 = reinterpret_cast<const float4*>(lo_s + t * kRank + q * kRdSegLen + 8 * i);
                const float4 x0 = l4[0], x1 = l4[1];
                float a = acc0[t], b = acc1[t];
                a = fmaf(wf[0], x0.x, a);
                b = fmaf(wf[4], x1.x, b);
                a = fmaf(wf[1], x0.y, a);
                b = fmaf(wf[5], x1.y, b);
                a = fmaf(wf[2], x0.z, a);
                b = fmaf(wf[6], x1.z, b);
                a = fmaf(wf[3], x0.w, a);
                b = fmaf(wf[7], x1.w, b);
                acc0[t] = a;
                acc1[t] = b;
            }
        }
#pragma unroll
        for (int t = 0; t < T; ++t) part_s[(t * kRdSegs + q) * kRdRows + r] = acc0[t] + acc1[t];
    }
    __syncthreads();

    // 5. u of (token, row): the segments added in order, then the gate; the four
    //    streams of a column meet in shared memory; then the mix and the three images
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int e = tid + h * kDownThreads;
        if (e >= T * kRdRows) continue;
        const int t = e / kRdRows, r = e % kRdRows;
        const float* p = part_s + t * kRdSegs * kRdRows + r;
        float u = p[0];
#pragma unroll
        for (int q = 1; q < kRdSegs; ++q) u += p[q * kRdRows];
        g_s[t][r / kRdCols][r % kRdCols] = gate_value(u, rp[h]);
    }
    __syncthreads();
    for (int i = tid; i < T * kStreams * kRdCols; i += kDownThreads) {
        const int l = i % kRdCols, o = (i / kRdCols) % kStreams, t = i / (kRdCols * kStreams);
        const float m = ok ? mix_row(&m_s[t][o * 4], g_s[t][0][l], g_s[t][1][l], g_s[t][2][l],
                                     g_s[t][3][l])
                           : __int_as_float(0x7fc00000);
        const size_t off = (size_t)t * kCols + o * kWidth + cbase + l;
        if (!HC_IN_RANGE(off, 1, act_extent, status)) continue;
        out_f32[off] = m;
        out_bf16[off] = to_bf16_bits(m);
        out_fp16[off] = to_fp16_bits(m);
    }
}

// Launch with programmatic stream serialisation (see pdl_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The up kernel of every read is the tcgen05 one. Measured, µs per read with P, for
// T = 1..8: 6.13, 6.14, 6.67, 7.21, 7.94, 8.68, 9.63, 10.20, against 5.0, 6.1, 7.1,
// 7.9, 8.8, 9.7, 10.8, 12.2 with the CUDA-core up kernel it replaced. One kernel for
// every T keeps a token's bits independent of the other tokens of its call.

// Devices (bits) on which up_mix_tc_kernel<TM> has been allowed its dynamic shared
// memory, for TM = 1..8 and then 16, 32, 64. hc_read_init clears a device's bits
// (decode_forget_smem), so the attributes are set again after a device reset.
// Then the multi-chunk down kernels of 5..8 tokens a chunk (flags 12..15), whose
// staged activations and exchange arrays exceed the default 48 KB.
constexpr int kSmemFlags = kDecodeMaxT + 8;
std::atomic<unsigned long long> g_smem_set[kSmemFlags];
template <int TM> constexpr int smem_flag() { return TM <= 8 ? TM : TM == 16 ? 9 : TM == 32 ? 10 : 11; }

// Allows `kernel` `bytes` of dynamic shared memory on this device, once per device.
template <typename K>
cudaError_t allow_smem(K kernel, int bytes, int device, std::atomic<unsigned long long>& done) {
    if (bytes == 0) return cudaSuccess;
    const unsigned long long bit = device >= 0 && device < 64 ? 1ull << device : 0;
    if (bit != 0 && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
    return e;
}

template <int TM>
cudaError_t allow_up_tc(int device) {
    return allow_smem(up_mix_tc_kernel<TM>, kTcSmem<TM>, device, g_smem_set[smem_flag<TM>()]);
}

template <int TC>
cudaError_t allow_down_multi(int device) {
    return allow_smem(down_slice_kernel<TC, true>, kDownDynSmem<TC>, device, g_smem_set[7 + TC]);
}

// One decode pass over n <= 64 tokens starting at token t0: the down kernel in chunks
// of TC tokens (one pass over its weights), then the up kernel for all n tokens.
template <int TC, int TM>
cudaError_t launch_pass(const Ctx& ctx, const ReadArgs& a, int t0, int n, cudaStream_t st) {
    constexpr bool kMulti = TM > 8;
    const size_t off = (size_t)t0 * kCols;
    const float* R = a.R + off;
    const float* P = a.P ? a.P + off : nullptr;
    float* lo = ctx.s.lo + (size_t)t0 * kRank;
    const CUtensorMap* tm_wu = decode_w_up_map(ctx, a.W_up);
    if (tm_wu == nullptr) return cudaErrorInvalidValue;
    cudaError_t e = allow_up_tc<TM>(ctx.device);
    if (e == cudaSuccess && kMulti) e = allow_down_multi<TC>(ctx.device);
    if (e != cudaSuccess) return e;
    e = launch_pdl(down_slice_kernel<TC, kMulti>, dim3(kDownSlices, kDownRowBlocks), dim3(kDownThreads),
                   (size_t)kDownDynSmem<TC>, st, R, P, a.w_norm, a.W_down, lo, ctx.eps, n,
                   ctx.s.status);
    if (e != cudaSuccess) return e;
    return launch_pdl(up_mix_tc_kernel<TM>, dim3(kWidth / kTcCols), dim3(kTcThreads),
                      (size_t)kTcSmem<TM>, st, *tm_wu, R, P, (const float*)lo,
                      a.Rmix + (size_t)t0 * 16, a.out_f32 + off, a.out_bf16 + off,
                      a.out_fp16 + off, ctx.s.status, n);
}

// n tokens (9..64) read with the weights streamed once: chunks of TC = ceil(n / chunks)
// tokens in the down kernel, the smallest wide up kernel that holds n.
template <int TM>
cudaError_t launch_wide_tc(const Ctx& ctx, const ReadArgs& a, int t0, int n, int tc, cudaStream_t st) {
    switch (tc) {
        case 5: return launch_pass<5, TM>(ctx, a, t0, n, st);
        case 6: return launch_pass<6, TM>(ctx, a, t0, n, st);
        case 7: return launch_pass<7, TM>(ctx, a, t0, n, st);
        default: return launch_pass<8, TM>(ctx, a, t0, n, st);
    }
}

cudaError_t launch_wide(const Ctx& ctx, const ReadArgs& a, int t0, int n, cudaStream_t st) {
    const int chunks = (n + kDecodeMaxT - 1) / kDecodeMaxT;
    const int tc = (n + chunks - 1) / chunks;       // 5..8 for n in 9..64
    if (n <= 16) return launch_wide_tc<16>(ctx, a, t0, n, tc, st);
    if (n <= 32) return launch_wide_tc<32>(ctx, a, t0, n, tc, st);
    return launch_wide_tc<64>(ctx, a, t0, n, tc, st);
}

// One-kernel read of a chunk of T <= 8 tokens starting at token t0.
template <int T>
cudaError_t launch_read_chunk(const Ctx& ctx, const ReadArgs& a, int t0, cudaStream_t st) {
    const size_t off = (size_t)t0 * kCols;
    return launch_pdl(decode_read_kernel<T>, dim3(kDownSlices, kDownRowBlocks), dim3(kDownThreads),
                      (size_t)kRdSmem<T>, st, a.R + off, a.P ? a.P + off : nullptr, a.w_norm,
                      a.W_down, a.W_up, a.Rmix + (size_t)t0 * 16, a.out_f32 + off,
                      a.out_bf16 + off, a.out_fp16 + off, ctx.s.lo + (size_t)t0 * kRank, ctx.s.sync,
                      ctx.eps, ctx.s.status, ctx.lo_wait_ns);
}

template <int T>
cudaError_t allow_read_smem() {
    return cudaFuncSetAttribute(decode_read_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kRdSmem<T>);
}

}  // namespace

cudaError_t decode_fused_setup(bool* usable) {
    *usable = false;
    cudaError_t e = allow_read_smem<1>();
    if (e == cudaSuccess) e = allow_read_smem<2>();
    if (e == cudaSuccess) e = allow_read_smem<3>();
    if (e == cudaSuccess) e = allow_read_smem<4>();
    if (e == cudaSuccess) e = allow_read_smem<5>();
    if (e == cudaSuccess) e = allow_read_smem<6>();
    if (e == cudaSuccess) e = allow_read_smem<7>();
    if (e == cudaSuccess) e = allow_read_smem<8>();
    if (e != cudaSuccess) return e;
    // every cluster of the grid must be resident at once (the CTAs wait on each other);
    // otherwise the read keeps the two-kernel decode path
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kDownSlices, kDownRowBlocks);
    cfg.blockDim = dim3(kDownThreads);
    cfg.dynamicSmemBytes = kRdSmem<kDecodeMaxT>;
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, decode_read_kernel<kDecodeMaxT>, &cfg);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return cudaSuccess;
    }
    *usable = clusters >= kDownRowBlocks;
    return cudaSuccess;
}

cudaError_t launch_decode_fused(const Ctx& ctx, const ReadArgs& a, cudaStream_t st) {
    for (int t0 = 0; t0 < a.T; t0 += kDecodeMaxT) {
        const int n = a.T - t0 < kDecodeMaxT ? a.T - t0 : kDecodeMaxT;
        cudaError_t e;
        switch (n) {
            case 1: e = launch_read_chunk<1>(ctx, a, t0, st); break;
            case 2: e = launch_read_chunk<2>(ctx, a, t0, st); break;
            case 3: e = launch_read_chunk<3>(ctx, a, t0, st); break;
            case 4: e = launch_read_chunk<4>(ctx, a, t0, st); break;
            case 5: e = launch_read_chunk<5>(ctx, a, t0, st); break;
            case 6: e = launch_read_chunk<6>(ctx, a, t0, st); break;
            case 7: e = launch_read_chunk<7>(ctx, a, t0, st); break;
            default: e = launch_read_chunk<8>(ctx, a, t0, st); break;
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

const CUtensorMap* decode_w_up_map(const Ctx& ctx, const uint16_t* W_up) {
    WupMapCache& c = ctx.wu_maps;
    // Fibonacci hashing of the address: weight sets allocated back to back sit a fixed
    // stride apart, which a plain modulus would send to one slot
    const uint64_t h = (static_cast<uint64_t>(reinterpret_cast<uintptr_t>(W_up)) >> 8) *
                       0x9E3779B97F4A7C15ull;
    const int slot = static_cast<int>(h >> 58);   // 64 slots
    if (c.key[slot] == W_up) return &c.map[slot];
    c.key[slot] = nullptr;
    if (!encode_w_up_bf16(&c.map[slot], W_up, kTcCols)) return nullptr;
    c.key[slot] = W_up;
    return &c.map[slot];
}

void decode_forget_smem(int device) {
    if (device < 0 || device >= 64) return;
    for (auto& bits : g_smem_set) bits.fetch_and(~(1ull << device), std::memory_order_acq_rel);
}

cudaError_t decode_setup(int device) {
    decode_forget_smem(device);
    cudaError_t e = allow_up_tc<1>(device);
    if (e == cudaSuccess) e = allow_up_tc<2>(device);
    if (e == cudaSuccess) e = allow_up_tc<3>(device);
    if (e == cudaSuccess) e = allow_up_tc<4>(device);
    if (e == cudaSuccess) e = allow_up_tc<5>(device);
    if (e == cudaSuccess) e = allow_up_tc<6>(device);
    if (e == cudaSuccess) e = allow_up_tc<7>(device);
    if (e == cudaSuccess) e = allow_up_tc<8>(device);
    if (e == cudaSuccess) e = allow_up_tc<16>(device);
    if (e == cudaSuccess) e = allow_up_tc<32>(device);
    if (e == cudaSuccess) e = allow_up_tc<64>(device);
    if (e == cudaSuccess) e = allow_down_multi<5>(device);
    if (e == cudaSuccess) e = allow_down_multi<6>(device);
    if (e == cudaSuccess) e = allow_down_multi<7>(device);
    if (e == cudaSuccess) e = allow_down_multi<8>(device);
    return e;
}

// Any T: passes of up to 64 tokens. A pass of 1-8 tokens is one chunk (down and up
// kernels of exactly that many tokens); 17-64 tokens stream the weights once (one
// down kernel in chunks, one up kernel); 9-16 tokens run as two chunks of up to 8,
// whose kernels overlap by programmatic dependent launch. Measured on GB300 (µs per
// read with P, one weight set): one pass 20.4 / 36.8 / 71.8 at 16 / 32 / 64 tokens
// against 19.4 / 38.7 / 77.2 in chunks of 8. The time grows with the tokens in the
// down kernel's staging and dot products (about 5-7 µs per chunk of 8), not with the
// weight stream.
constexpr int kWideMinT = 17;

cudaError_t launch_decode(const Ctx& ctx, const ReadArgs& a, cudaStream_t st) {
    for (int t0 = 0; t0 < a.T;) {
        const int left = a.T - t0;
        const int n = left >= kWideMinT ? (left < kWideMaxT ? left : kWideMaxT)
                                        : (left < kDecodeMaxT ? left : kDecodeMaxT);
        const int p0 = t0;                       // first token of this pass
        t0 += n;
        cudaError_t e;
        switch (n) {
            case 1: e = launch_pass<1, 1>(ctx, a, p0, 1, st); break;
            case 2: e = launch_pass<2, 2>(ctx, a, p0, 2, st); break;
            case 3: e = launch_pass<3, 3>(ctx, a, p0, 3, st); break;
            case 4: e = launch_pass<4, 4>(ctx, a, p0, 4, st); break;
            case 5: e = launch_pass<5, 5>(ctx, a, p0, 5, st); break;
            case 6: e = launch_pass<6, 6>(ctx, a, p0, 6, st); break;
            case 7: e = launch_pass<7, 7>(ctx, a, p0, 7, st); break;
            case 8: e = launch_pass<8, 8>(ctx, a, p0, 8, st); break;
            default: e = launch_wide(ctx, a, p0, n, st); break;
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace hc
