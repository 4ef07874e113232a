// Decode path of the hyper-connection read: 1-8 tokens per launch, bound by the
// 13 MB of bf16 weights every read streams.
//
// Two kernels per chunk of up to 8 tokens, chained by programmatic dependent
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
//  up_mix_tc_kernel - the up projection of all the chunk's tokens at once on the
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

template <int T>
__global__ void __cluster_dims__(kDownSlices, 1, 1) __launch_bounds__(kDownThreads)
down_slice_kernel(const float* R, const float* P, const uint16_t* __restrict__ w_norm,
                  const uint16_t* __restrict__ W_down, float* lo, float eps) {
    namespace cg = cooperative_groups;
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

    // 1. weights first (layer parameters may be read before the previous kernel
    //    on the stream has finished): 8 rows x 8 columns, one 16-byte load per row
    uint4 wv[8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
        wv[r] = ldg_stream_v4(W_down + (size_t)(j0 + r) * kCols + k0 + col);
    const uint2 wn = *reinterpret_cast<const uint2*>(w_norm + k0 + 4 * tid);
    // first half of a cluster barrier: the wait before the pushes of step 4 then
    // finds every CTA of the cluster started (their shared memory exists)
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    // the activations into L2 while the previous kernel finishes (read after the wait)
#pragma unroll
    for (int t = 0; t < T; ++t) {
        if ((tid & 7) == 0) {   // one prefetch per 128-byte line
            prefetch_l2(R + (size_t)t * kCols + k0 + 4 * tid);
            if (P != nullptr) prefetch_l2(P + (size_t)t * kCols + k0 + 4 * tid);
        }
    }
    pdl_launch_dependents();
    pdl_wait();

    // 2. activations a = R' * w_norm (fp32) and per-token sums of squares of R'.
    //    Smem layout: a lane's 8 columns are stored as two float4 runs, 128 floats
    //    apart, so that consecutive lanes read consecutive 16-byte words.
    __shared__ float4 a_s[T][kDownSliceCols / 4];
    __shared__ float red_ss[kDownThreads / 32][T];
    __shared__ float red[T][kDownColGroups][kDownRowsPerCta];
    __shared__ float ss_s[T];                      // this slice's sums of squares
    __shared__ float inbox[kDownSlices][T][3];     // pushed by each slice: 2 partials, ss

    float4 xs[T];
#pragma unroll
    for (int t = 0; t < T; ++t)
        xs[t] = *reinterpret_cast<const float4*>(R + (size_t)t * kCols + k0 + 4 * tid);
    if (P != nullptr) {
#pragma unroll
        for (int t = 0; t < T; ++t) {
            const float4 p = *reinterpret_cast<const float4*>(P + (size_t)t * kCols + k0 + 4 * tid);
            xs[t].x += p.x; xs[t].y += p.y; xs[t].z += p.z; xs[t].w += p.w;
        }
    }
    const float w0 = bf16_lo(wn.x), w1 = bf16_hi(wn.x), w2 = bf16_lo(wn.y), w3 = bf16_hi(wn.y);
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
    if (tid < T) {
        float ss = 0.f;
#pragma unroll
        for (int w = 0; w < kDownThreads / 32; ++w) ss += red_ss[w][tid];
        ss_s[tid] = ss;
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
    __syncthreads();

    // 4. this slice's partial for its 16 rows, column groups summed in order, pushed
    //    into the shared memory of the CTA that finishes the row: CTA d finishes rows
    //    2d and 2d+1 of the block and receives, from every slice r, those two
    //    partials and r's sums of squares. Remote stores need no round trip, and after
    //    the one cluster barrier that publishes them no CTA touches another's memory.
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    cg::cluster_group cluster = cg::this_cluster();
    if (tid < T * kDownRowsPerCta) {
        const int t = tid / kDownRowsPerCta, j = tid % kDownRowsPerCta;
        float v = red[t][0][j];
#pragma unroll
        for (int g = 1; g < kDownColGroups; ++g) v += red[t][g][j];
        *cluster.map_shared_rank(&inbox[sl][t][j & 1], j >> 1) = v;
    } else if (tid >= 128 && tid < 128 + T * kDownSlices) {
        const int t = (tid - 128) / kDownSlices, d = (tid - 128) % kDownSlices;
        *cluster.map_shared_rank(&inbox[sl][t][2], d) = ss_s[t];
    }
    cluster.sync();

    // 5. CTA `sl` finishes rows 2*sl and 2*sl+1 of the block, summing the slices of
    //    each stream in order and applying that stream's rs
    if (tid < T * 2) {
        const int t = tid >> 1, jj = tid & 1;
        float v = 0.f;
#pragma unroll
        for (int st = 0; st < kStreams; ++st) {
            const float ss = inbox[2 * st][t][2] + inbox[2 * st + 1][t][2];
            const float rs = inv_rms(fmaf(ss, 1.0f / (float)kWidth, eps));
            const float d = inbox[2 * st][t][jj] + inbox[2 * st + 1][t][jj];
            v = fmaf(rs, d, v);
        }
        lo[t * kRank + rb * kDownRowsPerCta + 2 * sl + jj] = v;
    }
}

// ---------------------------------------------------------------------------
// up_mix_tc_kernel - the up projection of a decode chunk on the tcgen05 tensor
// cores: all of the chunk's tokens in one pass of MMAs instead of a loop over them.
// A CTA owns 32 output columns: A = their 128 W_up rows (4 streams x 32 columns,
// bf16 as stored, loaded by TMA before the dependency wait). B = lo of the chunk's
// tokens as three bf16 terms hi + mid + low (x - hi and x - hi - mid are exact in
// fp32, so the three carry x to about 2^-27 of its size), the terms side by side as
// B rows term * T + t, so that one MMA takes all three: N = 16 up to 5 tokens, 32
// above. D = 128 x N fp32 in TMEM; each bf16 product is exact in fp32 and each term
// accumulates 20 MMAs deep; the epilogue adds a token's three columns, smallest
// first. TMEM lane = row, so warp w holds stream w and lane l column l; the gate is
// applied there, the four streams of a column meet in shared memory, and the mix
// writes each output row with stores that are contiguous across the warp.
// ---------------------------------------------------------------------------
constexpr int kTcCols = 32;                          // output columns per CTA
constexpr int kTcRows = kStreams * kTcCols;          // 128 W_up rows: MMA M
constexpr int kTcKB = 64;                            // K per 128-byte swizzle row
constexpr int kTcKBlocks = kRank / kTcKB;            // 5
template <int T> constexpr int kTcN = 3 * T <= 16 ? 16 : 32;   // MMA N: 3 terms x T tokens
constexpr int kTcABytes = kTcRows * kTcKB * 2;       // 16 KB per K block
constexpr int kTcBBytesMax = 32 * kTcKB * 2;         // 4 KB per K block at N = 32
constexpr int kTcThreads = 128;
constexpr int kTcSmem = kTcKBlocks * kTcABytes + kTcKBlocks * kTcBBytesMax + 1024;
constexpr int kTcTmemCols = 32;                      // the smallest TMEM allocation

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

template <int T>
__global__ void __launch_bounds__(kTcThreads, 1)
up_mix_tc_kernel(const __grid_constant__ CUtensorMap tm_wu, const float* R, const float* P,
                 const float* lo, const float* Rmix, float* out_f32, uint16_t* out_bf16,
                 uint16_t* out_fp16, int* status) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned: the 128-byte swizzle pattern repeats every 8 rows of 128 B
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int kN = kTcN<T>, kBBytes = kN * kTcKB * 2;
    uint8_t* sA = smem;                                  // [K block][128 rows][128 B]
    uint8_t* sB = smem + kTcKBlocks * kTcABytes;         // [K block][N rows][128 B]
    __shared__ __align__(8) uint64_t w_full, mma_done;
    __shared__ uint32_t tmem_slot;
    __shared__ float g_s[T][kStreams][kTcCols];
    __shared__ __align__(16) float m_s[T][16];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x * kTcCols + lane;           // this thread's output column

    if (tid == 0) {
        tc::mbar_init(&w_full, 1);
        tc::mbar_init(&mma_done, 1);
        tc::fence_barrier_init();
    }
    if (warp == 0) tc::tmem_alloc(&tmem_slot, kTcTmemCols);
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
#pragma unroll
        for (int t = 0; t < T; ++t) {
            prefetch_l2(R + (size_t)t * kCols + warp * kWidth + c);
            if (P != nullptr) prefetch_l2(P + (size_t)t * kCols + warp * kWidth + c);
        }
    }
    pdl_launch_dependents();
    pdl_wait();

    // 2. lo of the chunk as three bf16 terms in the B tiles (K-major, 128-byte
    //    swizzled, tokens as rows), R' of this thread's (stream, column), the mix
    float rp[T];
#pragma unroll
    for (int t = 0; t < T; ++t) rp[t] = R[(size_t)t * kCols + warp * kWidth + c];
    if (P != nullptr) {
#pragma unroll
        for (int t = 0; t < T; ++t) rp[t] += P[(size_t)t * kCols + warp * kWidth + c];
    }
    // (rows past 3 T stay unwritten: they only feed D columns nobody reads)
    constexpr int kQuads = T * kRank / 4;                // float4 granules of lo
    constexpr int kIters = (kQuads + kTcThreads - 1) / kTcThreads;
    float4 xq[kIters];
#pragma unroll
    for (int i = 0; i < kIters; ++i) {                   // every load in flight at once
        const int e = tid + i * kTcThreads;
        if (e < kQuads) xq[i] = reinterpret_cast<const float4*>(lo)[e];
    }
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
        const int e = tid + i * kTcThreads;
        if (e >= kQuads) continue;
        const int t = e / (kRank / 4), k = 4 * (e % (kRank / 4));
        uint32_t h0, m0, l0, h1, m1, l1;
        split3_bf16(xq[i].x, xq[i].y, h0, m0, l0);
        split3_bf16(xq[i].z, xq[i].w, h1, m1, l1);
        uint8_t* b = sB + (k / kTcKB) * kBBytes;
        const int kin = k % kTcKB;
        *reinterpret_cast<uint2*>(b + tc::sw128_offset(t, kin)) = make_uint2(h0, h1);
        *reinterpret_cast<uint2*>(b + tc::sw128_offset(T + t, kin)) = make_uint2(m0, m1);
        *reinterpret_cast<uint2*>(b + tc::sw128_offset(2 * T + t, kin)) = make_uint2(l0, l1);
    }
    if (tid < T * 4) reinterpret_cast<float4*>(&m_s[0][0])[tid] = reinterpret_cast<const float4*>(Rmix)[tid];
    tc::fence_proxy_async_smem();
    __syncthreads();

    // 3. the MMAs, issued by one thread once the weights have landed
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
                                tc::desc_sw128(tc::smem_u32(sB + kb * kBBytes) + kk * 32), idesc,
                                (kb | kk) != 0);
            tc::mma_commit(&mma_done);
        }
        ok_s = ok;
    }
    __syncthreads();
    const bool ok = ok_s && tc_wait(&mma_done, 0, status);

    // 4. gate in place (warp = stream, lane = column), the streams meet in shared
    //    memory, then the mix and the three images
    if (ok) {
        tc::tc_fence_after();
        float u[32];
        tc::tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16), u);
#pragma unroll
        for (int t = 0; t < T; ++t)
            g_s[t][warp][lane] = gate_value((u[2 * T + t] + u[T + t]) + u[t], rp[t]);
    }
    tc::tc_fence_before();
    __syncthreads();
#pragma unroll
    for (int t = 0; t < T; ++t) {
        // a CTA whose wait gave up writes NaN, so that even a caller without a status
        // word (the allocation-free entry) finds no stale values in its outputs
        const float m = ok ? mix_row(&m_s[t][warp * 4], g_s[t][0][lane], g_s[t][1][lane],
                                     g_s[t][2][lane], g_s[t][3][lane])
                           : __int_as_float(0x7fc00000);
        const size_t off = (size_t)t * kCols + warp * kWidth + c;
        out_f32[off] = m;
        out_bf16[off] = to_bf16_bits(m);
        out_fp16[off] = to_fp16_bits(m);
    }
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTcTmemCols);
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

// The up kernel of every chunk is the tcgen05 one. Measured, µs per read with P, for
// T = 1..8: 6.13, 6.14, 6.67, 7.21, 7.94, 8.68, 9.63, 10.20, against 5.0, 6.1, 7.1,
// 7.9, 8.8, 9.7, 10.8, 12.2 with the CUDA-core up kernel it replaced. One kernel for
// every T keeps a token's bits independent of the other tokens of its call.

// Devices (bits) on which up_mix_tc_kernel<T> has been allowed its dynamic shared
// memory. hc_read_init clears a device's bits (decode_forget_smem), so the attribute
// is set again after a device reset.
std::atomic<unsigned long long> g_smem_set[kDecodeMaxT + 1];

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

template <int T>
cudaError_t allow_up_tc(int device) {
    return allow_smem(up_mix_tc_kernel<T>, kTcSmem, device, g_smem_set[T]);
}


template <int T>
cudaError_t launch_chunk(const Ctx& ctx, const ReadArgs& a, int t0, cudaStream_t st) {
    const size_t off = (size_t)t0 * kCols;
    const float* R = a.R + off;
    const float* P = a.P ? a.P + off : nullptr;
    float* lo = ctx.s.lo + (size_t)t0 * kRank;
    CUtensorMap tm_wu;
    if (!encode_w_up_bf16(&tm_wu, a.W_up, kTcCols)) return cudaErrorInvalidValue;
    cudaError_t e = allow_up_tc<T>(ctx.device);
    if (e != cudaSuccess) return e;
    e = launch_pdl(down_slice_kernel<T>, dim3(kDownSlices, kDownRowBlocks), dim3(kDownThreads), 0,
                   st, R, P, a.w_norm, a.W_down, lo, ctx.eps);
    if (e != cudaSuccess) return e;
    return launch_pdl(up_mix_tc_kernel<T>, dim3(kWidth / kTcCols), dim3(kTcThreads),
                      (size_t)kTcSmem, st, tm_wu, R, P, (const float*)lo,
                      a.Rmix + (size_t)t0 * 16, a.out_f32 + off, a.out_bf16 + off,
                      a.out_fp16 + off, ctx.s.status);
}

}  // namespace

void decode_forget_smem(int device) {
    if (device < 0 || device >= 64) return;
    for (auto& bits : g_smem_set) bits.fetch_and(~(1ull << device), std::memory_order_acq_rel);
}

namespace {
template <int T>
cudaError_t allow_chunk(int device) {
    return allow_up_tc<T>(device);
}
}  // namespace

cudaError_t decode_setup(int device) {
    decode_forget_smem(device);
    cudaError_t e = allow_chunk<1>(device);
    if (e == cudaSuccess) e = allow_chunk<2>(device);
    if (e == cudaSuccess) e = allow_chunk<3>(device);
    if (e == cudaSuccess) e = allow_chunk<4>(device);
    if (e == cudaSuccess) e = allow_chunk<5>(device);
    if (e == cudaSuccess) e = allow_chunk<6>(device);
    if (e == cudaSuccess) e = allow_chunk<7>(device);
    if (e == cudaSuccess) e = allow_chunk<8>(device);
    return e;
}

cudaError_t launch_decode(const Ctx& ctx, const ReadArgs& a, cudaStream_t st) {
    for (int t0 = 0; t0 < a.T; t0 += kDecodeMaxT) {
        const int n = a.T - t0 < kDecodeMaxT ? a.T - t0 : kDecodeMaxT;
        cudaError_t e;
        switch (n) {
            case 1: e = launch_chunk<1>(ctx, a, t0, st); break;
            case 2: e = launch_chunk<2>(ctx, a, t0, st); break;
            case 3: e = launch_chunk<3>(ctx, a, t0, st); break;
            case 4: e = launch_chunk<4>(ctx, a, t0, st); break;
            case 5: e = launch_chunk<5>(ctx, a, t0, st); break;
            case 6: e = launch_chunk<6>(ctx, a, t0, st); break;
            case 7: e = launch_chunk<7>(ctx, a, t0, st); break;
            default: e = launch_chunk<8>(ctx, a, t0, st); break;
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace hc
