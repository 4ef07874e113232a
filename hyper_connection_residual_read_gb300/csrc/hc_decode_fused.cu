// Decode read in one kernel: down projection, norm fold, lo exchange, up projection,
// gate and mix, for up to 8 tokens per launch.
//
// "#2226 STRATA_HC_PERSIST=1 (opt-in, HIP): the verifier's hyper-connection read as one
// persistent kernel", Summary: at 1-8 tokens the read is dominated by its launches
// and global dependencies, and runs faster as one kernel whose blocks split the down
// projection by column slices, reduce, then run the up projection. Here:
//
//  * 160 CTAs = 20 clusters of 8. CTA (slice sl, row block rb) owns 16 rows x 1280
//    columns of W_down (kept in registers) and 16 output columns x 4 streams of
//    W_up (copied into shared memory by the bulk-copy engine). Both weight streams
//    are issued before the programmatic-dependent-launch wait, so they overlap the
//    previous kernel on the stream.
//  * The norm is folded into the down projection ("#2488 sycl/A770: faster
//    hyper-connection read on Arc A-series", Summary, change 4) and the 8 slices of
//    a row block reduce through distributed shared memory in a fixed order (the
//    page's change 1 does it with the last slice to finish).
//  * Each CTA publishes its 2 rows of lo with a release-add on a counter; every CTA
//    waits, bounded by %globaltimer, until all 160 have published, then reads lo and
//    runs its up projection, gate and 4x4 mix. The last CTA to read lo resets the
//    counters for the next call.
//
// All CTAs are resident before any of them waits: a dependent launch cannot start
// until every CTA of this grid has issued launch_dependents, and the previous
// kernel on the stream finishes on its own. A wait that still runs out of time
// (after the context's bound, 2 s unless a test shortened it) records a timeout in
// the device status word and the CTA goes on without lo; the exchange counters may
// then be left mid-count, and hc_read_status, which reports the timeout, resets them.
#include <cooperative_groups.h>

#include "hc_common.cuh"
#include "hc_internal.h"

namespace hc {

namespace {

constexpr int kThreads = 320;              // 10 warps
constexpr int kColGroups = 5;              // down: 5 x 256 columns = 1280
constexpr int kClusters = kDownRowBlocks;  // 20
constexpr int kCtas = kDownSlices * kDownRowBlocks;   // 160
constexpr int kUpColsPerCta = kWidth / kCtas;         // 16
constexpr int kParts = 16;                 // up: 16 lanes per column, 20 inputs each
constexpr int kPartLen = kRank / kParts;   // 20
constexpr uint64_t kWaitNs = 2000000000ull;   // bound of the bulk-copy wait
constexpr int kWupBytes = kStreams * kUpColsPerCta * kRank * 2;   // 40 KB

constexpr int dyn_smem(int T) { return kWupBytes + T * kDownSliceCols * 4 + T * kRank * 4; }

__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t ld_acquire(const unsigned* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

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
__global__ void __cluster_dims__(kDownSlices, 1, 1) __launch_bounds__(kThreads, 2)
decode_fused_kernel(const float* R, const float* P, const uint16_t* __restrict__ w_norm,
                    const uint16_t* __restrict__ W_down, const uint16_t* __restrict__ W_up,
                    const float* Rmix, float* out_f32, uint16_t* out_bf16, uint16_t* out_fp16,
                    float* lo, unsigned* sync, float eps, int* status, uint64_t lo_wait_ns) {
    namespace cg = cooperative_groups;
    const int sl = blockIdx.x, rb = blockIdx.y;
    const int cid = rb * kDownSlices + sl;                 // 0..159
    const int s = sl >> 1;
    const int c0 = (sl & 1) * kDownSliceCols;
    const int k0 = s * kWidth + c0;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rg = warp / kColGroups, cgp = warp % kColGroups;
    const int j0 = rb * kDownRowsPerCta + rg * 8;
    const int col = cgp * 256 + lane * 8;
    const int cbase = cid * kUpColsPerCta;                 // first output column of this CTA

    // dynamic shared memory: W_up rows (40 KB), a = R' * w_norm, lo
    extern __shared__ __align__(16) uint8_t dsm[];
    auto wup_s = reinterpret_cast<uint16_t (*)[kUpColsPerCta][kRank]>(dsm);
    auto a_s = reinterpret_cast<float4 (*)[kDownSliceCols / 4]>(dsm + kWupBytes);
    auto lo_s = reinterpret_cast<float (*)[kRank]>(dsm + kWupBytes + T * kDownSliceCols * 4);
    __shared__ float red_ss[kThreads / 32][T];
    __shared__ float red[T][kColGroups][kDownRowsPerCta];
    __shared__ float part_s[T][kDownRowsPerCta];
    __shared__ float ss_s[T];
    __shared__ __align__(16) float m_s[T][16];
    __shared__ __align__(8) uint64_t wbar;
    __shared__ int s_ok;

    // 1. weight streams: W_up rows of this CTA's columns into shared memory by bulk
    //    copy (4 contiguous runs of 16 rows), W_down into registers
    const uint32_t wbar_a = static_cast<uint32_t>(__cvta_generic_to_shared(&wbar));
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(wbar_a));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(wbar_a),
                     "r"((uint32_t)kWupBytes)
                     : "memory");
#pragma unroll
        for (int st = 0; st < kStreams; ++st) {
            const size_t wi = (size_t)(st * kWidth + cbase) * kRank;
            const uint16_t* src = W_up + wi;
            const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(&wup_s[st][0][0]));
            if (HC_IN_RANGE(wi, kUpColsPerCta * kRank, (size_t)kCols * kRank, status)) {
                asm volatile(
                    "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
                        "r"(dst), "l"(src), "r"((uint32_t)(kUpColsPerCta * kRank * 2)), "r"(wbar_a)
                    : "memory");
            } else {
                // the copy is skipped: its bytes still count, so the wait below ends
                asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(wbar_a),
                             "r"((uint32_t)(kUpColsPerCta * kRank * 2))
                             : "memory");
            }
        }
    }
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
    pdl_launch_dependents();
    pdl_wait();

    // 2. activations a = R' * w_norm and the slice's sums of squares
    float4 xs[T];
#pragma unroll
    for (int t = 0; t < T; ++t)
        xs[t] = HC_IN_RANGE((size_t)t * kCols + k0 + 4 * tid, 4, (size_t)T * kCols, status)
                    ? *reinterpret_cast<const float4*>(R + (size_t)t * kCols + k0 + 4 * tid)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
    if (P != nullptr) {
#pragma unroll
        for (int t = 0; t < T; ++t) {
            if (!HC_IN_RANGE((size_t)t * kCols + k0 + 4 * tid, 4, (size_t)T * kCols, status)) continue;
            const float4 p = *reinterpret_cast<const float4*>(P + (size_t)t * kCols + k0 + 4 * tid);
            xs[t].x += p.x; xs[t].y += p.y; xs[t].z += p.z; xs[t].w += p.w;
        }
    }
    const float w0 = bf16_lo(wn.x), w1 = bf16_hi(wn.x), w2 = bf16_lo(wn.y), w3 = bf16_hi(wn.y);
    {
        const int c = 4 * tid;
        const int scg = c >> 8, slane = (c & 255) >> 3, half = (c & 7) >> 2;
        const int slot = scg * 64 + half * 32 + slane;
#pragma unroll
        for (int t = 0; t < T; ++t) {
            const float4 x = xs[t];
            float ss = x.x * x.x;
            ss = fmaf(x.y, x.y, ss);
            ss = fmaf(x.z, x.z, ss);
            ss = fmaf(x.w, x.w, ss);
            a_s[t][slot] = make_float4(x.x * w0, x.y * w1, x.z * w2, x.w * w3);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            if (lane == 0) red_ss[warp][t] = ss;
        }
    }
    __syncthreads();
    if (tid < T) {
        float ss = 0.f;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) ss += red_ss[w][tid];
        ss_s[tid] = ss;
    }

    // 3. partial dots: 8 rows x this lane's 8 columns, reduced over the warp
    {
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
    }
    __syncthreads();
    if (tid < T * kDownRowsPerCta) {
        const int t = tid / kDownRowsPerCta, j = tid % kDownRowsPerCta;
        float v = red[t][0][j];
#pragma unroll
        for (int g = 1; g < kColGroups; ++g) v += red[t][g][j];
        part_s[t][j] = v;
    }

    // 4. reduce over the cluster's 8 slices (distributed shared memory), publish lo
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    if (tid < T * 2) {
        const int t = tid >> 1, j = 2 * sl + (tid & 1);
        // all 16 remote loads first, then the arithmetic (each is a round trip)
        float ssv[kDownSlices], pv[kDownSlices];
#pragma unroll
        for (int r = 0; r < kDownSlices; ++r) {
            ssv[r] = *cluster.map_shared_rank(&ss_s[t], r);
            pv[r] = *cluster.map_shared_rank(&part_s[t][j], r);
        }
        float v = 0.f;
#pragma unroll
        for (int st = 0; st < kStreams; ++st) {
            const float ss = ssv[2 * st] + ssv[2 * st + 1];
            const float rs = inv_rms(fmaf(ss, 1.0f / (float)kWidth, eps));
            const float d = pv[2 * st] + pv[2 * st + 1];
            v = fmaf(rs, d, v);
        }
        if (HC_IN_RANGE(t * kRank + rb * kDownRowsPerCta + j, 1, T * kRank, status))
            lo[t * kRank + rb * kDownRowsPerCta + j] = v;
    }
    // publish this CTA's rows: the CTA barrier orders the stores before thread 0's
    // release-add at GPU scope. (No CTA leaves before every CTA has published, so the
    // shared memory read above stays alive without a second cluster barrier.)
    __syncthreads();
    if (tid == 0)
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&sync[0]) : "memory");
    // the gate needs R' of this lane's (token, stream, column): load it before waiting
    const int up_cl = (warp & 7) * 2 + (lane >> 4), up_sp = (lane & 15) & 3;
    float rp[T];
#pragma unroll
    for (int t = 0; t < T; ++t) {
        const size_t off = (size_t)t * kCols + up_sp * kWidth + cbase + up_cl;
        const bool in = HC_IN_RANGE(off, 1, (size_t)T * kCols, status);
        rp[t] = in ? R[off] : 0.f;
        if (P != nullptr && in) rp[t] += P[off];
    }

    // 5. wait for every cluster's lo, then read it with R' and the mix
    if (tid == 0) {
        int ok = 1;
        if (ld_acquire(&sync[0]) < (unsigned)kCtas) {
            const uint64_t t0 = gtimer();
            while (ld_acquire(&sync[0]) < (unsigned)kCtas) {
                if (gtimer() - t0 > lo_wait_ns) {
                    atomicOr(status, kStatusTimeout);
                    ok = 0;
                    break;
                }
            }
        }
        s_ok = ok;
    }
    __syncthreads();
    for (int e = tid; e < T * kRank / 4; e += kThreads) {
        const float4 v = HC_IN_RANGE(4 * (size_t)e, 4, (size_t)T * kRank, status)
                             ? __ldcg(reinterpret_cast<const float4*>(lo) + e)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
        reinterpret_cast<float4*>(&lo_s[0][0])[e] = v;
    }
    if (tid < T * 4 && HC_IN_RANGE(4 * (size_t)tid, 4, (size_t)T * 16, status))
        reinterpret_cast<float4*>(&m_s[0][0])[tid] = reinterpret_cast<const float4*>(Rmix)[tid];
    __syncthreads();
    // the last CTA to have read lo resets the counters for the next call
    if (tid == 0) {
        if (atomicAdd(&sync[1], 1u) == (unsigned)(kCtas - 1)) {
            sync[1] = 0u;
            sync[0] = 0u;
        }
    }

    // 6. up projection of 16 columns x 4 streams: warp w (0..7) owns 2 columns, 16
    //    lanes per column, each summing 20 of the 320 inputs for all 4 stream rows
    if (warp < 8) {
        // W_up in shared memory (bounded wait)
        uint32_t done = 0;
        const uint64_t t0 = gtimer();
        while (true) {
            asm volatile(
                "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0; "
                "selp.u32 %0, 1, 0, p; }"
                : "=r"(done)
                : "r"(wbar_a)
                : "memory");
            if (done) break;
            if (gtimer() - t0 > kWaitNs) {
                atomicOr(status, kStatusTimeout);
                break;
            }
        }
        const int cc = lane >> 4, part = lane & 15;
        const int cl = warp * 2 + cc;                        // column within the CTA
        const int c = cbase + cl;
        const int sp = part & 3;
        uint2 wr[kStreams][5];                               // 20 bf16 per stream row
#pragma unroll
        for (int st = 0; st < kStreams; ++st) {
            const uint2* src = reinterpret_cast<const uint2*>(&wup_s[st][cl][part * kPartLen]);
#pragma unroll
            for (int i = 0; i < 5; ++i) wr[st][i] = src[i];
        }
#pragma unroll
        for (int t = 0; t < T; ++t) {
            const float4* l4 = reinterpret_cast<const float4*>(&lo_s[t][part * kPartLen]);
            float acc[kStreams] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < 5; ++i) {
                const float4 x = l4[i];
#pragma unroll
                for (int st = 0; st < kStreams; ++st) {
                    const uint2 w = wr[st][i];
                    float v = acc[st];
                    v = fmaf(bf16_lo(w.x), x.x, v);
                    v = fmaf(bf16_hi(w.x), x.y, v);
                    v = fmaf(bf16_lo(w.y), x.z, v);
                    v = fmaf(bf16_hi(w.y), x.w, v);
                    acc[st] = v;
                }
            }
#pragma unroll
            for (int st = 0; st < kStreams; ++st) {
                acc[st] += __shfl_xor_sync(0xffffffffu, acc[st], 8);
                acc[st] += __shfl_xor_sync(0xffffffffu, acc[st], 4);
                acc[st] += __shfl_xor_sync(0xffffffffu, acc[st], 2);
                acc[st] += __shfl_xor_sync(0xffffffffu, acc[st], 1);
            }
            const float u = sp == 0 ? acc[0] : sp == 1 ? acc[1] : sp == 2 ? acc[2] : acc[3];
            const float g = gate_value(u, rp[t]);
            const int base = lane & ~15;
            const float g0 = __shfl_sync(0xffffffffu, g, base + 0);
            const float g1 = __shfl_sync(0xffffffffu, g, base + 1);
            const float g2 = __shfl_sync(0xffffffffu, g, base + 2);
            const float g3 = __shfl_sync(0xffffffffu, g, base + 3);
            if (part < 4) {
                const float m = mix_row(&m_s[t][part * 4], g0, g1, g2, g3);
                const size_t off = (size_t)t * kCols + part * kWidth + c;
                if (HC_IN_RANGE(off, 1, (size_t)T * kCols, status)) {
                    out_f32[off] = m;
                    out_bf16[off] = to_bf16_bits(m);
                    out_fp16[off] = to_fp16_bits(m);
                }
            }
        }
    }
    // no CTA leaves while a cluster peer might still read its shared memory (only
    // possible on the timeout path; in the normal path every read is long done)
    cluster.sync();
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, int smem, cudaStream_t st,
                       Args... args) {
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

template <int T>
cudaError_t launch_fused_chunk(const Ctx& ctx, const ReadArgs& a, int t0, cudaStream_t st) {
    const size_t off = (size_t)t0 * kCols;
    return launch_pdl(decode_fused_kernel<T>, dim3(kDownSlices, kDownRowBlocks), dim3(kThreads),
                      dyn_smem(T), st, a.R + off, a.P ? a.P + off : nullptr, a.w_norm, a.W_down, a.W_up,
                      a.Rmix + (size_t)t0 * 16, a.out_f32 + off, a.out_bf16 + off,
                      a.out_fp16 + off, ctx.s.lo + (size_t)t0 * kRank, ctx.s.sync, ctx.eps,
                      ctx.s.status, ctx.lo_wait_ns);
}

template <int T>
cudaError_t set_smem() {
    return cudaFuncSetAttribute(decode_fused_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                dyn_smem(T));
}

}  // namespace

cudaError_t decode_fused_setup(bool* usable) {
    cudaError_t e = cudaSuccess;
    *usable = false;
    if ((e = set_smem<1>()) || (e = set_smem<2>()) || (e = set_smem<3>()) || (e = set_smem<4>()) ||
        (e = set_smem<5>()) || (e = set_smem<6>()) || (e = set_smem<7>()) || (e = set_smem<8>()))
        return e;
    // every cluster of the grid must be resident at once (the CTAs wait on each other);
    // otherwise the read keeps the two-kernel decode path
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kDownSlices, kDownRowBlocks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = dyn_smem(kDecodeMaxT);
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, decode_fused_kernel<kDecodeMaxT>, &cfg);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return cudaSuccess;
    }
    *usable = clusters >= kClusters;
    return cudaSuccess;
}

cudaError_t launch_decode_fused(const Ctx& ctx, const ReadArgs& a, cudaStream_t st) {
    for (int t0 = 0; t0 < a.T; t0 += kDecodeMaxT) {
        const int n = a.T - t0 < kDecodeMaxT ? a.T - t0 : kDecodeMaxT;
        cudaError_t e;
        switch (n) {
            case 1: e = launch_fused_chunk<1>(ctx, a, t0, st); break;
            case 2: e = launch_fused_chunk<2>(ctx, a, t0, st); break;
            case 3: e = launch_fused_chunk<3>(ctx, a, t0, st); break;
            case 4: e = launch_fused_chunk<4>(ctx, a, t0, st); break;
            case 5: e = launch_fused_chunk<5>(ctx, a, t0, st); break;
            case 6: e = launch_fused_chunk<6>(ctx, a, t0, st); break;
            case 7: e = launch_fused_chunk<7>(ctx, a, t0, st); break;
            default: e = launch_fused_chunk<8>(ctx, a, t0, st); break;
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace hc
