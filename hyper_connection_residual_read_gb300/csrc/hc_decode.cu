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
//      cluster and reduce through distributed shared memory in a fixed order
//      (the page's change 1 does it with the last slice to finish; a cluster
//      needs no global counter), so the result is bitwise repeatable.
//
//  up_mix_kernel - a warp owns 4 output columns; 8 lanes per column each sum 40
//      of the 320 inputs for all 4 up rows i = s*2560 + c of that column, an xor
//      tree finishes the dots, then the gate and the 4x4 mix run in registers
//      ("#1370 prefill: opt-in STRATA_HC_UPMIX=1 on CUDA ...", "What it does":
//      the mix in registers, writing mixed with its BF16 / FP16 images).
//
// Weights are loaded straight into registers with 16-byte streaming loads issued
// before anything else, so a kernel's whole weight matrix is in flight at once.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "hc_common.cuh"
#include "hc_internal.h"

namespace hc {

namespace {

constexpr int kDownThreads = 320;   // 10 warps, 128 columns of the slice each
constexpr int kUpThreads = 256;     // 8 warps: 4 M tiles x 2 K halves
constexpr int kUpColsPerCta = 16;   // 2560 columns over 160 CTAs
constexpr int kUpRows = kStreams * kUpColsPerCta;   // 64 W_up rows per CTA
constexpr int kAStride = kDownSliceCols + 16;       // floats per token row of a (bank spread)
constexpr int kWStride = kRank + 8;                 // bf16 per W_up row in shared memory
constexpr int kLStride = kRank + 8;                 // bf16 per token row of a lo term
constexpr int kUpSmem = kUpRows * kWStride * 2 + 3 * 8 * kLStride * 2;   // 57,728 B
constexpr uint64_t kWaitNs = 2000000000ull;

__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// mma.sync m16n8k16, bf16 inputs, fp32 accumulation: D += A (16x16) * B (16x8).
// Fragments (g = lane / 4, q = lane % 4): a0 = A[g][2q..2q+1], a1 = A[g+8][2q..],
// a2 = A[g][2q+8..], a3 = A[g+8][2q+8..]; b0 = B[2q..2q+1][g], b1 = B[2q+8..2q+9][g];
// d0 = D[g][2q], d1 = D[g][2q+1], d2 = D[g+8][2q], d3 = D[g+8][2q+1].
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// x = hi + mid + lo with each term bf16 (round to nearest): 24 bits of x, so a
// product with an exact bf16 weight loses nothing before the fp32 sum.
__device__ __forceinline__ void split3(float x0, float x1, uint32_t (&t)[3]) {
    float r0 = x0, r1 = x1;
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(r0, r1);
        t[i] = *reinterpret_cast<const uint32_t*>(&h);
        r0 -= __low2float(h);
        r1 -= __high2float(h);
    }
}

template <int T>
__global__ void __cluster_dims__(kDownSlices, 1, 1) __launch_bounds__(kDownThreads, 2)
down_slice_kernel(const float* __restrict__ R, const float* __restrict__ P,
                  const uint16_t* __restrict__ w_norm, const uint16_t* __restrict__ W_down,
                  float* __restrict__ lo, float eps) {
    namespace cg = cooperative_groups;
    const int sl = blockIdx.x;                 // K slice 0..7 == rank in the cluster
    const int rb = blockIdx.y;                 // row block 0..19 == the cluster
    const int s = sl >> 1;                     // stream of the slice
    const int c0 = (sl & 1) * kDownSliceCols;  // first column of the slice in the stream
    const int k0 = s * kWidth + c0;            // first column on the 10240 axis
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, q = lane & 3;

    __shared__ __align__(16) float a_s[T][kAStride];
    __shared__ float red_ss[kDownThreads / 32][T];
    __shared__ float dred[kDownThreads / 32][kDownRowsPerCta][8];
    __shared__ float part_s[T][kDownRowsPerCta];   // this slice's partial dots
    __shared__ float ss_s[T];                      // this slice's sums of squares

    // 1. weights first (layer parameters may be read before the previous kernel on
    //    the stream has finished): the tensor-core A fragments of this warp's 128
    //    columns, 8 k-steps x rows (g, g+8). The 16 K values of a step are taken in
    //    the order that gives each thread 4 consecutive columns (8-byte loads); the
    //    activations use the same order.
    uint2 wa[8][2];
    {
        const uint16_t* r0 = W_down + (size_t)(rb * kDownRowsPerCta + g) * kCols + k0 + warp * 128 + 4 * q;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            wa[kk][0] = __ldg(reinterpret_cast<const uint2*>(r0 + kk * 16));
            wa[kk][1] = __ldg(reinterpret_cast<const uint2*>(r0 + 8 * (size_t)kCols + kk * 16));
        }
    }
    const uint2 wn = *reinterpret_cast<const uint2*>(w_norm + k0 + 4 * tid);
    pdl_launch_dependents();
    pdl_wait();

    // 2. activations a = R' * w_norm (fp32) and per-token sums of squares of R'
    {
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
#pragma unroll
        for (int t = 0; t < T; ++t) {
            const float4 x = xs[t];
            float ss = x.x * x.x;
            ss = fmaf(x.y, x.y, ss);
            ss = fmaf(x.z, x.z, ss);
            ss = fmaf(x.w, x.w, ss);
            *reinterpret_cast<float4*>(&a_s[t][4 * tid]) =
                make_float4(x.x * w0, x.y * w1, x.z * w2, x.w * w3);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            if (lane == 0) red_ss[warp][t] = ss;
        }
    }
    __syncthreads();
    if (tid < T) {
        float ss = 0.f;
#pragma unroll
        for (int w = 0; w < kDownThreads / 32; ++w) ss += red_ss[w][tid];
        ss_s[tid] = ss;
    }

    // 3. partial dots on the tensor cores: D[16 rows][8 tokens] over this warp's 128
    //    columns; B = a split into 3 bf16 terms (token g; tokens >= T are zero), one
    //    accumulator per term so the three MMA chains are independent
    {
        float dt[3][4] = {};
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (g < T) x = *reinterpret_cast<const float4*>(&a_s[g < T ? g : 0][warp * 128 + kk * 16 + 4 * q]);
            uint32_t b0[3], b1[3];
            split3(x.x, x.y, b0);
            split3(x.z, x.w, b1);
            const uint32_t a0 = wa[kk][0].x, a2 = wa[kk][0].y, a1 = wa[kk][1].x, a3 = wa[kk][1].y;
#pragma unroll
            for (int term = 0; term < 3; ++term) mma_bf16(dt[term], a0, a1, a2, a3, b0[term], b1[term]);
        }
        dred[warp][g][2 * q] = (dt[0][0] + dt[1][0]) + dt[2][0];
        dred[warp][g][2 * q + 1] = (dt[0][1] + dt[1][1]) + dt[2][1];
        dred[warp][g + 8][2 * q] = (dt[0][2] + dt[1][2]) + dt[2][2];
        dred[warp][g + 8][2 * q + 1] = (dt[0][3] + dt[1][3]) + dt[2][3];
    }
    __syncthreads();

    // 4. this slice's partial for its 16 rows, the 10 warps summed in order
    if (tid < T * kDownRowsPerCta) {
        const int t = tid / kDownRowsPerCta, j = tid % kDownRowsPerCta;
        float v = dred[0][j][t];
#pragma unroll
        for (int w = 1; w < kDownThreads / 32; ++w) v += dred[w][j][t];
        part_s[t][j] = v;
    }

    // 5. reduce over the 8 slices of the row block through distributed shared
    //    memory: CTA `sl` finishes rows 2*sl and 2*sl+1 of the block, summing the
    //    slices of each stream in order and applying that stream's rs.
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
            const float rs = 1.0f / sqrtf(ss / (float)kWidth + eps);
            const float d = pv[2 * st] + pv[2 * st + 1];
            v = fmaf(rs, d, v);
        }
        lo[t * kRank + rb * kDownRowsPerCta + j] = v;
    }
    cluster.sync();   // keep this CTA's shared memory alive until every reader is done
}

template <int T>
__global__ void __launch_bounds__(kUpThreads)
up_mix_kernel(const float* __restrict__ R, const float* __restrict__ P,
              const uint16_t* __restrict__ W_up, const float* __restrict__ lo,
              const float* __restrict__ Rmix, float* __restrict__ out_f32,
              uint16_t* __restrict__ out_bf16, uint16_t* __restrict__ out_fp16,
              int* __restrict__ status) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, q = lane & 3;
    const int cbase = blockIdx.x * kUpColsPerCta;   // first output column of this CTA

    // dynamic shared memory: the 64 W_up rows (padded; shared row 4 * column + stream,
    // so the 16 rows of an M tile are consecutive) and the 3 bf16 terms of lo
    extern __shared__ __align__(16) uint8_t dsm[];
    uint16_t* wup_s = reinterpret_cast<uint16_t*>(dsm);
    uint16_t* lob_s = reinterpret_cast<uint16_t*>(dsm + kUpRows * kWStride * 2);
    __shared__ __align__(16) float m_s[T][16];
    __shared__ float ured[4][32][4];
    __shared__ __align__(8) uint64_t wbar;

    // 1. W_up rows by the bulk-copy engine (layer parameters: before the wait)
    const uint32_t wbar_a = static_cast<uint32_t>(__cvta_generic_to_shared(&wbar));
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(wbar_a));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(wbar_a),
                     "r"((uint32_t)(kUpRows * kRank * 2))
                     : "memory");
    }
    __syncthreads();
    if (warp == 0) {
        for (int r = lane; r < kUpRows; r += 32) {
            const int st = r / kUpColsPerCta, cl = r % kUpColsPerCta;
            const uint16_t* src = W_up + (size_t)(st * kWidth + cbase + cl) * kRank;
            const uint32_t dst = static_cast<uint32_t>(
                __cvta_generic_to_shared(wup_s + (cl * kStreams + st) * kWStride));
            asm volatile(
                "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
                    "r"(dst), "l"(src), "r"((uint32_t)(kRank * 2)), "r"(wbar_a)
                : "memory");
        }
    }
    pdl_launch_dependents();
    pdl_wait();

    // warp w owns M tile mt = w / 2 (columns 4mt..4mt+3 of the CTA; tile row
    // m = 4 * column + stream) and K half kh = w % 2. Thread rows g and g+8 of the
    // tile: stream g % 4, columns 4mt + g/4 and 4mt + 2 + g/4.
    const int mt = warp >> 1, kh = warp & 1;
    const int us = g & 3, ucA = 4 * mt + (g >> 2), ucB = ucA + 2;
    // 2. R' for the gate at (tokens 2q and 2q+1, stream us, columns ucA and ucB)
    float rp[2][2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int t = 2 * q + i;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            float v = 0.f;
            if (t < T) {
                const size_t off = (size_t)t * kCols + us * kWidth + cbase + (cc ? ucB : ucA);
                v = R[off];
                if (P != nullptr) v += P[off];
            }
            rp[i][cc] = v;
        }
    }
    // lo as 3 bf16 terms (tokens >= T are zero) and the mix matrices
    for (int e = tid; e < 8 * kRank / 2; e += kUpThreads) {
        const int t = e / (kRank / 2), k = 2 * (e % (kRank / 2));
        float2 v = make_float2(0.f, 0.f);
        if (t < T) v = *reinterpret_cast<const float2*>(lo + t * kRank + k);
        uint32_t terms[3];
        split3(v.x, v.y, terms);
#pragma unroll
        for (int term = 0; term < 3; ++term)
            *reinterpret_cast<uint32_t*>(lob_s + (term * 8 + t) * kLStride + k) = terms[term];
    }
    if (tid < T * 4) reinterpret_cast<float4*>(&m_s[0][0])[tid] = reinterpret_cast<const float4*>(Rmix)[tid];
    __syncthreads();

    // 3. the W_up rows must have arrived (bounded wait)
    {
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
    }

    // 4. u = W_up . lo on the tensor cores over this warp's K half (10 k-steps), A by
    //    ldmatrix from the W_up rows, B = the lo terms; one accumulator per term
    float d[4];
    {
        const uint32_t arow = static_cast<uint32_t>(__cvta_generic_to_shared(
            wup_s + (16 * mt + (lane & 15)) * kWStride + (lane >> 4) * 8));
        float dt[3][4] = {};
#pragma unroll
        for (int ks = 0; ks < 10; ++ks) {
            const int kb = kh * 160 + ks * 16;
            uint32_t a0, a1, a2, a3;
            asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                         : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                         : "r"(arow + kb * 2));
#pragma unroll
            for (int term = 0; term < 3; ++term) {
                const uint16_t* bt = lob_s + (term * 8 + g) * kLStride + kb + 2 * q;
                const uint32_t b0 = *reinterpret_cast<const uint32_t*>(bt);
                const uint32_t b1 = *reinterpret_cast<const uint32_t*>(bt + 8);
                mma_bf16(dt[term], a0, a1, a2, a3, b0, b1);
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) d[i] = (dt[0][i] + dt[1][i]) + dt[2][i];
    }
    // the two K halves of an M tile, in order (half 0 + half 1)
    if (kh == 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) ured[mt][lane][i] = d[i];
    }
    __syncthreads();
    if (kh == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) d[i] += ured[mt][lane][i];
        // 5. gate, then mix across the 4 stream lanes of a column (lane stride 4)
        float gv[2][2];
        gv[0][0] = gate_value(d[0], rp[0][0]);   // token 2q,   column A
        gv[1][0] = gate_value(d[1], rp[1][0]);   // token 2q+1, column A
        gv[0][1] = gate_value(d[2], rp[0][1]);   // token 2q,   column B
        gv[1][1] = gate_value(d[3], rp[1][1]);   // token 2q+1, column B
        const int base = (lane & ~15) | q;       // lane of stream 0 for this (column, q)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const float g0 = __shfl_sync(0xffffffffu, gv[i][cc], base);
                const float g1 = __shfl_sync(0xffffffffu, gv[i][cc], base + 4);
                const float g2 = __shfl_sync(0xffffffffu, gv[i][cc], base + 8);
                const float g3 = __shfl_sync(0xffffffffu, gv[i][cc], base + 12);
                const int t = 2 * q + i;
                if (t < T) {
                    const float m = mix_row(&m_s[t][us * 4], g0, g1, g2, g3);
                    const size_t off = (size_t)t * kCols + us * kWidth + cbase + (cc ? ucB : ucA);
                    out_f32[off] = m;
                    out_bf16[off] = to_bf16_bits(m);
                    out_fp16[off] = to_fp16_bits(m);
                }
            }
        }
    }
}

// Launch with programmatic stream serialisation (see pdl_wait).
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

// The up kernel's dynamic shared memory size is set once per device and T.
template <int T>
cudaError_t ensure_attrs() {
    static bool done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (done[dev]) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(up_mix_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kUpSmem);
    if (e == cudaSuccess) done[dev] = true;
    return e;
}

template <int T>
cudaError_t launch_chunk(const Ctx& ctx, const ReadArgs& a, int t0, cudaStream_t st) {
    cudaError_t e = ensure_attrs<T>();
    if (e != cudaSuccess) return e;
    const size_t off = (size_t)t0 * kCols;
    const float* R = a.R + off;
    const float* P = a.P ? a.P + off : nullptr;
    float* lo = ctx.s.lo + (size_t)t0 * kRank;
    e = launch_pdl(down_slice_kernel<T>, dim3(kDownSlices, kDownRowBlocks), dim3(kDownThreads), 0,
                   st, R, P, a.w_norm, a.W_down, lo, ctx.eps);
    if (e != cudaSuccess) return e;
    return launch_pdl(up_mix_kernel<T>, dim3(kWidth / kUpColsPerCta), dim3(kUpThreads), kUpSmem, st,
                      R, P, a.W_up, (const float*)lo, a.Rmix + (size_t)t0 * 16, a.out_f32 + off,
                      a.out_bf16 + off, a.out_fp16 + off, ctx.s.status);
}

}  // namespace

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
