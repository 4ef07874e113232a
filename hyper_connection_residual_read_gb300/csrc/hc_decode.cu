// Decode path of the hyper-connection read: 1-8 tokens per launch, bound by the
// 13 MB of bf16 weights every read streams.
//
// Two kernels per chunk of up to 8 tokens:
//
//  down_slice_kernel  - the down projection split into K slices (half a stream,
//      1280 columns) x row blocks (16 of the 320 rows). The norm is folded in
//      ("#2488 sycl/A770: faster hyper-connection read on Arc A-series",
//      Summary, change 4): a slice stages R' * w_norm unscaled together with its
//      per-token sum of squares, and the reduce applies each stream's rs to that
//      stream's partial dots. The last slice of a row block to finish sums the
//      slice partials in a fixed order (same page, change 1), so the result is
//      bitwise repeatable and there is no separate reduce launch.
//
//  up_mix_kernel - one warp per output column c: 8 lanes per up row
//      i = s*2560 + c (one row per stream), lane sums over 40 of the 320 inputs,
//      an xor tree in the 8-lane group, then the gate and the 4x4 mix in
//      registers ("#1370 prefill: opt-in STRATA_HC_UPMIX=1 on CUDA ...", "What
//      it does": the mix runs in registers and writes mixed with its BF16 / FP16
//      images).
//
// Weights are loaded straight into registers with 16-byte streaming loads that
// are issued before anything else, so the whole matrix is in flight at once.
#include "hc_common.cuh"
#include "hc_internal.h"

namespace hc {

namespace {

constexpr int kDownThreads = 320;   // 10 warps: 2 row groups x 5 column groups
constexpr int kDownColGroups = 5;   // 5 x 256 columns = 1280
constexpr int kUpColsPerCta = 8;    // one warp per column
constexpr int kUpThreads = 32 * kUpColsPerCta;

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
__global__ void __launch_bounds__(kDownThreads)
down_slice_kernel(const float* __restrict__ R, const float* __restrict__ P,
                  const uint16_t* __restrict__ w_norm, const uint16_t* __restrict__ W_down,
                  float* __restrict__ partials, float* __restrict__ ssq,
                  unsigned* __restrict__ counters, float* __restrict__ lo, float eps) {
    const int sl = blockIdx.x;                 // K slice 0..7
    const int rb = blockIdx.y;                 // row block 0..19
    const int s = sl >> 1;                     // stream of the slice
    const int c0 = (sl & 1) * kDownSliceCols;  // first column of the slice in the stream
    const int k0 = s * kWidth + c0;            // first column on the 10240 axis
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int rg = warp / kDownColGroups, cg = warp % kDownColGroups;
    const int j0 = rb * kDownRowsPerCta + rg * 8;
    const int col = cg * 256 + lane * 8;       // this lane's 8 columns within the slice

    // 1. weights first: 8 rows x 8 columns, one 16-byte load per row
    uint4 wv[8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
        wv[r] = ldg_stream_v4(W_down + (size_t)(j0 + r) * kCols + k0 + col);

    // 2. activations a = R' * w_norm (fp32) and per-token sums of squares of R'
    __shared__ float4 a_s[T][kDownSliceCols / 4];
    __shared__ float red_ss[kDownThreads / 32][T];
    __shared__ float red[T][kDownColGroups][kDownRowsPerCta];
    __shared__ int s_last;

    const uint2 wn = *reinterpret_cast<const uint2*>(w_norm + k0 + 4 * tid);
    const float w0 = bf16_lo(wn.x), w1 = bf16_hi(wn.x), w2 = bf16_lo(wn.y), w3 = bf16_hi(wn.y);
#pragma unroll
    for (int t = 0; t < T; ++t) {
        const size_t off = (size_t)t * kCols + k0 + 4 * tid;
        float4 x = *reinterpret_cast<const float4*>(R + off);
        if (P != nullptr) {
            const float4 p = *reinterpret_cast<const float4*>(P + off);
            x.x += p.x; x.y += p.y; x.z += p.z; x.w += p.w;
        }
        float ss = x.x * x.x;
        ss = fmaf(x.y, x.y, ss);
        ss = fmaf(x.z, x.z, ss);
        ss = fmaf(x.w, x.w, ss);
        a_s[t][tid] = make_float4(x.x * w0, x.y * w1, x.z * w2, x.w * w3);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) red_ss[warp][t] = ss;
    }
    __syncthreads();
    if (tid < T) {
        float ss = 0.f;
#pragma unroll
        for (int w = 0; w < kDownThreads / 32; ++w) ss += red_ss[w][tid];
        ssq[(rb * kDownSlices + sl) * kDecodeMaxT + tid] = ss;
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
        const float4 x0 = a_s[t][col / 4];
        const float4 x1 = a_s[t][col / 4 + 1];
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
        if ((lane & 3) == 0) red[t][cg][rg * 8 + ((lane >> 2) & 7)] = sum;
    }
    __syncthreads();

    // 4. this slice's partial for its 16 rows, column groups summed in order
    if (tid < T * kDownRowsPerCta) {
        const int t = tid / kDownRowsPerCta, j = tid % kDownRowsPerCta;
        float v = red[t][0][j];
#pragma unroll
        for (int g = 1; g < kDownColGroups; ++g) v += red[t][g][j];
        partials[(sl * kDecodeMaxT + t) * kRank + rb * kDownRowsPerCta + j] = v;
    }

    // 5. the last slice of this row block to arrive reduces (no waiting)
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(&counters[rb], 1u) == (unsigned)(kDownSlices - 1));
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (tid < T * kDownRowsPerCta) {
        const int t = tid / kDownRowsPerCta, j = tid % kDownRowsPerCta;
        const int row = rb * kDownRowsPerCta + j;
        float v = 0.f;
#pragma unroll
        for (int st = 0; st < kStreams; ++st) {
            const int sa = 2 * st, sb = 2 * st + 1;
            const float ss = __ldcg(&ssq[(rb * kDownSlices + sa) * kDecodeMaxT + t]) +
                             __ldcg(&ssq[(rb * kDownSlices + sb) * kDecodeMaxT + t]);
            const float rs = 1.0f / sqrtf(ss / (float)kWidth + eps);
            const float d = __ldcg(&partials[(sa * kDecodeMaxT + t) * kRank + row]) +
                            __ldcg(&partials[(sb * kDecodeMaxT + t) * kRank + row]);
            v = fmaf(rs, d, v);
        }
        lo[t * kRank + row] = v;
    }
    if (tid == 0) counters[rb] = 0u;
}

template <int T>
__global__ void __launch_bounds__(kUpThreads)
up_mix_kernel(const float* __restrict__ R, const float* __restrict__ P,
              const uint16_t* __restrict__ W_up, const float* __restrict__ lo,
              const float* __restrict__ Rmix, float* __restrict__ out_f32,
              uint16_t* __restrict__ out_bf16, uint16_t* __restrict__ out_fp16) {
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x * kUpColsPerCta + warp;   // output column 0..2559
    const int s = lane >> 3;                             // stream of this lane's row
    const int part = lane & 7;                           // which 40 of the 320 inputs
    const int i = s * kWidth + c;                        // up row

    uint4 wv[5];
    const uint16_t* wrow = W_up + (size_t)i * kRank + part * 40;
#pragma unroll
    for (int q = 0; q < 5; ++q) wv[q] = ldg_stream_v4(wrow + 8 * q);

    __shared__ __align__(16) float lo_s[T][kRank];
    for (int e = tid; e < T * kRank; e += kUpThreads) lo_s[e / kRank][e % kRank] = lo[e];
    __syncthreads();

    float wf[40];
#pragma unroll
    for (int q = 0; q < 5; ++q) {
        wf[8 * q + 0] = bf16_lo(wv[q].x); wf[8 * q + 1] = bf16_hi(wv[q].x);
        wf[8 * q + 2] = bf16_lo(wv[q].y); wf[8 * q + 3] = bf16_hi(wv[q].y);
        wf[8 * q + 4] = bf16_lo(wv[q].z); wf[8 * q + 5] = bf16_hi(wv[q].z);
        wf[8 * q + 6] = bf16_lo(wv[q].w); wf[8 * q + 7] = bf16_hi(wv[q].w);
    }

#pragma unroll 1
    for (int t = 0; t < T; ++t) {
        const float4* l4 = reinterpret_cast<const float4*>(&lo_s[t][part * 40]);
        float acc = 0.f;
#pragma unroll
        for (int q = 0; q < 10; ++q) {
            const float4 x = l4[q];
            acc = fmaf(wf[4 * q + 0], x.x, acc);
            acc = fmaf(wf[4 * q + 1], x.y, acc);
            acc = fmaf(wf[4 * q + 2], x.z, acc);
            acc = fmaf(wf[4 * q + 3], x.w, acc);
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 4);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);

        const size_t off = (size_t)t * kCols + i;
        float rp = R[off];
        if (P != nullptr) rp += P[off];
        const float g = gate_value(acc, rp);
        const float g0 = __shfl_sync(0xffffffffu, g, 0);
        const float g1 = __shfl_sync(0xffffffffu, g, 8);
        const float g2 = __shfl_sync(0xffffffffu, g, 16);
        const float g3 = __shfl_sync(0xffffffffu, g, 24);
        if (part == 0) {
            const float m = mix_row(Rmix + (size_t)t * 16 + s * 4, g0, g1, g2, g3);
            out_f32[off] = m;
            out_bf16[off] = to_bf16_bits(m);
            out_fp16[off] = to_fp16_bits(m);
        }
    }
}

template <int T>
cudaError_t launch_chunk(const Ctx& ctx, const ReadArgs& a, int t0, cudaStream_t st) {
    const size_t off = (size_t)t0 * kCols;
    const float* R = a.R + off;
    const float* P = a.P ? a.P + off : nullptr;
    float* lo = ctx.s.lo + (size_t)t0 * kRank;
    down_slice_kernel<T><<<dim3(kDownSlices, kDownRowBlocks), kDownThreads, 0, st>>>(
        R, P, a.w_norm, a.W_down, ctx.s.partials, ctx.s.ssq, ctx.s.counters, lo, ctx.eps);
    up_mix_kernel<T><<<kWidth / kUpColsPerCta, kUpThreads, 0, st>>>(
        R, P, a.W_up, lo, a.Rmix + (size_t)t0 * 16, a.out_f32 + off, a.out_bf16 + off,
        a.out_fp16 + off);
    return cudaGetLastError();
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
