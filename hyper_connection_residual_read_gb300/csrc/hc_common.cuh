// Device helpers shared by the kernels of the library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace hc {

// Range checks of the bounds-checked build (compiled with -DHC_BOUNDS_CHECK): before a
// hand-indexed global access the kernel asks whether elements [i, i + n) lie within
// the buffer's extent as the kernel's own arguments give it; if not, the access is
// skipped and bit 2 of the device status word is set (hc_read_status reports
// HC_ERR_BOUNDS). There is no trap: the context stays usable. The normal build
// compiles every check to `true`. (TMA accesses need no check: the hardware clips
// them to the tensor map.)
#ifdef HC_BOUNDS_CHECK
__device__ __forceinline__ bool hc_in_range(size_t i, size_t n, size_t extent, int* status) {
    if (i + n <= extent) return true;
    if (status != nullptr) atomicOr(status, 2);
    return false;
}
#define HC_IN_RANGE(i, n, extent, status) \
    ::hc::hc_in_range(static_cast<size_t>(i), static_cast<size_t>(n), static_cast<size_t>(extent), (status))
#else
#define HC_IN_RANGE(i, n, extent, status) true
#endif

// 16-byte streaming load that skips L1 (each weight byte is read once per call).
__device__ __forceinline__ uint4 ldg_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Asks L2 to fetch the line holding p. It returns nothing, so it may run before the
// data is final: a later write updates the L2 line and a later load reads it there.
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Programmatic dependent launch. A kernel launched with programmatic stream
// serialisation may start while the previous kernel on the stream is still
// running; `pdl_wait` blocks until that kernel has completed and its writes are
// visible, and `pdl_launch_dependents` lets the next kernel start early. Only
// layer parameters (weights) may be read before `pdl_wait`.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Low and high bf16 of a packed pair, widened exactly to fp32.
__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

// The two 16-bit images of an fp32 value, round to nearest even.
__device__ __forceinline__ uint16_t to_bf16_bits(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
__device__ __forceinline__ uint16_t to_fp16_bits(float x) {
    return __half_as_ushort(__float2half_rn(x));
}

// x0 and x1 each as the sum of three bf16 terms, packed in pairs: hi = bf16(x),
// mid = bf16(x - hi), low = bf16(x - hi - mid), all round to nearest even. Both
// differences are exact in fp32, so the three terms carry x to about 2^-27 of its size
// with fp32's exponent range; the tensor cores multiply each term by a bf16 weight
// exactly and sum the products in fp32.
__device__ __forceinline__ void split3_bf16(float x0, float x1, uint32_t& hi, uint32_t& mid,
                                            uint32_t& low) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float r0 = x0 - __low2float(h), r1 = x1 - __high2float(h);
    const __nv_bfloat162 m = __floats2bfloat162_rn(r0, r1);
    const __nv_bfloat162 l = __floats2bfloat162_rn(r0 - __low2float(m), r1 - __high2float(m));
    hi = *reinterpret_cast<const uint32_t*>(&h);
    mid = *reinterpret_cast<const uint32_t*>(&m);
    low = *reinterpret_cast<const uint32_t*>(&l);
}

// The same split by truncation: hi = the top 16 bits of x (sign, exponent, 7 fraction
// bits), mid = the top 16 bits of x - hi, low = the top 16 bits of x - hi - mid. Both
// differences are exact, and each term takes the next 8 significant bits, so for a
// normal x whose remainders stay normal the three terms sum to x exactly (24 bits);
// masks and byte permutes replace split3_bf16's conversions. Packed as split3_bf16.
__device__ __forceinline__ void split3_trunc(float x0, float x1, uint32_t& hi, uint32_t& mid,
                                             uint32_t& low) {
    const uint32_t a0 = __float_as_uint(x0) & 0xFFFF0000u, a1 = __float_as_uint(x1) & 0xFFFF0000u;
    const float r0 = x0 - __uint_as_float(a0), r1 = x1 - __uint_as_float(a1);
    const uint32_t b0 = __float_as_uint(r0) & 0xFFFF0000u, b1 = __float_as_uint(r1) & 0xFFFF0000u;
    const float s0 = r0 - __uint_as_float(b0), s1 = r1 - __uint_as_float(b1);
    hi = __byte_perm(a0, a1, 0x7632);
    mid = __byte_perm(b0, b1, 0x7632);
    low = __byte_perm(__float_as_uint(s0), __float_as_uint(s1), 0x7632);
}

// The gate: logistic sigmoid of the up projection times the residual value. expf is
// the accurate one; the reciprocal is the fast one (within 2 ulp, and 0 when
// expf(-u) overflows).
__device__ __forceinline__ float gate_value(float u, float rp) {
    return rp * __fdividef(1.0f, 1.0f + expf(-u));
}

// The RMS-norm scale 1 / sqrt(a) of a stream, a = mean(R'^2) + eps. The hardware
// reciprocal square root (rsqrtf, within 2 ulp) refined by one step of Newton's method
// for f(y) = 1/y^2 - a, y <- y (3 - a y^2) / 2, which about doubles its correct bits:
// within about 1 ulp, as close as 1 / sqrtf(a) with its two roundings, but without the
// IEEE square root and division, whose latency sat on the decode read's critical path.
__device__ __forceinline__ float inv_rms(float a) {
    const float y = rsqrtf(a);
    return y * fmaf(-0.5f * a, y * y, 1.5f);
}

// Row s of the token's 4x4 mix applied to the 4 gated values (q = 0..3 in order).
__device__ __forceinline__ float mix_row(const float* m_row, float g0, float g1, float g2,
                                         float g3) {
    float v = m_row[0] * g0;
    v = fmaf(m_row[1], g1, v);
    v = fmaf(m_row[2], g2, v);
    v = fmaf(m_row[3], g3, v);
    return v;
}

}  // namespace hc
