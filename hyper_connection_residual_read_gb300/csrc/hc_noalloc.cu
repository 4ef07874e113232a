// hc_read_noalloc: the decode read for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc at all:
//   * code that runs as a plug-in inside a host engine or framework that owns every
//     byte of device memory and hands out fixed workspaces, so an allocation behind
//     its back breaks its memory accounting or fails under its cap;
//   * latency-critical loops that must never stall the device, where cudaMalloc and
//     cudaFree may synchronise;
//   * callers that never call hc_read_init, whose only job is to allocate the
//     library's scratch.
// For them this entry point runs the same decode kernels as hc_read, with the one
// piece of scratch they need (lo, the down projection's output, T x 320 floats)
// kept in a file-scope __device__ array of fixed size. The CUDA runtime reserves
// that array on every device that loads this library, and it stays there until the
// process exits; the library itself allocates nothing on this path.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "hc_internal.h"

namespace hc {
namespace {

constexpr int kNoAllocMaxTokens = 64;     // lo for up to 64 tokens: 80 KB per device
constexpr int kNoAllocMaxDevices = 64;

// lo [kNoAllocMaxTokens][kRank]. No entry needs to start at zero: the down kernel
// writes every value the up kernel then reads.
static __device__ __align__(256) float g_noalloc_lo[kNoAllocMaxTokens * kRank];

// Per device: the device address of g_noalloc_lo, valid for the CUDA context it was
// looked up in (identified by the driver's context ID, never reused within a
// process). A reset of the device creates a new context, in which the module, and so
// the array, may sit elsewhere: the next call then looks the address up again. Only
// a successful set-up is remembered.
struct DeviceScratch {
    std::mutex m;
    unsigned long long ctx_id = 0;
    float* lo = nullptr;
};
DeviceScratch g_scratch[kNoAllocMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// The driver's ID of the calling thread's current context (0 if it cannot be read).
unsigned long long current_ctx_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS ||
        ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// In host code g_noalloc_lo names a host-side stand-in, not device memory: the device
// address is looked up with the device current, once per device and context. The
// same first call sets the decode kernels' shared-memory attributes for every chunk
// size (1-8 tokens), so that no later call, with any token count, changes a kernel
// attribute: one call on a device before any stream capture is enough.
float* scratch_for(int device, cudaError_t* err) {
    DeviceScratch& d = g_scratch[device];
    std::lock_guard<std::mutex> lock(d.m);
    const unsigned long long id = current_ctx_id();
    if (d.lo != nullptr && id != 0 && id == d.ctx_id) {
        *err = cudaSuccess;
        return d.lo;
    }
    float* lo = nullptr;
    if ((*err = cudaGetSymbolAddress(reinterpret_cast<void**>(&lo), g_noalloc_lo)) != cudaSuccess ||
        (*err = decode_setup(device)) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    d.lo = lo;
    // the lookup has made the context current if it was not; an ID of 0 (unreadable)
    // means the address is looked up again on every call
    d.ctx_id = current_ctx_id();
    return lo;
}

bool device_ptr_ok(const void* p, int device) {
    if (p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u)) return false;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (at.type == cudaMemoryTypeManaged) return true;
    return at.type == cudaMemoryTypeDevice && at.device == device;
}

bool disjoint(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x + na <= y || y + nb <= x;
}

}  // namespace
}  // namespace hc

using namespace hc;

extern "C" int hc_read_noalloc(int tokens, const float* R, const float* P,
                               const uint16_t* w_norm, const uint16_t* W_down,
                               const uint16_t* W_up, const float* Rmix, float* out_f32,
                               uint16_t* out_bf16, uint16_t* out_fp16, float eps,
                               void* stream) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return HC_ERR_CUDA;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return HC_ERR_ARG;
    if (tokens < 0 || tokens > kNoAllocMaxTokens) return HC_ERR_ARG;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return HC_ERR_CUDA;
    if (major != 10 || minor != 3) return HC_ERR_ARCH;

    const void* ins[] = {R, w_norm, W_down, W_up, Rmix};
    for (const void* p : ins)
        if (!device_ptr_ok(p, dev)) return HC_ERR_ARG;
    if (P != nullptr && !device_ptr_ok(P, dev)) return HC_ERR_ARG;
    const void* outs[] = {out_f32, out_bf16, out_fp16};
    for (const void* p : outs)
        if (!device_ptr_ok(p, dev)) return HC_ERR_ARG;
    const size_t act = (size_t)tokens * kCols;
    const size_t out_bytes[3] = {act * 4, act * 2, act * 2};
    const void* in_ptr[6] = {R, P, w_norm, W_down, W_up, Rmix};
    const size_t in_bytes[6] = {act * 4, P ? act * 4 : 0, (size_t)kCols * 2,
                                (size_t)kRank * kCols * 2, (size_t)kCols * kRank * 2,
                                (size_t)tokens * 64};
    for (int i = 0; i < 3; ++i) {
        for (int j = i + 1; j < 3; ++j)
            if (!disjoint(outs[i], out_bytes[i], outs[j], out_bytes[j])) return HC_ERR_ARG;
        for (int j = 0; j < 6; ++j)
            if (in_ptr[j] && !disjoint(outs[i], out_bytes[i], in_ptr[j], in_bytes[j]))
                return HC_ERR_ARG;
    }
    if (tokens == 0) return HC_OK;

    cudaError_t err;
    float* lo = scratch_for(dev, &err);
    if (lo == nullptr) return HC_ERR_CUDA;

    Ctx c;                        // a view over the static scratch; owns nothing
    c.ready = true;
    c.device = dev;
    c.max_tokens = kNoAllocMaxTokens;
    c.eps = eps > 0.f ? eps : 1e-6f;
    c.s.lo = lo;
    ReadArgs a{tokens, R, P, w_norm, W_down, W_up, Rmix, out_f32, out_bf16, out_fp16};
    return launch_decode(c, a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? HC_OK
                                                                                : HC_ERR_CUDA;
}
