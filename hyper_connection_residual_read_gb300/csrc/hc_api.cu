// C ABI of the hyper-connection read: contexts, argument checks, path choice,
// the once-per-device self check and the status word.
//
// The self check follows "#315 hc: the multi-token hyper-connection read split
// finer", "Exactness": at start-up every card runs the read on random bf16
// weights and inputs for 1..8 tokens, with and without the pending write, and
// compares outputs bit for bit before trusting a kernel.
#include <cuda_runtime.h>
#include <errno.h>
#include <limits.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "hc_common.cuh"
#include "hc_internal.h"

namespace hc {
namespace {

constexpr int kMaxDevices = 64;
Ctx g_ctx[kMaxDevices];

Ctx* current_ctx(int* err) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *err = HC_ERR_CUDA;
        return nullptr;
    }
    if (!g_ctx[dev].ready) {
        *err = HC_ERR_NOT_INIT;
        return nullptr;
    }
    *err = HC_OK;
    return &g_ctx[dev];
}

void free_ctx(Ctx& c) {
    if (c.device >= 0) cudaSetDevice(c.device);
    cudaFree(c.s.lo);
    cudaFree(c.s.status);
    cudaFree(c.s.sync);
    cudaFree(c.s.sched);
    cudaFree(c.partials);
    cudaFree(c.ssq);
    cudaFree(c.lo3);
    cudaFree(c.gated);
    c = Ctx();
}

struct Range {
    uintptr_t lo, hi;
};

bool overlaps(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

// A pointer the kernels may dereference: not null, 16-byte aligned, and device
// (or managed) memory of the context's device. Host pointers are refused here
// so that no kernel ever receives one.
int check_ptr(const void* p, int device) {
    if (p == nullptr) return HC_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(p) & 15u) return HC_ERR_ARG;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return HC_ERR_ARG;
    }
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) return HC_ERR_ARG;
    if (at.type == cudaMemoryTypeDevice && at.device != device) return HC_ERR_ARG;
    return HC_OK;
}

int validate(const Ctx& c, const ReadArgs& a) {
    if (a.T < 0 || a.T > c.max_tokens) return HC_ERR_ARG;
    // the y read-out has no mix matrix (Rmix is null there and not checked)
    const bool y = a.out_cols == kWidth;
    const void* ptrs[] = {a.R, a.w_norm, a.W_down, a.W_up, y ? a.R : a.Rmix, a.out_f32,
                          a.out_bf16, a.out_fp16};
    for (const void* p : ptrs)
        if (int e = check_ptr(p, c.device)) return e;
    if (a.P != nullptr)
        if (int e = check_ptr(a.P, c.device)) return e;
    const size_t act = (size_t)a.T * kCols;
    const size_t out = (size_t)a.T * a.out_cols;
    auto rng = [](const void* p, size_t bytes) {
        uintptr_t b = reinterpret_cast<uintptr_t>(p);
        return Range{b, b + bytes};
    };
    const Range outs[3] = {rng(a.out_f32, out * 4), rng(a.out_bf16, out * 2),
                           rng(a.out_fp16, out * 2)};
    Range ins[6] = {rng(a.R, act * 4), rng(a.w_norm, (size_t)kCols * 2),
                    rng(a.W_down, (size_t)kRank * kCols * 2),
                    rng(a.W_up, (size_t)kCols * kRank * 2),
                    y ? Range{0, 0} : rng(a.Rmix, (size_t)a.T * 64), Range{0, 0}};
    if (a.P) ins[5] = rng(a.P, act * 4);
    for (int i = 0; i < 3; ++i) {
        for (int j = i + 1; j < 3; ++j)
            if (overlaps(outs[i], outs[j])) return HC_ERR_ARG;
        for (const Range& r : ins)
            if (r.hi > r.lo && overlaps(outs[i], r)) return HC_ERR_ARG;
    }
    return HC_OK;
}

int run(int path, const ReadArgs& a, cudaStream_t st) {
    int err;
    Ctx* c = current_ctx(&err);
    if (!c) return err;
    if (path < HC_PATH_AUTO || path > HC_PATH_PREFILL_BF16_LO) return HC_ERR_ARG;
    if (int e = validate(*c, a)) return e;
    if (a.T == 0) return HC_OK;
    if (path == HC_PATH_AUTO) path = a.T <= c->auto_decode_max_t ? HC_PATH_DECODE : HC_PATH_PREFILL;
    cudaError_t ce;
    switch (path) {
        case HC_PATH_DECODE:
            ce = launch_decode(*c, a, st);
            break;
        case HC_PATH_DECODE_ONE_KERNEL:
            if (!c->fused_decode) return HC_ERR_ARG;   // its clusters cannot all be resident here
            ce = launch_decode_fused(*c, a, st);
            break;
        case HC_PATH_PREFILL:
            ce = launch_prefill(*c, a, PrefillMode::kFused, st);
            c->lo_tokens = a.T;
            break;
        case HC_PATH_PREFILL_BF16_LO:
            ce = launch_prefill(*c, a, PrefillMode::kFusedBf16Lo, st);
            c->lo_tokens = a.T;
            break;
        default:
            if (c->gated == nullptr) {
                // the unfused pair keeps gated in scratch: allocated on first use
                if (cudaMalloc(&c->gated, sizeof(float) * (size_t)c->max_tokens * kCols) !=
                    cudaSuccess) {
                    cudaGetLastError();
                    c->gated = nullptr;
                    return HC_ERR_NOMEM;
                }
            }
            ce = launch_prefill(*c, a, PrefillMode::kUnfused, st);
            c->lo_tokens = a.T;
            break;
    }
    return ce == cudaSuccess ? HC_OK : HC_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// self check helpers: device-side generator and comparisons
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
    // splitmix64 finaliser (Steele, Lea, Flood, "Fast splittable pseudorandom
    // number generators", 2014)
    z += 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ float unit_uniform(uint64_t seed, uint64_t i) {
    // 24 random bits -> [-1, 1)
    return (float)(mix64(seed ^ mix64(i)) >> 40) * (2.0f / 16777216.0f) - 1.0f;
}

__global__ void fill_f32(float* x, size_t n, uint64_t seed, float scale, float offset) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x)
        x[i] = offset + scale * unit_uniform(seed, i);
}

__global__ void fill_bf16(uint16_t* x, size_t n, uint64_t seed, float scale, float offset) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x)
        x[i] = to_bf16_bits(offset + scale * unit_uniform(seed, i));
}

__global__ void fill_mix(float* m, int T, uint64_t seed) {
    const int row = blockIdx.x * blockDim.x + threadIdx.x;  // token * 4 + stream
    if (row >= T * 4) return;
    float v[4], sum = 0.f;
    for (int q = 0; q < 4; ++q) {
        v[q] = 1.0f + unit_uniform(seed, (uint64_t)row * 4 + q);  // [0, 2)
        v[q] = v[q] * 0.5f + 0.01f;
        sum += v[q];
    }
    for (int q = 0; q < 4; ++q) m[row * 4 + q] = v[q] / sum;
}

__global__ void add_f32(const float* a, const float* b, float* c, size_t n) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x)
        c[i] = a[i] + b[i];
}

// res[0]: bit mismatches; res[1]: max |a - b| bits; res[2]: max |a| bits;
// res[3]: bf16 image mismatches of a; res[4]: fp16 image mismatches of a.
__global__ void compare_out(const float* a, const float* b, const uint16_t* ab16,
                            const uint16_t* ah16, size_t n, unsigned* res) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x) {
        const float x = a[i], y = b[i];
        if (__float_as_uint(x) != __float_as_uint(y)) atomicAdd(&res[0], 1u);
        atomicMax(&res[1], __float_as_uint(fabsf(x - y)));
        atomicMax(&res[2], __float_as_uint(fabsf(x)));
        if (ab16 && ab16[i] != to_bf16_bits(x)) atomicAdd(&res[3], 1u);
        if (ah16 && ah16[i] != to_fp16_bits(x)) atomicAdd(&res[4], 1u);
    }
}

struct CheckBufs {
    float *R = nullptr, *P = nullptr, *Rpre = nullptr, *M = nullptr;
    uint16_t *w = nullptr, *Wd = nullptr, *Wu = nullptr;
    float *o1 = nullptr, *o2 = nullptr;
    uint16_t *b1 = nullptr, *h1 = nullptr, *b2 = nullptr, *h2 = nullptr;
    unsigned* res = nullptr;
    void release() {
        void* all[] = {R, P, Rpre, M, w, Wd, Wu, o1, o2, b1, h1, b2, h2, res};
        for (void* p : all) cudaFree(p);
    }
};

}  // namespace
}  // namespace hc

using namespace hc;

extern "C" int hc_read_version(void) { return 102; }

extern "C" int hc_read_bounds_checked(void) {
#ifdef HC_BOUNDS_CHECK
    return 1;
#else
    return 0;
#endif
}

extern "C" const char* hc_read_strerror(int code) {
    switch (code) {
        case HC_OK: return "ok";
        case HC_ERR_ARG: return "invalid argument (null, size, alignment, overlap, or not device memory)";
        case HC_ERR_NOT_INIT: return "hc_read_init was not called for the current device";
        case HC_ERR_ARCH: return "device is not compute capability 10.3 (GB300)";
        case HC_ERR_CUDA: return "CUDA runtime or launch error";
        case HC_ERR_TIMEOUT: return "a bounded device-side wait gave up";
        case HC_ERR_CHECK: return "self check found a mismatch";
        case HC_ERR_NOMEM: return "scratch allocation failed";
        case HC_ERR_BOUNDS: return "the bounds-checked build skipped an out-of-range access";
        default: return "unknown status";
    }
}

namespace {
// The crossover of HC_PATH_AUTO from the environment: HC_READ_DECODE_MAX_T, a decimal
// token count >= 0 (a debugging aid). Unset, empty or not such a number: the measured
// default.
int auto_decode_max_t_from_env() {
    const char* v = getenv("HC_READ_DECODE_MAX_T");
    if (v == nullptr || *v == '\0') return kAutoDecodeMaxT;
    char* end = nullptr;
    errno = 0;
    const long t = strtol(v, &end, 10);
    if (errno != 0 || end == v || *end != '\0' || t < 0 || t > INT_MAX) return kAutoDecodeMaxT;
    return static_cast<int>(t);
}
}  // namespace

extern "C" int hc_read_init(int device, int max_tokens, float eps) {
    if (device < 0 || device >= kMaxDevices || max_tokens < 1) return HC_ERR_ARG;
    if (cudaSetDevice(device) != cudaSuccess) return HC_ERR_CUDA;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return HC_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return HC_ERR_ARCH;
    Ctx& c = g_ctx[device];
    if (c.ready) free_ctx(c);
    c.device = device;
    c.max_tokens = max_tokens;
    c.eps = eps > 0.f ? eps : 1e-6f;
    c.auto_decode_max_t = auto_decode_max_t_from_env();
    c.sm_count = prop.multiProcessorCount;
    strncpy(c.name, prop.name, sizeof(c.name) - 1);
    bool ok = true;
    ok &= cudaMalloc(&c.s.lo, sizeof(float) * (size_t)max_tokens * kRank) == cudaSuccess;
    ok &= cudaMalloc(&c.s.status, sizeof(int)) == cudaSuccess;
    ok &= cudaMalloc(&c.s.sync, kSyncWords * sizeof(unsigned)) == cudaSuccess;
    ok &= cudaMalloc(&c.s.sched, 2 * kSchedPairs * sizeof(int)) == cudaSuccess;
    const size_t ts = (size_t)partial_tiles(max_tokens) * 128;
    ok &= cudaMalloc(&c.partials, sizeof(float) * ts * kStreams * 4 * kRank) == cudaSuccess;
    ok &= cudaMalloc(&c.ssq, sizeof(float) * ts * kStreams * 4) == cudaSuccess;
    ok &= cudaMalloc(&c.lo3, sizeof(uint16_t) * 3 * (size_t)max_tokens * kRank) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        free_ctx(c);
        return HC_ERR_NOMEM;
    }
    if (cudaMemset(c.s.status, 0, sizeof(int)) != cudaSuccess ||
        cudaMemset(c.s.sync, 0, kSyncWords * sizeof(unsigned)) != cudaSuccess ||
        cudaMemset(c.s.sched, 0, 2 * kSchedPairs * sizeof(int)) != cudaSuccess ||
        decode_setup(device) != cudaSuccess ||
        decode_fused_setup(&c.fused_decode) != cudaSuccess ||
        cudaMemset(c.lo3, 0, sizeof(uint16_t) * 3 * (size_t)max_tokens * kRank) != cudaSuccess ||
        prefill_setup(c) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        free_ctx(c);
        return HC_ERR_CUDA;
    }
    c.ready = true;
    return HC_OK;
}

extern "C" int hc_read_path(int path, int tokens, const float* R, const float* P,
                            const uint16_t* w_norm, const uint16_t* W_down,
                            const uint16_t* W_up, const float* Rmix, float* out_f32,
                            uint16_t* out_bf16, uint16_t* out_fp16, void* stream) {
    ReadArgs a{tokens, R, P, w_norm, W_down, W_up, Rmix, out_f32, out_bf16, out_fp16};
    return run(path, a, static_cast<cudaStream_t>(stream));
}

extern "C" int hc_read(int tokens, const float* R, const float* P, const uint16_t* w_norm,
                       const uint16_t* W_down, const uint16_t* W_up, const float* Rmix,
                       float* out_f32, uint16_t* out_bf16, uint16_t* out_fp16, void* stream) {
    return hc_read_path(HC_PATH_AUTO, tokens, R, P, w_norm, W_down, W_up, Rmix, out_f32,
                        out_bf16, out_fp16, stream);
}

extern "C" int hc_read_upmix(int path, int tokens, const float* R, const float* P,
                             const uint16_t* W_up, const float* Rmix, float* out_f32,
                             uint16_t* out_bf16, uint16_t* out_fp16, void* stream) {
    int err;
    Ctx* c = current_ctx(&err);
    if (!c) return err;
    PrefillMode mode;
    if (path == HC_PATH_PREFILL) mode = PrefillMode::kFused;
    else if (path == HC_PATH_PREFILL_UNFUSED) mode = PrefillMode::kUnfused;
    else if (path == HC_PATH_PREFILL_BF16_LO) mode = PrefillMode::kFusedBf16Lo;
    else return HC_ERR_ARG;
    // lo must hold what this stage reads: the last tile-path call's lo, for at least
    // these tokens (every tile-path call leaves all three of its bf16 terms)
    if (tokens > c->lo_tokens) return HC_ERR_ARG;
    // w_norm and W_down are not used by this stage: validated against W_up, which is
    ReadArgs a{tokens, R, P, W_up, W_up, W_up, Rmix, out_f32, out_bf16, out_fp16};
    if (int e = validate(*c, a)) return e;
    if (tokens == 0) return HC_OK;
    if (mode == PrefillMode::kUnfused && c->gated == nullptr) {
        if (cudaMalloc(&c->gated, sizeof(float) * (size_t)c->max_tokens * kCols) != cudaSuccess) {
            cudaGetLastError();
            c->gated = nullptr;
            return HC_ERR_NOMEM;
        }
    }
    return launch_prefill_upmix(*c, a, mode, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? HC_OK
               : HC_ERR_CUDA;
}

extern "C" int hc_read_y(int tokens, const float* R, const float* P, const uint16_t* w_norm,
                         const uint16_t* W_down, const uint16_t* W_up, float* out_f32,
                         uint16_t* out_bf16, uint16_t* out_fp16, void* stream) {
    int err;
    Ctx* c = current_ctx(&err);
    if (!c) return err;
    ReadArgs a{tokens, R, P, w_norm, W_down, W_up, nullptr, out_f32, out_bf16, out_fp16, kWidth};
    if (int e = validate(*c, a)) return e;
    if (tokens == 0) return HC_OK;
    const cudaError_t ce = launch_prefill(*c, a, PrefillMode::kReadoutY,
                                          static_cast<cudaStream_t>(stream));
    c->lo_tokens = tokens;
    return ce == cudaSuccess ? HC_OK : HC_ERR_CUDA;
}

extern "C" int hc_read_lo_bf16(int tokens, uint16_t* lo_out, void* stream) {
    int err;
    Ctx* c = current_ctx(&err);
    if (!c) return err;
    if (tokens < 0 || tokens > c->lo_tokens) return HC_ERR_ARG;
    if (tokens == 0) return HC_OK;
    if (lo_out == nullptr || (reinterpret_cast<uintptr_t>(lo_out) & 15) != 0) return HC_ERR_ARG;
    if (int e = check_ptr(lo_out, c->device)) return e;
    return cudaMemcpyAsync(lo_out, c->lo3, sizeof(uint16_t) * (size_t)tokens * kRank,
                           cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? HC_OK
               : HC_ERR_CUDA;
}

extern "C" int hc_read_set_wait_limit(uint64_t ns) {
    int err;
    Ctx* c = current_ctx(&err);
    if (!c) return err;
    c->lo_wait_ns = ns > 0 ? ns : kDefaultWaitNs;
    return HC_OK;
}

extern "C" int hc_read_status(void* stream) {
    int err;
    Ctx* c = current_ctx(&err);
    if (!c) return err;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return HC_ERR_CUDA;
    int word = 0;
    if (cudaMemcpy(&word, c->s.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(c->s.status, 0, sizeof(int)) != cudaSuccess)
        return HC_ERR_CUDA;
    if (word & kStatusTimeout) {
        // a kernel that gave up may have left its scheduler pair or the one-kernel
        // decode read's exchange counters mid-count (the stream is idle here)
        if (cudaMemset(c->s.sched, 0, 2 * kSchedPairs * sizeof(int)) != cudaSuccess ||
            cudaMemset(c->s.sync, 0, kSyncWords * sizeof(unsigned)) != cudaSuccess)
            return HC_ERR_CUDA;
        return HC_ERR_TIMEOUT;
    }
    return (word & kStatusBounds) ? HC_ERR_BOUNDS : HC_OK;
}

extern "C" int hc_read_check(int max_tokens, uint64_t seed, hc_check_report* rep) {
    int err;
    Ctx* c = current_ctx(&err);
    if (!c) return err;
    if (max_tokens < 1) return HC_ERR_ARG;
    const int Tm = max_tokens < kDecodeMaxT ? max_tokens : kDecodeMaxT;
    if (Tm > c->max_tokens) return HC_ERR_ARG;
    hc_check_report r;
    memset(&r, 0, sizeof(r));
    r.device = c->device;
    r.sm_count = c->sm_count;
    r.tokens_checked = Tm;
    r.repeat_bitwise = r.pending_write_bitwise = r.images_bitwise = r.paths_agree = 1;
    r.max_rel_tol = 2e-6;
    strncpy(r.device_name, c->name, sizeof(r.device_name) - 1);

    CheckBufs b;
    const size_t act = (size_t)Tm * kCols;
    bool ok = true;
    ok &= cudaMalloc(&b.R, act * 4) == cudaSuccess;
    ok &= cudaMalloc(&b.P, act * 4) == cudaSuccess;
    ok &= cudaMalloc(&b.Rpre, act * 4) == cudaSuccess;
    ok &= cudaMalloc(&b.M, (size_t)Tm * 64) == cudaSuccess;
    ok &= cudaMalloc(&b.w, (size_t)kCols * 2) == cudaSuccess;
    ok &= cudaMalloc(&b.Wd, (size_t)kRank * kCols * 2) == cudaSuccess;
    ok &= cudaMalloc(&b.Wu, (size_t)kCols * kRank * 2) == cudaSuccess;
    ok &= cudaMalloc(&b.o1, act * 4) == cudaSuccess;
    ok &= cudaMalloc(&b.o2, act * 4) == cudaSuccess;
    ok &= cudaMalloc(&b.b1, act * 2) == cudaSuccess;
    ok &= cudaMalloc(&b.h1, act * 2) == cudaSuccess;
    ok &= cudaMalloc(&b.b2, act * 2) == cudaSuccess;
    ok &= cudaMalloc(&b.h2, act * 2) == cudaSuccess;
    ok &= cudaMalloc(&b.res, 5 * sizeof(unsigned)) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        b.release();
        return HC_ERR_NOMEM;
    }
    const int G = 4 * c->sm_count, B = 256;
    fill_f32<<<G, B>>>(b.R, act, seed ^ 0x11, 1.7f, 0.f);
    fill_f32<<<G, B>>>(b.P, act, seed ^ 0x22, 0.17f, 0.f);
    add_f32<<<G, B>>>(b.R, b.P, b.Rpre, act);
    fill_mix<<<(Tm * 4 + 127) / 128, 128>>>(b.M, Tm, seed ^ 0x33);
    fill_bf16<<<G, B>>>(b.w, kCols, seed ^ 0x44, 0.17f, 1.f);
    fill_bf16<<<G, B>>>(b.Wd, (size_t)kRank * kCols, seed ^ 0x55, 0.035f, 0.f);
    fill_bf16<<<G, B>>>(b.Wu, (size_t)kCols * kRank, seed ^ 0x66, 0.035f, 0.f);

    int rc = HC_OK;
    double max_rel = 0.0;
    auto read = [&](int path, int T, const float* R, const float* P, float* o, uint16_t* bb,
                    uint16_t* hh) {
        return hc_read_path(path, T, R, P, b.w, b.Wd, b.Wu, b.M, o, bb, hh, nullptr);
    };
    auto compare = [&](const float* x, const float* y, const uint16_t* xb, const uint16_t* xh,
                       size_t n, unsigned out[5]) {
        cudaMemset(b.res, 0, 5 * sizeof(unsigned));
        compare_out<<<G, B>>>(x, y, xb, xh, n, b.res);
        cudaMemcpy(out, b.res, 5 * sizeof(unsigned), cudaMemcpyDeviceToHost);
    };
    for (int T = 1; T <= Tm && rc == HC_OK; ++T) {
        const size_t n = (size_t)T * kCols;
        for (int withP = 0; withP < 2 && rc == HC_OK; ++withP) {
            const float* P = withP ? b.P : nullptr;
            unsigned res[5];
            if ((rc = read(HC_PATH_DECODE, T, b.R, P, b.o1, b.b1, b.h1)) != HC_OK) break;
            if ((rc = read(HC_PATH_DECODE, T, b.R, P, b.o2, b.b2, b.h2)) != HC_OK) break;
            compare(b.o1, b.o2, b.b1, b.h1, n, res);
            if (res[0] != 0) r.repeat_bitwise = 0;
            if (res[3] != 0 || res[4] != 0) r.images_bitwise = 0;
            if (withP) {
                if ((rc = read(HC_PATH_DECODE, T, b.Rpre, nullptr, b.o2, b.b2, b.h2)) != HC_OK)
                    break;
                compare(b.o1, b.o2, nullptr, nullptr, n, res);
                if (res[0] != 0) r.pending_write_bitwise = 0;
            }
            // the tile path, where built, must agree with the decode path
            int e = read(HC_PATH_PREFILL, T, b.R, P, b.o2, b.b2, b.h2);
            if (e == HC_OK) {
                compare(b.o1, b.o2, nullptr, nullptr, n, res);
                float d, m;
                memcpy(&d, &res[1], 4);
                memcpy(&m, &res[2], 4);
                const double rel = m > 0.f ? (double)d / (double)m : (double)d;
                if (rel > max_rel) max_rel = rel;
            } else if (e != HC_ERR_ARG) {
                rc = e;
            }
        }
    }
    if (cudaDeviceSynchronize() != cudaSuccess) rc = HC_ERR_CUDA;
    b.release();
    r.max_rel_diff = max_rel;
    r.paths_agree = max_rel <= r.max_rel_tol;
    if (rc == HC_OK && !(r.repeat_bitwise && r.pending_write_bitwise && r.images_bitwise &&
                         r.paths_agree))
        rc = HC_ERR_CHECK;
    if (rep) *rep = r;
    return rc;
}

extern "C" void hc_read_shutdown(void) {
    for (int d = 0; d < kMaxDevices; ++d)
        if (g_ctx[d].ready) free_ctx(g_ctx[d]);
}
