// Internal declarations shared by the translation units of the library.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "hc_read.h"

namespace hc {

constexpr int kStreams = HC_READ_STREAMS;        // n
constexpr int kWidth = HC_READ_WIDTH;            // C
constexpr int kRank = HC_READ_RANK;              // r
constexpr int kCols = kStreams * kWidth;         // N = n*C = 10240

// Decode path geometry (see hc_decode.cu).
constexpr int kDecodeMaxT = 8;                   // tokens per decode launch
constexpr int kDownSliceCols = 1280;             // K-slice of the down kernel (half a stream)
constexpr int kDownSlices = kCols / kDownSliceCols;   // 8
constexpr int kDownRowsPerCta = 16;
constexpr int kDownRowBlocks = kRank / kDownRowsPerCta;  // 20

// Tokens at or below which HC_PATH_AUTO runs the decode kernels.
constexpr int kAutoDecodeMaxT = 8;

// Device status word bits.
constexpr int kStatusTimeout = 1;

struct Scratch {
    float* lo = nullptr;             // [max_tokens][kRank], the down projection's output
    int* status = nullptr;           // device status word
};

struct Ctx {
    bool ready = false;
    int device = -1;
    int max_tokens = 0;
    float eps = 1e-6f;
    int sm_count = 0;
    char name[64] = {0};
    Scratch s;
    float* gated = nullptr;          // [max_tokens][kCols], unfused prefill only
};

struct ReadArgs {
    int T;
    const float* R;
    const float* P;
    const uint16_t* w_norm;
    const uint16_t* W_down;
    const uint16_t* W_up;
    const float* Rmix;
    float* out_f32;
    uint16_t* out_bf16;
    uint16_t* out_fp16;
};

// Decode kernels for any T: launched in chunks of kDecodeMaxT tokens.
cudaError_t launch_decode(const Ctx& ctx, const ReadArgs& a, cudaStream_t st);

}  // namespace hc
