// Internal declarations shared by the translation units of the library.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
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

// Tokens at or below which HC_PATH_AUTO runs the decode kernels (up to 64 tokens in one
// pass over the weights). Measured on GB300 with one weight set and a pending write,
// us per read: decode 34.4 vs tile path 51.1 at 32 tokens, 52.1 vs 52.0 at 48, 66.6 vs
// 53.3 at 64.
constexpr int kAutoDecodeMaxT = 48;

// Scheduler pairs in Scratch::sched.
constexpr int kSchedUp = 0;
constexpr int kSchedDown = 1;
constexpr int kSchedPairs = 2;

// Device status word bits.
constexpr int kStatusTimeout = 1;
constexpr int kStatusBounds = 2;     // the range-checked build skipped an access
// Bound of a device-side wait on other CTAs before it gives up and reports a timeout.
constexpr uint64_t kDefaultWaitNs = 2000000000ull;   // 2 s

struct Scratch {
    float* lo = nullptr;             // [max_tokens][kRank], the down projection's output
    int* status = nullptr;           // device status word
    // tile-path schedulers: per kernel kind a pair {next tile, CTAs finished}; the
    // last CTA of a launch resets its pair to 0 for the next launch
    int* sched = nullptr;
    // one-kernel decode read: [0..19] CTAs of each row block that published their lo
    // rows, over all calls; [20] calls completed (zeroed with the status word after a
    // timeout)
    unsigned* sync = nullptr;
};
constexpr int kSyncWords = 32;

// Tensor maps over the caller's W_up for the decode up kernel, by W_up's address (a
// map depends on nothing else): encoding one costs host time on every call otherwise.
// Direct-mapped by a hash of the address; a collision only re-encodes.
struct WupMapCache {
    static constexpr int kSize = 64;
    const void* key[kSize] = {};
    CUtensorMap map[kSize];
};

struct Ctx {
    bool ready = false;
    int device = -1;
    int max_tokens = 0;
    float eps = 1e-6f;
    int sm_count = 0;
    bool fused_decode = false;       // the one-kernel decode read can run on this device
    // bound of the one-kernel decode read's wait for every CTA's lo (a test may shorten
    // it to make the wait run out; hc_read_set_wait_limit)
    uint64_t lo_wait_ns = kDefaultWaitNs;
    // HC_PATH_AUTO runs the decode kernels at or below this many tokens:
    // kAutoDecodeMaxT, or the HC_READ_DECODE_MAX_T environment variable as read by
    // hc_read_init
    int auto_decode_max_t = kAutoDecodeMaxT;
    char name[64] = {0};
    Scratch s;
    // prefill scratch
    // down partials, tile-blocked, in column quads, token-minor: [tiles][kStreams]
    // [4 K quarters][kRank / 4][128 tokens][4], and the sums of squares of R'
    // [tiles][kStreams][4 K quarters][128 tokens], tiles = partial_tiles(max_tokens)
    float* partials = nullptr;
    float* ssq = nullptr;
    // lo as three bf16 terms [3][max_tokens][kRank] (hi, mid, low; hi alone is lo
    // rounded once to bf16)
    uint16_t* lo3 = nullptr;
    float* gated = nullptr;          // [max_tokens][kCols], unfused prefill only (lazy)
    CUtensorMap tm_lo;               // TMA map over lo3
    // tokens whose lo the last tile-path call left in lo3 (0: none)
    int lo_tokens = 0;
    mutable WupMapCache wu_maps;     // decode: W_up tensor maps by address
};

// 128-token tiles of the partials.
inline int partial_tiles(int max_tokens) { return (max_tokens + 127) / 128; }

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
    int out_cols = kCols;            // output floats per token (kWidth for the y read-out)
};

// A TMA map over the caller's W_up [kCols][kRank] bf16, in boxes of 64 K x box_rows
// rows with the 128-byte swizzle (the K-major layout of a tcgen05 operand).
bool encode_w_up_bf16(CUtensorMap* map, const uint16_t* W_up, int box_rows);
// The decode up kernel's map over W_up (boxes of 64 K x 32 rows), from the context's
// cache or encoded into it; nullptr if it cannot be encoded.
const CUtensorMap* decode_w_up_map(const Ctx& ctx, const uint16_t* W_up);

// Forgets which decode kernels were allowed their shared memory on `device`, then
// sets those attributes for every chunk size, so that no launch inside a stream
// capture needs to (hc_read_init calls it; the attributes also survive a device
// reset that is followed by a new hc_read_init).
void decode_forget_smem(int device);
cudaError_t decode_setup(int device);

// Decode kernels for any T: launched in chunks of kDecodeMaxT tokens.
cudaError_t launch_decode(const Ctx& ctx, const ReadArgs& a, cudaStream_t st);

// Decode read as one kernel per chunk of up to 8 tokens (needs s.lo and s.sync; in
// hc_decode.cu). Sets kernel attributes; *usable tells whether all 20 clusters can be
// resident at once.
cudaError_t decode_fused_setup(bool* usable);
cudaError_t launch_decode_fused(const Ctx& ctx, const ReadArgs& a, cudaStream_t st);

// Prefill (tensor-core tile) path: TMA maps and kernel attributes, then the launch.
cudaError_t prefill_setup(Ctx& ctx);
// kReadoutY: the 2560-wide read-out y = sum of the gated streams, [T][2560] outputs.
enum class PrefillMode { kFused, kUnfused, kFusedBf16Lo, kReadoutY };
cudaError_t launch_prefill(const Ctx& ctx, const ReadArgs& a, PrefillMode mode, cudaStream_t st);
// The two halves of the tile path: down GEMM and lo split; then the up GEMM with its
// gate + mix epilogue (fused) or writing gated + the mix (unfused).
cudaError_t launch_prefill_down(const Ctx& ctx, const ReadArgs& a, cudaStream_t st);
// pdl: launched with programmatic dependent launch right after lo_split (inside a
// read); the stage run alone is an ordinary launch (its predecessor may write R).
cudaError_t launch_prefill_upmix(const Ctx& ctx, const ReadArgs& a, PrefillMode mode,
                                 cudaStream_t st, bool pdl = false);

}  // namespace hc
