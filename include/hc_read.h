/*
 * hc_read.h - C ABI of the GB300 hyper-connection residual read.
 *
 * One call reads T tokens. Per token it takes 4 residual streams of width 2560
 * and computes, in this order:
 *
 *   1. R' = R + P                   (optional pending write, one fp32 add)
 *   2. per-stream RMS norm of R', times w_norm
 *   3. lo = W_down . xn             (10240 -> 320, bf16 weights, fp32 sums)
 *   4. gated = sigmoid(W_up . lo) * R'   (320 -> 10240, the gate)
 *   5. mixed[s] = sum_q Rmix[s][q] * gated[q]   (per-token 4x4 mix), written as
 *      fp32 together with its bf16 and fp16 images.
 *
 * Sources (pages by title and section):
 *   "#315 hc: the multi-token hyper-connection read split finer" - "What changes"
 *       (norm per token and stream; down projection), "Exactness" (reads with and
 *       without the pending write; the once-per-card bitwise check).
 *   "#1370 prefill: opt-in STRATA_HC_UPMIX=1 on CUDA - the hyper-connection up
 *       projection with gr_mix_r as its epilogue (sm_80+)" - "Why" (the up GEMM
 *       writes gated, gr_mix_r reads it back with R), "What it does" (the fused
 *       up projection + mix writing mixed with its BF16 / FP16 images).
 *   "#2488 sycl/A770: faster hyper-connection read on Arc A-series" - "Summary"
 *       changes 1 (last slice reduces the slice partials in a fixed order) and 4
 *       (norm folded into the down projection).
 *   "#2226 STRATA_HC_PERSIST=1 (opt-in, HIP): the verifier's hyper-connection read
 *       as one persistent kernel" - "Summary" (the read at 1-8 tokens).
 *
 * Shapes are fixed: n = 4 streams, C = 2560, N = n*C = 10240, r = 320.
 *
 * Layouts (all row-major, contiguous, caller-owned DEVICE memory on the device
 * given to hc_read_init, 16-byte aligned):
 *   R, P      float    [T][4][2560]   residual and pending write (P may be NULL)
 *   w_norm    uint16_t [4][2560]      bf16 bits
 *   W_down    uint16_t [320][10240]   bf16 bits, [out][in], in index k = s*2560 + c
 *   W_up      uint16_t [10240][320]   bf16 bits, [out][in], out index i = s*2560 + c
 *   Rmix      float    [T][4][4]      row s mixes the 4 gated streams into stream s
 *   out_f32   float    [T][4][2560]   mixed
 *   out_bf16  uint16_t [T][4][2560]   bf16 bits, round-to-nearest-even of out_f32
 *   out_fp16  uint16_t [T][4][2560]   IEEE half bits, round-to-nearest-even of out_f32
 *
 * Ownership: the caller owns every tensor; they must stay valid until the work
 * enqueued on `stream` has completed. Outputs must not overlap each other or any
 * input. R and P are only read (R is not updated with P). The library owns its
 * scratch (slice partials, counters, lo, a device status word), allocated by
 * hc_read_init for up to max_tokens tokens.
 *
 * Ordering: the weights (w_norm, W_down, W_up) are layer parameters. The library
 * may start reading them before the kernel that precedes the call on `stream`
 * has finished (programmatic dependent launch), so they must not be produced by
 * that preceding kernel. R, P and Rmix are read only after it has finished.
 * Calls that share one device context must be issued on one stream at a time
 * (they share scratch).
 *
 * Errors: every function returns HC_OK (0) or a negative code. Argument errors
 * are detected on the host before anything is enqueued. Kernel-side faults that
 * the kernels can detect themselves (a bounded wait that ran out) set a device
 * status word, reported by hc_read_status(). hc_read never synchronises and
 * never falls back to another implementation.
 */
#ifndef HC_READ_H
#define HC_READ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HC_READ_STREAMS 4
#define HC_READ_WIDTH 2560
#define HC_READ_RANK 320

enum hc_status {
    HC_OK = 0,
    HC_ERR_ARG = -1,       /* null pointer, bad size, misalignment, overlap, host pointer */
    HC_ERR_NOT_INIT = -2,  /* hc_read_init was not called for the current device */
    HC_ERR_ARCH = -3,      /* the device is not compute capability 10.3 */
    HC_ERR_CUDA = -4,      /* a CUDA runtime call or a launch failed */
    HC_ERR_TIMEOUT = -5,   /* a bounded device-side wait gave up (status word) */
    HC_ERR_CHECK = -6,     /* hc_read_check found a mismatch */
    HC_ERR_NOMEM = -7,     /* scratch allocation failed */
    HC_ERR_BOUNDS = -8     /* the bounds-checked build skipped an out-of-range access
                              (status word; see hc_read_bounds_checked) */
};

/* Which kernels run. HC_PATH_AUTO picks the decode kernels for T <= 48 (the measured
 * crossover) and the tensor-core tile path above that; the others force one path
 * (tests, bench). The environment variable HC_READ_DECODE_MAX_T, a decimal token count
 * >= 0 read by hc_read_init, moves the crossover for that context (a debugging aid;
 * unset, empty or malformed keeps 48). Both paths are valid at every T. */
enum hc_path {
    HC_PATH_AUTO = 0,
    HC_PATH_DECODE = 1,            /* per 8 tokens: sliced down kernel (CUDA cores, clusters),
                                      then the up + gate + mix kernel (tcgen05) */
    HC_PATH_PREFILL = 2,           /* tile down, fused up + gate + mix epilogue (tcgen05;
                                      activations as three bf16 terms, fp32-accurate over
                                      fp32's whole range, weights used as stored) */
    HC_PATH_PREFILL_UNFUSED = 3,   /* tile down, up GEMM writing gated, then the mix */
    HC_PATH_DECODE_ONE_KERNEL = 4, /* per 8 tokens: one kernel, the decode down phase, an
                                      in-kernel lo exchange, an up + gate + mix on the CUDA
                                      cores (fp32 FMAs; within the tolerance of the others,
                                      not bitwise equal to them); HC_ERR_ARG where its 160
                                      CTAs cannot all be resident */
    HC_PATH_PREFILL_BF16_LO = 5    /* the pages' prefill numerics: tile down as in
                                      HC_PATH_PREFILL, then lo rounded once to bf16 and a
                                      single-term bf16 up GEMM on the caller's W_up with the
                                      fused epilogue ("#1370 prefill: opt-in STRATA_HC_UPMIX=1
                                      on CUDA ...", "What it does": the BF16 mma). Its output
                                      is exact to fp32 tolerance only against the read computed
                                      from that bf16 lo (hc_read_lo_bf16), not against the
                                      fp32-accurate read: expect about 1e-3 relative there. */
};

/* Creates the context of `device` (makes it current), checks that it is sm_103,
 * and allocates scratch for up to `max_tokens` tokens per call. eps <= 0 selects
 * 1e-6. Calling it again on the same device re-sizes the context. Returns
 * HC_ERR_ARG for max_tokens < 1, HC_ERR_ARCH, HC_ERR_NOMEM or HC_ERR_CUDA. */
int hc_read_init(int device, int max_tokens, float eps);

/* The read of `tokens` tokens (0 <= tokens <= max_tokens; 0 enqueues nothing),
 * asynchronous on `stream` (a cudaStream_t; NULL = the legacy default stream).
 * Output is bitwise deterministic for a given path and T. */
int hc_read(int tokens,
            const float* R, const float* P,
            const uint16_t* w_norm, const uint16_t* W_down, const uint16_t* W_up,
            const float* Rmix,
            float* out_f32, uint16_t* out_bf16, uint16_t* out_fp16,
            void* stream);

/* hc_read with an explicit path (enum hc_path). Same arguments and errors. The
 * unfused prefill path keeps gated [T][10240] fp32 in library scratch, which it
 * allocates on its first use (the only call that may allocate after init). */
int hc_read_path(int path, int tokens,
                 const float* R, const float* P,
                 const uint16_t* w_norm, const uint16_t* W_down, const uint16_t* W_up,
                 const float* Rmix,
                 float* out_f32, uint16_t* out_bf16, uint16_t* out_fp16,
                 void* stream);

/* Runs again only the second half of the tile path for the tokens of the most
 * recent tile-path call on this context: the up projection on the lo that call left
 * in the context's scratch (as three bf16 terms, whatever the call's path), with the
 * gate and the 4x4 mix, as `path` says: HC_PATH_PREFILL (fused epilogue),
 * HC_PATH_PREFILL_UNFUSED (up GEMM writing gated, then the mix) or
 * HC_PATH_PREFILL_BF16_LO (the first term alone, fused). W_up (bf16, [10240][320]) is
 * read by all three. R, P, W_up and Rmix must be that call's (or equal) tensors.
 * HC_ERR_ARG if the last tile-path call read fewer tokens (or none), or for any path
 * but these three. Stage timing and the fused-versus-unfused comparison use it; a read
 * needs only hc_read. Otherwise the checks and errors of hc_read. The pages have no
 * counterpart of it. */
int hc_read_upmix(int path, int tokens,
                  const float* R, const float* P, const uint16_t* W_up, const float* Rmix,
                  float* out_f32, uint16_t* out_bf16, uint16_t* out_fp16,
                  void* stream);

/* The read with a 2560-wide read-out instead of the 4x4 mix: per token and column,
 * y[c] = gated[0][c] + gated[1][c] + gated[2][c] + gated[3][c] (streams summed in
 * that order in fp32), written as out_f32 [T][2560] fp32 and its round-to-nearest-
 * even bf16 / fp16 images out_bf16, out_fp16 [T][2560]. Steps 1-4 are those of
 * hc_read (tensor-core tile path, fp32-accurate, any T). The pages have no entry
 * point of this shape: it is the read-out under which "#1370 prefill: opt-in
 * STRATA_HC_UPMIX=1 on CUDA ...", "Why" (gr_mix_r moving about 102 KB per token)
 * adds up, 40 KB of gated and 40 KB of residual in and a 2560-wide fp32 + bf16 +
 * fp16 row out. Same checks and errors as hc_read, with no Rmix. */
int hc_read_y(int tokens,
              const float* R, const float* P,
              const uint16_t* w_norm, const uint16_t* W_down, const uint16_t* W_up,
              float* out_f32, uint16_t* out_bf16, uint16_t* out_fp16,
              void* stream);

/* Copies lo of the most recent tile-path call on this context, rounded once to bf16
 * (round to nearest even; [tokens][320] bf16 bits, row-major), into lo_out (device
 * memory, 16-byte aligned, caller-owned), asynchronously on `stream`. It is what the
 * up GEMM of HC_PATH_PREFILL_BF16_LO takes as its A operand, the stage input that
 * checks of that path condition on. HC_ERR_ARG if tokens exceeds the token count of
 * that call (or there was none), or lo_out is null, misaligned or not device memory of
 * the context's device. */
int hc_read_lo_bf16(int tokens, uint16_t* lo_out, void* stream);

/* Result of the once-per-device self check. */
typedef struct hc_check_report {
    int device;
    int sm_count;
    int tokens_checked;          /* 1..tokens_checked, each with and without P */
    int repeat_bitwise;          /* 1 if two runs of every case gave the same bits */
    int pending_write_bitwise;   /* 1 if read(R, P) == read(R + P, NULL) bit for bit */
    int images_bitwise;          /* 1 if the bf16/fp16 outputs are the RNE images of out_f32 */
    int paths_agree;             /* 1 if decode and prefill agree within max_rel_tol */
    double max_rel_diff;         /* max |decode - prefill| / max |decode| over all cases */
    double max_rel_tol;          /* the tolerance used for paths_agree */
    char device_name[64];
} hc_check_report;

/* Runs both paths on device-generated pseudo-random inputs (seeded) for
 * 1..max_tokens tokens (at most 8), with and without a pending write, and checks
 * run-to-run bitwise repeat, the pending-write identity, the image rounding and
 * the agreement of the two paths. Synchronises the device. Allocates and frees
 * its own buffers. Returns HC_OK or HC_ERR_CHECK (report filled either way if
 * rep is not NULL). */
int hc_read_check(int max_tokens, uint64_t seed, hc_check_report* rep);

/* Waits for `stream`, then reads and clears the device status word of the current
 * device's context: HC_OK, or HC_ERR_TIMEOUT if a bounded wait gave up since the last
 * call (the outputs of that call are then unspecified; the library resets its own
 * schedulers, so the next call runs normally), or HC_ERR_BOUNDS if the bounds-checked
 * build skipped an access. HC_ERR_CUDA if the stream itself reports an error. */
int hc_read_status(void* stream);

/* Sets the bound of the one-kernel decode read's device-side wait for the other
 * CTAs' lo (HC_PATH_DECODE_ONE_KERNEL) on the current device's context, in
 * nanoseconds; 0 restores the default of 2 s. Failure-detection tests shorten it so
 * that the wait runs out: the read then returns, hc_read_status reports
 * HC_ERR_TIMEOUT and resets the exchange counters, and the next read runs normally.
 * Only this wait, which has no copy in flight, is affected. The pages' persistent
 * read has the same kind of bound ("#2226 STRATA_HC_PERSIST=1 (opt-in, HIP): the
 * verifier's hyper-connection read as one persistent kernel", "What changed": a
 * barrier timeout after which the read falls back). HC_ERR_NOT_INIT without a
 * context. */
int hc_read_set_wait_limit(uint64_t ns);

/* Static description of a status code. */
const char* hc_read_strerror(int code);

/* Frees the scratch of every device context. */
void hc_read_shutdown(void);

/* The decode read for callers that cannot allocate device memory: plug-ins that
 * run inside a host engine which owns all device memory and hands out fixed
 * workspaces, latency-critical loops where cudaMalloc/cudaFree could synchronise
 * the device, and callers that never call hc_read_init (which allocates). The
 * pages have no counterpart of this entry point.
 *
 * Same arguments and layouts as hc_read, plus eps (<= 0 selects 1e-6); no
 * hc_read_init is needed. It runs the decode kernels for 0 <= tokens <= 64 and
 * keeps their scratch (the down projection's output, 64 x 320 floats = 80 KB) in
 * a fixed array in device memory that the CUDA runtime reserves on every device
 * that loads the library, until the process exits. It calls no cudaMalloc,
 * cudaFree or other allocating routine. Returns HC_ERR_ARG for tokens > 64 or the
 * pointer errors hc_read refuses, HC_ERR_ARCH off sm_103, HC_ERR_CUDA otherwise.
 *
 * The first call with tokens >= 1 on a device (with that device current) looks up
 * the array's device address and sets the decode kernels' shared-memory attributes
 * for every chunk size, so that one such call before any stream capture is enough
 * for calls of any token count after it. After a device reset (a new CUDA context)
 * the next call does that set-up again. Every call on a device shares the one array:
 * calls that may overlap on the GPU (on different streams without ordering between
 * them) race and must not be made.
 *
 * This entry has no device status word. If one of its bounded device waits gives up
 * (after 2 s, which only a stalled device causes), the kernels write NaN into the
 * outputs of the tokens concerned instead of leaving stale values there. */
int hc_read_noalloc(int tokens,
                    const float* R, const float* P,
                    const uint16_t* w_norm, const uint16_t* W_down, const uint16_t* W_up,
                    const float* Rmix,
                    float* out_f32, uint16_t* out_bf16, uint16_t* out_fp16,
                    float eps, void* stream);

/* ABI version (major * 100 + minor). */
int hc_read_version(void);

/* 1 if this library was compiled with -DHC_BOUNDS_CHECK, else 0. In that build every
 * hand-indexed global access of every kernel is first checked against its buffer's
 * extent as the kernel's arguments give it; an access out of range is skipped, and
 * hc_read_status reports HC_ERR_BOUNDS. There is no trap, so the context stays
 * usable. The normal build has no checks. It stands in for a memory checker, and
 * the pages have no counterpart of it. */
int hc_read_bounds_checked(void);

#ifdef __cplusplus
}
#endif

#endif /* HC_READ_H */
