// Prefill path of the hyper-connection read: thousands of tokens per call, on the
// tcgen05 tensor cores with accumulators in tensor memory and operands fed by TMA.
//
//   down_tile        the down projection per (128-token tile, stream, quarter of the
//                    stream's 2560 columns): A = R' * w_norm split on the fly into three
//                    bf16 terms, B = those columns of the caller's bf16 W_down as stored,
//                    D = 128 x 320 fp32 in TMEM. The epilogue stores the unscaled
//                    partial dots and the quarter's sums of squares of R'.
//   lo_split         the norm fold of "#2488 sycl/A770: faster hyper-connection read
//                    on Arc A-series", Summary, change 4: each stream's rs applied to
//                    that stream's partial dots, summed in a fixed order; lo is stored
//                    as three bf16 terms for the up projection's A operand.
//   upmix_tile       the up projection per (128-token tile, 64 columns x 4 streams) on
//                    the caller's bf16 W_up, D = 128 x 256 fp32, double-buffered in
//                    TMEM; the epilogue applies the gate and the 4x4 mix and writes
//                    mixed with its bf16 and fp16 images, so `gated` never reaches
//                    memory ("#1370 prefill: opt-in STRATA_HC_UPMIX=1 on CUDA - the
//                    hyper-connection up projection with gr_mix_r as its epilogue
//                    (sm_80+)", "Why" and "What it does"). The unfused variant stores
//                    `gated` instead, and mix_gated applies the same mix afterwards
//                    (bitwise the same result).
//
// Three bf16 terms per activation reproduce fp32 accuracy with fp32's exponent range,
// so the path takes any finite fp32 input: the down tile's activations split by
// truncation (split3_trunc, exact), lo by rounding (split3_bf16, whose hi term is lo's
// bf16 image for the bf16-lo mode). The weights are used as the caller stores them
// (bf16, exact), each product of the MMA is exact, and the sums are fp32 in TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "hc_common.cuh"
#include "hc_internal.h"
#include "hc_tc.cuh"

namespace hc {
namespace {

using namespace tc;

constexpr int kTileM = 128;            // tokens per tile (TMEM lanes)
constexpr int kBK = 64;                // K of a W_up box for the decode up kernel (128-byte swizzle)
constexpr int kTerms = 3;              // bf16 terms of an activation (split3_bf16)

// down_tile
constexpr int kDownN = kRank;          // 320 accumulator columns (two MMAs of N = 160)
// K blocks of 32. A stage holds the block's A operand (three 8 KB bf16 terms of 128
// tokens x 32, 64-byte swizzled) and its W_down columns (20 KB: two 64-byte-swizzled
// boxes of 160 rows); four stages. R comes through a ring of its own (128 tokens x 32
// fp32, 16 KB a slot, 128-byte swizzled), read by the converter warps only.
constexpr int kDownBK = 32;
constexpr int kDownStages = 4;
constexpr int kDownRSlots = 2;
constexpr int kDownTileBytes = kTileM * kDownBK * 2;   // 8 KB: one 128 x 32 bf16 term
constexpr int kDownBBytes = kDownN * kDownBK * 2;      // 20 KB
constexpr int kDownStageBytes = kTerms * kDownTileBytes + kDownBBytes;
constexpr int kDownRBytes = kTileM * kDownBK * 4;      // 16 KB
constexpr int kDownKBlocks = kWidth / kDownBK;         // 80 per stream
// Each stream's K is split into quarters with an accumulator (and a partial) each:
// the tensor cores' fp32 accumulation rounds toward zero at every MMA, so the depth
// of one accumulation (here 20 K blocks x 2 steps x 3 terms = 120 MMAs) bounds the
// relative shrink of the result.
constexpr int kDownKSplit = 4;
constexpr int kDownKBlocksPerTile = kDownKBlocks / kDownKSplit;   // 20
// TMA, MMA, 8 converter warps, 4 epilogue warps (one per TMEM lane quarter): the
// epilogue of one tile runs while the converters already produce the next tile's A
constexpr int kDownThreads = 448;
// tiles from a run-time counter, as in the up tile below; the queue's consumers are
// the MMA issuer, 8 converter warps and 4 epilogue warps
constexpr int kDownTileQ = 4;
// The 320-column accumulator as two halves of 160 columns, rotating through three
// half-buffers of TMEM (480 of its 512 columns): tile lt writes half-buffer uses 2 lt
// and 2 lt + 1, so its MMAs need only the first half of the previous tile drained.
constexpr int kDownHalf = kDownN / 2;
constexpr int kDownHalfBufs = 3;
// R blocks are asked into L2 this many K blocks before their TMA load
constexpr int kDownPrefetch = 6;
constexpr int kDownTileQConsumers = 1 + 8 + 4;
// K blocks whose first-half MMAs are issued before the wait for a tile's second
// half-buffer (at most kDownStages)
constexpr int kDownAhead = 2;
static_assert(kDownAhead >= 1 && kDownAhead <= kDownStages, "MMA issue order");
constexpr int kDownSmem = kDownStages * kDownStageBytes + kDownRSlots * kDownRBytes + 1024;

// upmix_tile
constexpr int kUpCols = 64;            // output columns per tile (x 4 streams = N 256)
constexpr int kUpN = kStreams * kUpCols;
// K blocks of 32 (one 64-byte swizzle row): three stages of 40 KB (three 8 KB lo
// terms and 16 KB of W_up) leave room for three R slots per epilogue group below
constexpr int kUpBK = 32;
constexpr int kUpStages = 3;
constexpr int kUpTileBytes = kTileM * kUpBK * 2;  // 8 KB: one 128 x 32 bf16 lo term
constexpr int kUpBBytes = kUpN * kUpBK * 2;       // 16 KB
constexpr int kUpStageBytes = kTerms * kUpTileBytes + kUpBBytes;   // 40 KB
constexpr int kUpKBlocks = kRank / kUpBK;         // 10
constexpr int kUpColTiles = kWidth / kUpCols;     // 40
// Eight epilogue warps: two per TMEM lane quarter (32 tokens), one for each half of
// the tile's steps. The epilogue takes its tile in steps of 8 columns; a dedicated
// warp streams the R (and P) tiles of those steps, 128 tokens x 8 columns x 4
// streams, through a ring of 16 KB slots ahead of the epilogue warps. Each lane
// owns one token row and writes it with 32-byte stores: 8 fp32 columns of a
// stream per step, and 16 columns of each 16-bit image per pair of steps, so
// every store fills whole DRAM sectors and no output passes through shared memory.
constexpr int kUpEpiWarps = 8;
// Warpgroup 0: operand TMA, MMA issuer, R TMA and one idle warp; warpgroups 1-2: the
// epilogue. The block is launched with kUpRegsLaunch registers a thread; warpgroup 0
// then gives registers up and the epilogue takes them (setmaxnreg):
// 128 x (kUpRegsLaunch - kUpRegsLow) = 256 x (kUpRegsHigh - kUpRegsLaunch).
constexpr int kUpThreads = 128 + 32 * kUpEpiWarps;
constexpr int kUpRegsLaunch = 168, kUpRegsLow = 56, kUpRegsHigh = 224;
static_assert(128 * (kUpRegsLaunch - kUpRegsLow) == 256 * (kUpRegsHigh - kUpRegsLaunch),
              "the epilogue may take only what warpgroup 0 gives up");
constexpr int kEpiCols = 8;
// Tiles are handed out at run time: a CTA's first tile is its block index, the
// rest come from a global counter in index order, so a CTA that runs fast takes
// more tiles and all CTAs finish within about one tile of each other. The fetching
// thread passes each index through a small queue in shared memory to the CTA's
// other roles (MMA issuer, two R producers, 8 epilogue warps).
constexpr int kTileQ = 4;
constexpr int kTileQConsumers = 3 + kUpEpiWarps;
constexpr int kEpiRows = 32;
constexpr int kRSlot = kStreams * kTileM * kEpiCols * 4;        // 16 KB
// Each epilogue group has its own ring of R slots and its own producer, so every
// warp that waits on a slot's barrier consumes every fill of that slot. (With one
// ring shared by both groups a warp a tile ahead of the other group could wait on
// a slot whose previous fill, for the other group, was still in flight, and its
// parity wait would take the fill before that one as complete.)
constexpr int kRSlotsPerGroup = 3;
constexpr int kRSlots = 2 * kRSlotsPerGroup;
constexpr int kUpSmem = kUpStages * kUpStageBytes + kRSlots * kRSlot + 1024;
static_assert(kUpSmem <= 227 * 1024 - 1024, "up tile shared memory");
static_assert(kDownSmem <= 227 * 1024 - 2048, "down tile shared memory");

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// 32-byte global accesses (one whole DRAM sector per lane).
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t (&v)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v[0]),
                 "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// ---------------------------------------------------------------------------
// down projection, one (128-token tile, stream, K quarter) per tile, persistent CTAs
//
// Per K block of 32 columns, TMA brings R into a slot of the R ring (128-byte
// swizzled; rows past T read as zero) and the W_down columns into a stage. The
// converter warps take one token row a thread and half of the block's columns: a
// thread reads its 16 R values (the swizzle spreads the 32 lanes' rows over all
// banks), adds P, scales by w_norm, splits the products into three bf16 terms and
// stores them as 16-byte pieces of its row of the stage's 64-byte-swizzled A tiles
// (again on distinct banks). The converters set the tile's pace: a K block's
// conversion takes them longer than its 12 MMAs take the tensor core.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kDownThreads, 1)
down_tile_kernel(const float* __restrict__ P, const uint16_t* __restrict__ w_norm,
                 const __grid_constant__ CUtensorMap tm_wd, const __grid_constant__ CUtensorMap tm_r,
                 float* __restrict__ partials, float* __restrict__ ssq, int T,
                 int* __restrict__ status, int* __restrict__ sched) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    // per stage: A written by every converter thread and B landed (full_bar), the
    // stage's MMAs done (empty_bar); per R slot: landed (r_full), read by every
    // converter thread (r_empty)
    __shared__ __align__(8) uint64_t full_bar[kDownStages], empty_bar[kDownStages];
    __shared__ __align__(8) uint64_t r_full[kDownRSlots], r_empty[kDownRSlots];
    __shared__ __align__(8) uint64_t tq_full[kDownTileQ], tq_empty[kDownTileQ];
    __shared__ int tile_q[kDownTileQ];
    __shared__ __align__(8) uint64_t acc_full, acc_empty[kDownHalfBufs], ss_full[2];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;
    // per-row sums of squares by tile parity, one per K half of the row
    __shared__ float ss_s[2][2][kTileM];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles = ((T + kTileM - 1) / kTileM) * kStreams * kDownKSplit;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kDownStages; ++i) {
            mbar_init(&full_bar[i], 256 + 1);
            mbar_init(&empty_bar[i], 1);
        }
        for (int i = 0; i < kDownRSlots; ++i) {
            mbar_init(&r_full[i], 1);
            mbar_init(&r_empty[i], 256);
        }
        mbar_init(&acc_full, 1);
        for (int i = 0; i < kDownHalfBufs; ++i) mbar_init(&acc_empty[i], 128);
        mbar_init(&ss_full[0], 256);
        mbar_init(&ss_full[1], 256);
        for (int i = 0; i < kDownTileQ; ++i) {
            mbar_init(&tq_full[i], 1);
            mbar_init(&tq_empty[i], kDownTileQConsumers);
        }
        abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(&tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    auto sA = [&](int slot, int term) { return smem + slot * kDownStageBytes + term * kDownTileBytes; };
    auto sB = [&](int slot) { return smem + slot * kDownStageBytes + kTerms * kDownTileBytes; };
    auto sR = [&](int rs) { return smem + kDownStages * kDownStageBytes + rs * kDownRBytes; };
    // the CTA's i-th tile from the queue (n_tiles: no more tiles, or the CTA gave up),
    // taken by a whole warp (its lane 0 releases the entry once every lane has read
    // it) or by one thread
    auto take_tile = [&](int i, bool whole_warp) -> int {
        const int tile = mbar_wait(&tq_full[i % kDownTileQ], (i / kDownTileQ) & 1, &abort_flag, status)
                             ? tile_q[i % kDownTileQ]
                             : n_tiles;
        if (whole_warp) __syncwarp();
        if (!whole_warp || lane == 0) mbar_arrive(&tq_empty[i % kDownTileQ]);
        return tile;
    };

    if (warp == 0) {
        // producer: fetches the CTA's tiles; per K block the R block (into the R ring)
        // and the stream's W_down columns (320 rows as two boxes of 160, into a stage)
        if (lane == 0) {
            int it = 0;
            // the tile after the current one is fetched one tile early, so that its
            // first R blocks can be asked into L2 while the current tile is loaded
            int next = blockIdx.x;
            for (int i = 0; !abort_flag; ++i) {
                if (!mbar_wait(&tq_empty[i % kDownTileQ], ((i / kDownTileQ) & 1) ^ 1, &abort_flag, status))
                    break;
                const int tile = next;
                tile_q[i % kDownTileQ] = tile;
                mbar_arrive(&tq_full[i % kDownTileQ]);
                if (tile >= n_tiles) break;
                next = (int)gridDim.x + atomicAdd(sched, 1);
                const int tt = tile / (kStreams * kDownKSplit);
                const int s = (tile / kDownKSplit) % kStreams, kq = tile % kDownKSplit;
                const int ntt = next / (kStreams * kDownKSplit);
                const int ns = (next / kDownKSplit) % kStreams, nkq = next % kDownKSplit;
                for (int kb = kq * kDownKBlocksPerTile; kb < (kq + 1) * kDownKBlocksPerTile; ++kb, ++it) {
                    const int rs = it % kDownRSlots;
                    if (!mbar_wait(&r_empty[rs], ((it / kDownRSlots) & 1) ^ 1, &abort_flag, status)) break;
                    mbar_arrive_expect_tx(&r_full[rs], kDownRBytes);
                    tma_load_3d(sR(rs), &tm_r, kb * kDownBK, s, tt * kTileM, &r_full[rs]);
                    const int slot = it % kDownStages;
                    if (!mbar_wait(&empty_bar[slot], ((it / kDownStages) & 1) ^ 1, &abort_flag, status)) break;
                    mbar_arrive_expect_tx(&full_bar[slot], kDownBBytes);
                    const int x = s * kWidth + kb * kDownBK;
                    tma_load_2d(sB(slot), &tm_wd, x, 0, &full_bar[slot]);
                    tma_load_2d(sB(slot) + kDownBBytes / 2, &tm_wd, x, kDownN / 2, &full_bar[slot]);
                    // R of the block kDownPrefetch stages ahead into L2: later in this
                    // tile, or at the start of the next one
                    const int pk = kb - kq * kDownKBlocksPerTile + kDownPrefetch;
                    if (pk < kDownKBlocksPerTile)
                        tma_prefetch_3d(&tm_r, (kb + kDownPrefetch) * kDownBK, s, tt * kTileM);
                    else if (next < n_tiles)
                        tma_prefetch_3d(&tm_r, (nkq * kDownKBlocksPerTile + pk - kDownKBlocksPerTile) * kDownBK,
                                        ns, ntt * kTileM);
                }
            }
        }
    } else if (warp == 1) {
        // MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kTileM, kDownHalf);
            int it = 0;
            // waits until half-buffer use u may be written: its previous use drained
            auto half_free = [&](int u) {
                return mbar_wait(&acc_empty[u % kDownHalfBufs], ((u / kDownHalfBufs) & 1) ^ 1,
                                 &abort_flag, status);
            };
            for (int lt = 0; !abort_flag; ++lt) {
                if (take_tile(lt, false) >= n_tiles) break;
                // the tile's two halves go to half-buffer uses 2 lt and 2 lt + 1
                const uint32_t d0 = tmem + ((2 * lt) % kDownHalfBufs) * kDownHalf;
                const uint32_t d1 = tmem + ((2 * lt + 1) % kDownHalfBufs) * kDownHalf;
                if (!half_free(2 * lt)) break;
                tc_fence_after();
                bool ok = true;
                auto issue_half = [&](int h, int slot, int kl) {
                    const uint32_t b0 = smem_u32(sB(slot));
#pragma unroll
                    for (int term = 0; term < kTerms; ++term) {
                        const uint32_t a0 = smem_u32(sA(slot, term));
#pragma unroll
                        for (int kk = 0; kk < kDownBK / 16; ++kk)
                            mma_f16(h ? d1 : d0, desc_sw64(a0 + kk * 32),
                                    desc_sw64(b0 + h * (kDownBBytes / 2) + kk * 32), idesc,
                                    (kl | term | kk) != 0);
                    }
                };
                // the first kDownAhead K blocks' first-half MMAs go before the wait for
                // the second half-buffer, which the epilogue is usually still draining
                // from the previous tile; each half still accumulates in (K block, term,
                // K step) order
                for (int kl = 0; kl < kDownAhead; ++kl) {
                    const int slot = (it + kl) % kDownStages;
                    const uint32_t ph = ((it + kl) / kDownStages) & 1;
                    if (!mbar_wait(&full_bar[slot], ph, &abort_flag, status)) { ok = false; break; }
                    tc_fence_after();
                    issue_half(0, slot, kl);
                }
                if (ok) {
                    if (!half_free(2 * lt + 1)) ok = false;
                    else tc_fence_after();
                }
                for (int kl = 0; ok && kl < kDownAhead; ++kl) {
                    const int slot = (it + kl) % kDownStages;
                    issue_half(1, slot, kl);
                    mma_commit(&empty_bar[slot]);
                }
                it += kDownAhead;
                for (int kl = kDownAhead; ok && kl < kDownKBlocksPerTile; ++kl, ++it) {
                    const int slot = it % kDownStages;
                    const uint32_t ph = (it / kDownStages) & 1;
                    if (!mbar_wait(&full_bar[slot], ph, &abort_flag, status)) { ok = false; break; }
                    tc_fence_after();
                    issue_half(0, slot, kl);
                    issue_half(1, slot, kl);
                    mma_commit(&empty_bar[slot]);
                }
                if (!ok) break;
                mma_commit(&acc_full);
            }
        }
    } else if (warp < 10) {
        // 8 converter warps produce A: a thread takes token row m and half kh of each
        // K block (16 columns); warps 2-5 take the first halves of rows 32 (w % 4) +
        // lane, warps 6-9 the second
        const int m = (warp & 3) * 32 + lane;
        const int kh = (warp - 2) >> 2;
        // this row's 16-byte pieces 2 kh and 2 kh + 1 in a 64-byte-swizzled tile
        const uint32_t a_off = (m >> 3) * 512 + (m & 7) * 64;
        const uint32_t a_c0 = ((2 * kh) ^ ((m >> 1) & 3)) << 4, a_c1 = ((2 * kh + 1) ^ ((m >> 1) & 3)) << 4;
        int it = 0;
        for (int lt = 0; !abort_flag; ++lt) {
            const int tile = take_tile(lt, true);
            if (tile >= n_tiles) break;
            const int tt = tile / (kStreams * kDownKSplit);
            const int s = (tile / kDownKSplit) % kStreams, kq = tile % kDownKSplit;
            const int t = tt * kTileM + m;
            const bool valid = t < T;
            // sums of squares of the row's four column quads in this K half, each
            // accumulated over the tile's K blocks
            float ss[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) ss[j] = 0.f;
            // w_norm of this thread's 16 columns, loaded one K block ahead
            const int wk0 = s * kWidth + kq * kDownKBlocksPerTile * kDownBK + 16 * kh;
            uint4 wv_next[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
            if (HC_IN_RANGE(wk0, 16, kCols, status)) {
                wv_next[0] = *reinterpret_cast<const uint4*>(w_norm + wk0);
                wv_next[1] = *reinterpret_cast<const uint4*>(w_norm + wk0 + 8);
            }
            bool ok = true;
            for (int kb = kq * kDownKBlocksPerTile; kb < (kq + 1) * kDownKBlocksPerTile; ++kb, ++it) {
                const int slot = it % kDownStages, rs = it % kDownRSlots;
                const int k = s * kWidth + kb * kDownBK + 16 * kh;
                // P straight from global memory, issued before the wait
                float4 p[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) p[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (P != nullptr && valid && HC_IN_RANGE((size_t)t * kCols + k, 16, (size_t)T * kCols, status)) {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        p[j] = *reinterpret_cast<const float4*>(P + (size_t)t * kCols + k + 4 * j);
                }
                const uint4 wv[2] = {wv_next[0], wv_next[1]};
                if (kb + 1 < (kq + 1) * kDownKBlocksPerTile && HC_IN_RANGE(k + kDownBK, 16, kCols, status)) {
                    wv_next[0] = *reinterpret_cast<const uint4*>(w_norm + k + kDownBK);
                    wv_next[1] = *reinterpret_cast<const uint4*>(w_norm + k + kDownBK + 8);
                }
                if (!mbar_wait(&r_full[rs], (it / kDownRSlots) & 1, &abort_flag, status)) {
                    ok = false;
                    break;
                }
                // this row's 16 R values: 16-byte chunks 4 kh .. 4 kh + 3 of its 128-byte
                // row, each at its swizzled place
                float4 x[4];
                const uint8_t* rrow = sR(rs) + m * 128;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    x[j] = *reinterpret_cast<const float4*>(rrow + (((4 * kh + j) ^ (m & 7)) << 4));
                // R + P in that order: the pending write's single rounding
                if (P != nullptr) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        x[j].x = x[j].x + p[j].x; x[j].y = x[j].y + p[j].y;
                        x[j].z = x[j].z + p[j].z; x[j].w = x[j].w + p[j].w;
                    }
                }
                uint32_t hi[8], mid[8], low[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 r = x[j];
                    float sq = r.x * r.x;
                    sq = fmaf(r.y, r.y, sq);
                    sq = fmaf(r.z, r.z, sq);
                    sq = fmaf(r.w, r.w, sq);
                    ss[j] += sq;
                    const uint32_t wa = j < 2 ? (j == 0 ? wv[0].x : wv[0].z) : (j == 2 ? wv[1].x : wv[1].z);
                    const uint32_t wb = j < 2 ? (j == 0 ? wv[0].y : wv[0].w) : (j == 2 ? wv[1].y : wv[1].w);
                    // by truncation: exact, and cheaper than rounding
                    split3_trunc(r.x * bf16_lo(wa), r.y * bf16_hi(wa), hi[2 * j], mid[2 * j], low[2 * j]);
                    split3_trunc(r.z * bf16_lo(wb), r.w * bf16_hi(wb), hi[2 * j + 1], mid[2 * j + 1],
                                 low[2 * j + 1]);
                }
                // the R slot is handed back only now that its values have been used: the
                // TMA refill (async proxy) must not overtake these shared loads, and the
                // proxy fence orders them before it
                fence_proxy_async_smem();
                mbar_arrive(&r_empty[rs]);
                // the stage's previous MMAs are done with its A tiles
                if (!mbar_wait(&empty_bar[slot], ((it / kDownStages) & 1) ^ 1, &abort_flag, status)) {
                    ok = false;
                    break;
                }
                uint8_t* ahi = sA(slot, 0) + a_off;
                uint8_t* amid = sA(slot, 1) + a_off;
                uint8_t* alow = sA(slot, 2) + a_off;
                *reinterpret_cast<uint4*>(ahi + a_c0) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(ahi + a_c1) = make_uint4(hi[4], hi[5], hi[6], hi[7]);
                *reinterpret_cast<uint4*>(amid + a_c0) = make_uint4(mid[0], mid[1], mid[2], mid[3]);
                *reinterpret_cast<uint4*>(amid + a_c1) = make_uint4(mid[4], mid[5], mid[6], mid[7]);
                *reinterpret_cast<uint4*>(alow + a_c0) = make_uint4(low[0], low[1], low[2], low[3]);
                *reinterpret_cast<uint4*>(alow + a_c1) = make_uint4(low[4], low[5], low[6], low[7]);
                fence_proxy_async_smem();
                mbar_arrive(&full_bar[slot]);
            }
            if (!ok) break;
            // the row's sum of squares over this K half, ((q0 + q1) + (q2 + q3)); the
            // epilogue adds the two halves. The buffer of this parity was last read by
            // the epilogue two tiles ago, before it released that tile's second
            // half-buffer; this tile's MMAs, which the conversions run at most four
            // stages (of a tile's twenty K blocks) ahead of, waited for that release.
            ss_s[lt & 1][kh][m] = (ss[0] + ss[1]) + (ss[2] + ss[3]);
            mbar_arrive(&ss_full[lt & 1]);
        }
    } else {
        // 4 epilogue warps: TMEM lane quarter q = rows q*32..q*32+31, all 320 columns;
        // store this quarter's partial dots and its sums of squares
        const int q = warp & 3;
        const int m = q * 32 + lane;
        for (int lt = 0; !abort_flag; ++lt) {
            const int tile = take_tile(lt, true);
            if (tile >= n_tiles) break;
            const int tt = tile / (kStreams * kDownKSplit);
            const int s = (tile / kDownKSplit) % kStreams, kq = tile % kDownKSplit;
            const int t = tt * kTileM + m;
            const bool valid = t < T;
            if (!__all_sync(0xffffffffu, mbar_wait(&acc_full, lt & 1, &abort_flag, status))) break;
            tc_fence_after();
            const size_t prow = ((size_t)tt * kStreams + s) * kDownKSplit + kq;
            // the sums of squares first: the converters finished them before the last
            // MMA of the tile, and their buffer is rewritten two tiles later, which
            // cannot start before this tile's second half is drained below
            if (!__all_sync(0xffffffffu, mbar_wait(&ss_full[lt & 1], (lt >> 1) & 1, &abort_flag, status)))
                break;
            if (valid && HC_IN_RANGE(prow * kTileM + m, 1, (size_t)n_tiles * kTileM, status))
                ssq[prow * kTileM + m] = ss_s[lt & 1][0][m] + ss_s[lt & 1][1][m];
            // column quads, token-minor: [tile][stream][quarter][column / 4][128 tokens]
            // [4 columns], so a lane stores 16 bytes and a warp 512 contiguous bytes;
            // each half-buffer is released as soon as it has been read
            float4* dst = reinterpret_cast<float4*>(partials + prow * kRank * kTileM) + m;
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                const int hb = (2 * lt + h) % kDownHalfBufs;
#pragma unroll 1
                for (int c0 = 0; c0 < kDownHalf; c0 += 32) {
                    float v[32];
                    tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + hb * kDownHalf + c0, v);
                    if (valid) {
                        const int cq = (h * kDownHalf + c0) / 4;
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            if (HC_IN_RANGE(prow * kRank * kTileM + 4 * ((size_t)(cq + i) * kTileM + m), 4,
                                            (size_t)n_tiles * kRank * kTileM, status))
                                dst[(cq + i) * kTileM] =
                                    make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                    }
                }
                tc_fence_before();
                mbar_arrive(&acc_empty[hb]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (threadIdx.x == 0) {
        // every fetch of this CTA has returned its tile (the fetch loop ended on the
        // value it returned), so no fetch of this CTA can be performed after this
        // count; the last CTA to count resets the pair for the next launch
        if (atomicAdd(sched + 1, 1) == (int)gridDim.x - 1) {
            atomicExch(sched, 0);
            atomicExch(sched + 1, 0);
        }
    }
}

// ---------------------------------------------------------------------------
// lo = sum over the streams (in order) of rs times the sum of the stream's quarter
// partials (in order); stored as three bf16 terms [3][max_tokens][320] (hi, mid,
// low; the bf16-lo mode of the up tile reads hi alone, which is lo rounded once to
// bf16, nearest even). The partials come tile-blocked, in column quads, token-minor ([tile][stream]
// [quarter][column / 4][128 tokens][4 columns]). A CTA takes one tile's 128 tokens
// and 32 of the columns (8 quads): for each (stream, quarter) these are 16 KB in one
// piece, and a lane reads one token's quad, a warp 512 contiguous bytes; shared
// memory turns the block around so that each token's 32 columns leave as whole
// 32-byte sectors.
// ---------------------------------------------------------------------------
constexpr int kLoCols = 32;
// 8 warps, four (token, column quad) pairs a thread: 8 CTAs fit on an SM, so an 8K
// read's 640 CTAs run in one wave (with 512 threads a CTA, 1.05 waves: 8K read 0.381
// -> 0.376 ms)
constexpr int kLoThreads = 256;
constexpr int kLoPairs = kTileM * (kLoCols / 4) / kLoThreads;

__global__ void __launch_bounds__(kLoThreads)
lo_split_kernel(const float* __restrict__ partials, const float* __restrict__ ssq,
                uint16_t* __restrict__ lo3, int T, int max_tokens, float eps, int* status) {
    // extents (floats) of the partials and sums of squares of this call's tiles
    const size_t n_rows = (size_t)((T + kTileM - 1) / kTileM) * kStreams * kDownKSplit;
    (void)n_rows;
    // the up tile after it (launched with programmatic dependent launch inside a read)
    // may start its prologue, R stream and weight loads now; it waits for this grid
    // before it loads lo
    pdl_launch_dependents();
    __shared__ float lo_s[kTileM][kLoCols + 1];
    __shared__ float rs_s[kStreams][kTileM];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tt = blockIdx.x / (kRank / kLoCols), cg = blockIdx.x % (kRank / kLoCols);
    const size_t base = (size_t)tt * kStreams * kDownKSplit;   // first (stream, quarter) row
    // rs of the tile's tokens: warps 0-3 take a token quarter each
    if (warp < 4) {
        const int tr = warp * 32 + lane;
        const bool valid = tt * kTileM + tr < T;
#pragma unroll
        for (int s = 0; s < kStreams; ++s) {
            float ss = 0.f;
            const size_t qi = (base + (size_t)s * kDownKSplit) * kTileM + tr;
            if (valid && HC_IN_RANGE(qi + (size_t)(kDownKSplit - 1) * kTileM, 1, n_rows * kTileM, status)) {
                const float* q4 = ssq + qi;
                ss = q4[0];
#pragma unroll
                for (int q = 1; q < kDownKSplit; ++q) ss += q4[q * kTileM];
            }
            rs_s[s][tr] = inv_rms(fmaf(ss, 1.0f / (float)kWidth, eps));
        }
    }
    __syncthreads();
    // a thread takes (token, column quad) pairs: tokens across the lanes, so each load
    // instruction of a warp reads 512 contiguous bytes
#pragma unroll
    for (int i = 0; i < kLoPairs; ++i) {
        const int pidx = threadIdx.x + i * kLoThreads;
        const int tr = pidx & (kTileM - 1), jq = pidx >> 7;     // token, quad 0..7
        const float4* p = reinterpret_cast<const float4*>(partials) +
                          (base * (kRank / 4) + (size_t)cg * (kLoCols / 4) + jq) * kTileM + tr;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s = 0; s < kStreams; ++s) {
            const float4* ps = p + (size_t)s * kDownKSplit * (kRank / 4) * kTileM;
            const size_t last = 4 * (size_t)(ps + (size_t)(kDownKSplit - 1) * (kRank / 4) * kTileM -
                                             reinterpret_cast<const float4*>(partials));
            (void)last;
            float4 d = make_float4(0.f, 0.f, 0.f, 0.f);
            if (HC_IN_RANGE(last, 4, n_rows * kRank * kTileM, status)) {
                d = ps[0];
#pragma unroll
                for (int q = 1; q < kDownKSplit; ++q) {
                    const float4 w = ps[(size_t)q * (kRank / 4) * kTileM];
                    d.x += w.x; d.y += w.y; d.z += w.z; d.w += w.w;
                }
            }
            const float r = rs_s[s][tr];
            v[0] = fmaf(r, d.x, v[0]);
            v[1] = fmaf(r, d.y, v[1]);
            v[2] = fmaf(r, d.z, v[2]);
            v[3] = fmaf(r, d.w, v[3]);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) lo_s[tr][4 * jq + k] = v[k];
    }
    __syncthreads();
    // out: each token's 32 columns, 4 per lane, 8 lanes per token, 4 tokens per warp
    // and pass
    for (int r = warp * 4 + (lane >> 3); r < kTileM; r += (kLoThreads / 32) * 4) {
        const int trow = tt * kTileM + r;
        if (trow >= T) continue;
        const int c4 = 4 * (lane & 7);
        const float x0 = lo_s[r][c4], x1 = lo_s[r][c4 + 1], x2 = lo_s[r][c4 + 2], x3 = lo_s[r][c4 + 3];
        const size_t off = (size_t)trow * kRank + cg * kLoCols + c4;
        const size_t term = (size_t)max_tokens * kRank;
        if (!HC_IN_RANGE(2 * term + off, 4, 3 * term, status)) continue;
        uint32_t h0, m0, l0, h1, m1, l1;
        split3_bf16(x0, x1, h0, m0, l0);
        split3_bf16(x2, x3, h1, m1, l1);
        *reinterpret_cast<uint2*>(lo3 + off) = make_uint2(h0, h1);
        *reinterpret_cast<uint2*>(lo3 + term + off) = make_uint2(m0, m1);
        *reinterpret_cast<uint2*>(lo3 + 2 * term + off) = make_uint2(l0, l1);
    }
}

// ---------------------------------------------------------------------------
// up projection + gate (+ mix), one (128-token tile, 64 columns x 4 streams) per
// tile, persistent CTAs, two TMEM accumulators so the epilogue of one tile runs
// under the MMAs of the next. The epilogue's global traffic goes through TMA: R
// (and P) tiles are loaded into per-warp staging and the outputs are stored from it,
// so every transfer is a whole tile of 32-byte rows instead of scattered words.
// ---------------------------------------------------------------------------
struct EpiMaps {
    CUtensorMap R, P;
    CUtensorMap out;   // out_f32 in boxes of 8 columns x 1 stream x 32 tokens (mix only)
};

// kOut: what the epilogue writes. kOutGated: gated (fp32, the unfused pair's first
// half); kOutMix: the 4x4 mix with the bf16/fp16 images; kOutY: the 2560-wide
// read-out y[c] = sum_s gated[s][c] (streams in order) with its images.
// kLoTerms = 3: A is lo as its three bf16 terms (fp32-accurate); kLoTerms = 1: A is
// the first term alone, lo rounded once to bf16 (one MMA per step). B is the caller's
// bf16 W_up as stored in both.
constexpr int kOutGated = 0, kOutMix = 1, kOutY = 2;
template <int kOut, int kLoTerms>
__global__ void __launch_bounds__(kUpThreads, 1)
upmix_tile_kernel(const float* __restrict__ Rmix, const __grid_constant__ CUtensorMap tm_lo,
                  const __grid_constant__ CUtensorMap tm_wu, const __grid_constant__ EpiMaps em,
                  float* __restrict__ out_f32, uint16_t* __restrict__ out_bf16,
                  uint16_t* __restrict__ out_fp16, int has_P, int T, int* __restrict__ status,
                  int* __restrict__ sched, int pdl) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    __shared__ __align__(8) uint64_t full_bar[kUpStages], empty_bar[kUpStages];
    __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2];
    __shared__ __align__(8) uint64_t r_full[kRSlots], r_empty[kRSlots];
    __shared__ __align__(8) uint64_t tq_full[kTileQ], tq_empty[kTileQ];
    __shared__ int tile_q[kTileQ];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles = ((T + kTileM - 1) / kTileM) * kUpColTiles;
    constexpr int kSteps = kUpCols / kEpiCols;   // 8 epilogue steps per tile
    constexpr int kOutStreams = kOut == kOutY ? 1 : kStreams;   // output rows per token
    // the mix writes its fp32 rows back into the step's R slot, in place of R, and
    // stores them from there by TMA (one 1 KB box per stream and warp); the slot is
    // released once that store has read it
    constexpr bool kTmaOut = kOut == kOutMix;
    constexpr size_t kRowStride = kOut == kOutY ? kWidth : kCols;   // output floats per token
    // with a pending write a step needs two slots (R, then P)
    const int slots_per_step = has_P ? 2 : 1;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kUpStages; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 32 * kUpEpiWarps);
        }
        // each step is taken by one group of four epilogue warps
        for (int i = 0; i < kRSlots; ++i) {
            mbar_init(&r_full[i], 1);
            mbar_init(&r_empty[i], 4);
        }
        for (int i = 0; i < kTileQ; ++i) {
            mbar_init(&tq_full[i], 1);
            mbar_init(&tq_empty[i], kTileQConsumers);
        }
        abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(&tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    auto sA = [&](int slot, int term) { return smem + slot * kUpStageBytes + term * kUpTileBytes; };
    auto sB = [&](int slot) { return smem + slot * kUpStageBytes + kTerms * kUpTileBytes; };
    uint8_t* rring = smem + kUpStages * kUpStageBytes;
    // the CTA's i-th tile from the queue (n_tiles: no more tiles, or the CTA gave up)
    auto take_tile = [&](int i) -> int {
        if (!mbar_wait(&tq_full[i % kTileQ], (i / kTileQ) & 1, &abort_flag, status)) return n_tiles;
        return tile_q[i % kTileQ];
    };

    if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kUpRegsLow));
    if (warp == 0) {
        // operand producer: lo terms and W_up rows, K blocks of 64
        if (lane == 0) {
            // lo and W_up tiles are read again by the other CTAs of their token and
            // column tiles: keep them in L2 (evict_last) against the stream of R and
            // outputs. R and the outputs keep the default policy: a 32-byte box row
            // shares its 128-byte line with the next three steps, which find it in L2.
            const uint64_t keep = l2_policy_evict_last();
            // launched with programmatic dependent launch (inside a read, after lo_split):
            // W_up and R were final before lo_split started, lo only once it has ended
            bool lo_ready = !pdl;
            int it = 0;
            for (int i = 0; !abort_flag; ++i) {
                // fetch the next tile and publish it to the other roles
                if (!mbar_wait(&tq_empty[i % kTileQ], ((i / kTileQ) & 1) ^ 1, &abort_flag, status)) break;
                const int tile = i == 0 ? (int)blockIdx.x : (int)gridDim.x + atomicAdd(sched, 1);
                tile_q[i % kTileQ] = tile;
                mbar_arrive(&tq_full[i % kTileQ]);
                if (tile >= n_tiles) break;
                const int tt = tile / kUpColTiles, ct = tile % kUpColTiles;
                for (int kb = 0; kb < kUpKBlocks; ++kb, ++it) {
                    const int slot = it % kUpStages;
                    const uint32_t ph = (it / kUpStages) & 1;
                    if (!mbar_wait(&empty_bar[slot], ph ^ 1, &abort_flag, status)) break;
                    mbar_arrive_expect_tx(&full_bar[slot], kLoTerms * kUpTileBytes + kUpBBytes);
#pragma unroll
                    for (int s = 0; s < kStreams; ++s)
                        tma_load_2d_hint(sB(slot) + s * (kUpBBytes / kStreams), &tm_wu, kb * kUpBK,
                                         s * kWidth + ct * kUpCols, &full_bar[slot], keep);
                    if (!lo_ready) {
                        pdl_wait();
                        // lo was written by lo_split's ordinary stores; TMA reads it
                        asm volatile("fence.proxy.async.global;" ::: "memory");
                        lo_ready = true;
                    }
#pragma unroll
                    for (int term = 0; term < kLoTerms; ++term)
                        tma_load_3d_hint(sA(slot, term), &tm_lo, kb * kUpBK, tt * kTileM, term,
                                         &full_bar[slot], keep);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kTileM, kUpN);
            int it = 0;
            for (int lt = 0; !abort_flag; ++lt) {
                const int tile = take_tile(lt);
                mbar_arrive(&tq_empty[lt % kTileQ]);
                if (tile >= n_tiles) break;
                const int b = lt & 1;
                if (!mbar_wait(&acc_empty[b], ((lt >> 1) & 1) ^ 1, &abort_flag, status)) break;
                tc_fence_after();
                bool ok = true;
                for (int kb = 0; kb < kUpKBlocks; ++kb, ++it) {
                    const int slot = it % kUpStages;
                    const uint32_t ph = (it / kUpStages) & 1;
                    if (!mbar_wait(&full_bar[slot], ph, &abort_flag, status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t b0 = smem_u32(sB(slot));
#pragma unroll
                    for (int term = 0; term < kLoTerms; ++term) {
                        const uint32_t a0 = smem_u32(sA(slot, term));
#pragma unroll
                        for (int kk = 0; kk < kUpBK / 16; ++kk)
                            mma_f16(tmem + b * kUpN, desc_sw64(a0 + kk * 32),
                                    desc_sw64(b0 + kk * 32), idesc, (kb | term | kk) != 0);
                    }
                    mma_commit(&empty_bar[slot]);
                }
                if (!ok) break;
                mma_commit(&acc_full[b]);
            }
        }
    } else {
        // R (and P) producers, warp 2 for epilogue group 0 and warp 3 for group 1:
        // one slot of the group's ring per step (two with P), 4 streams per slot, in
        // the group's step order {2g, 2g+1, 4+2g, 5+2g}
        const int rg = warp - 2;
        if (lane == 0) {
            int u = 0;   // uses of this group's ring
            for (int i = 0; !abort_flag; ++i) {
                const int tile = take_tile(i);
                mbar_arrive(&tq_empty[i % kTileQ]);
                if (tile >= n_tiles) break;
                const int tt = tile / kUpColTiles, ct = tile % kUpColTiles;
                for (int sg = 0; sg < kSteps / 2; ++sg) {
                    const int k = 4 * (sg >> 1) + 2 * rg + (sg & 1);
                    for (int which = 0; which < slots_per_step; ++which, ++u) {
                        const int slot = rg * kRSlotsPerGroup + u % kRSlotsPerGroup;
                        if (!mbar_wait(&r_empty[slot], ((u / kRSlotsPerGroup) & 1) ^ 1, &abort_flag,
                                       status))
                            break;
                        mbar_arrive_expect_tx(&r_full[slot], kRSlot);
                        const CUtensorMap* map = which ? &em.P : &em.R;
#pragma unroll
                        for (int s = 0; s < kStreams; ++s)
                            tma_load_3d(rring + slot * kRSlot + s * (kRSlot / kStreams), map,
                                        ct * kUpCols + k * kEpiCols, s, tt * kTileM, &r_full[slot]);
                    }
                }
            }
        }
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kUpRegsHigh));
        // epilogue warp: TMEM lane quarter q = tokens q*32..q*32+31 of the tile; group
        // g takes the step pairs {2g, 2g+1} and {4+2g, 5+2g}
        const int ew = warp - 4, q = warp & 3, g = ew >> 2;
        const int row = q * kEpiRows + lane;         // this lane's token within the tile
        for (int lt = 0; !abort_flag; ++lt) {
            const int tile = take_tile(lt);
            __syncwarp();
            if (lane == 0) mbar_arrive(&tq_empty[lt % kTileQ]);
            if (tile >= n_tiles) break;
            const int tt = tile / kUpColTiles, ct = tile % kUpColTiles;
            const int b = lt & 1;
            const int t = tt * kTileM + row;
            const bool valid = t < T;
            float mx[16];
            if (kOut == kOutMix) {
                if (valid && HC_IN_RANGE((size_t)t * 16, 16, (size_t)T * 16, status)) {
                    const float4* m4 = reinterpret_cast<const float4*>(Rmix + (size_t)t * 16);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float4 v = m4[i];
                        mx[4 * i] = v.x; mx[4 * i + 1] = v.y; mx[4 * i + 2] = v.z; mx[4 * i + 3] = v.w;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) mx[i] = 0.f;
                }
            }
            if (!mbar_wait(&acc_full[b], (lt >> 1) & 1, &abort_flag, status)) break;
            tc_fence_after();
            const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) + b * kUpN;
            const int u_tile = lt * (kSteps / 2) * slots_per_step;   // uses of group g's ring
            bool ok = true;
#pragma unroll 1
            for (int pi = 0; pi < 2 && ok; ++pi) {
                const int k0 = 4 * pi + 2 * g;
                uint32_t bb[kOutStreams][8], hh[kOutStreams][8];   // 16 columns of the images
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int k = k0 + j;
                    const int c = ct * kUpCols + k * kEpiCols;
                    float v[kStreams][kEpiCols];
                    tmem_ld8x4<kUpCols>(tbase + k * kEpiCols, v);
                    // R' of this lane's token: slot layout [stream][128 tokens][8 columns]
                    float rp[kStreams][kEpiCols];
                    int rslot = 0;
                    for (int which = 0; which < slots_per_step; ++which) {
                        const int u = u_tile + (2 * pi + j) * slots_per_step + which;
                        const int slot = g * kRSlotsPerGroup + u % kRSlotsPerGroup;
                        if (which == 0) rslot = slot;
                        if (!mbar_wait(&r_full[slot], (u / kRSlotsPerGroup) & 1, &abort_flag, status)) {
                            ok = false;
                            break;
                        }
#pragma unroll
                        for (int s = 0; s < kStreams; ++s) {
                            const float4* r4 = reinterpret_cast<const float4*>(
                                rring + slot * kRSlot + s * (kRSlot / kStreams) + row * 32);
                            const float4 a = r4[0], bq = r4[1];
                            const float x[8] = {a.x, a.y, a.z, a.w, bq.x, bq.y, bq.z, bq.w};
#pragma unroll
                            for (int e = 0; e < kEpiCols; ++e) rp[s][e] = which ? rp[s][e] + x[e] : x[e];
                        }
                        // the next fill of this slot is a TMA write (async proxy): a slot
                        // released right after these reads orders them before it with a
                        // proxy fence. (The mix's R slot is released later, after the TMA
                        // store of the outputs written into it, behind the fence that
                        // precedes that store.)
                        const bool release_now = !(kTmaOut && which == 0);
                        if (release_now) fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0 && release_now) mbar_arrive(&r_empty[slot]);
                    }
                    if (!ok) break;
#pragma unroll
                    for (int s = 0; s < kStreams; ++s)
#pragma unroll
                        for (int e = 0; e < kEpiCols; ++e) v[s][e] = gate_value(v[s][e], rp[s][e]);
#pragma unroll
                    for (int so = 0; so < kOutStreams; ++so) {
                        float o[kEpiCols];
#pragma unroll
                        for (int e = 0; e < kEpiCols; ++e) {
                            if (kOut == kOutMix)
                                o[e] = mix_row(&mx[so * 4], v[0][e], v[1][e], v[2][e], v[3][e]);
                            else if (kOut == kOutY)
                                o[e] = ((v[0][e] + v[1][e]) + v[2][e]) + v[3][e];
                            else
                                o[e] = v[so][e];
                        }
                        if (kTmaOut) {
                            float4* f4 = reinterpret_cast<float4*>(
                                rring + rslot * kRSlot + so * (kRSlot / kStreams) + row * 32);
                            f4[0] = make_float4(o[0], o[1], o[2], o[3]);
                            f4[1] = make_float4(o[4], o[5], o[6], o[7]);
                        } else {
                            uint32_t w[8];
#pragma unroll
                            for (int e = 0; e < kEpiCols; ++e) w[e] = __float_as_uint(o[e]);
                            if (valid && HC_IN_RANGE((size_t)t * kRowStride + so * kWidth + c, 8,
                                                     (size_t)T * kRowStride, status))
                                st_global_v8(out_f32 + (size_t)t * kRowStride + so * kWidth + c, w);
                        }
                        if (kOut != kOutGated) {
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                bb[so][4 * j + i] = pack_bf16x2(o[2 * i], o[2 * i + 1]);
                                hh[so][4 * j + i] = pack_f16x2(o[2 * i], o[2 * i + 1]);
                            }
                        }
                    }
                    if (kTmaOut) {
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            const int t0 = tt * kTileM + q * kEpiRows;
#pragma unroll
                            for (int so = 0; so < kStreams; ++so)
                                tma_store_3d(&em.out, c, so, t0,
                                             rring + rslot * kRSlot + so * (kRSlot / kStreams) +
                                                 q * kEpiRows * 32);
                            bulk_commit();
                            bulk_wait_read_all();   // the slot may be refilled after this
                            mbar_arrive(&r_empty[rslot]);
                        }
                        __syncwarp();
                    }
                }
                if (!ok) break;
                if (kOut != kOutGated && valid) {
                    const size_t off = (size_t)t * kRowStride + ct * kUpCols + k0 * kEpiCols;
#pragma unroll
                    for (int so = 0; so < kOutStreams; ++so) {
                        if (!HC_IN_RANGE(off + so * kWidth, 16, (size_t)T * kRowStride, status)) continue;
                        st_global_v8(out_bf16 + off + so * kWidth, bb[so]);
                        st_global_v8(out_fp16 + off + so * kWidth, hh[so]);
                    }
                }
            }
            if (!ok) break;
            tc_fence_before();
            mbar_arrive(&acc_empty[b]);
        }
        if (kTmaOut && lane == 0) bulk_wait_all();   // outputs written before the CTA exits
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (threadIdx.x == 0) {
        // every fetch of this CTA has returned its tile (the fetch loop ended on the
        // value it returned), so no fetch of this CTA can be performed after this
        // count; the last CTA to count resets the pair for the next launch
        if (atomicAdd(sched + 1, 1) == (int)gridDim.x - 1) {
            atomicExch(sched, 0);
            atomicExch(sched + 1, 0);
        }
    }
}

// The mix of the unfused pair: reads gated back and applies the same 4x4 mix.
__global__ void mix_gated_kernel(const float* __restrict__ gated, const float* __restrict__ Rmix,
                                 float* __restrict__ out_f32, uint16_t* __restrict__ out_bf16,
                                 uint16_t* __restrict__ out_fp16, int T, int* status) {
    const int per_tok = kWidth / 4;
    const int n = T * per_tok;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const int t = i / per_tok, c = 4 * (i % per_tok);
        // every access of this element group lies in token t's rows
        if (!HC_IN_RANGE((size_t)t * kCols + 3 * kWidth + c, 4, (size_t)T * kCols, status) ||
            !HC_IN_RANGE((size_t)t * 16, 16, (size_t)T * 16, status))
            continue;
        float mx[16];
        const float4* m4 = reinterpret_cast<const float4*>(Rmix + (size_t)t * 16);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float4 v = m4[k];
            mx[4 * k] = v.x; mx[4 * k + 1] = v.y; mx[4 * k + 2] = v.z; mx[4 * k + 3] = v.w;
        }
        float g[kStreams][4];
#pragma unroll
        for (int s = 0; s < kStreams; ++s) {
            const float4 v = *reinterpret_cast<const float4*>(gated + (size_t)t * kCols + s * kWidth + c);
            g[s][0] = v.x; g[s][1] = v.y; g[s][2] = v.z; g[s][3] = v.w;
        }
#pragma unroll
        for (int so = 0; so < kStreams; ++so) {
            float o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) o[e] = mix_row(&mx[so * 4], g[0][e], g[1][e], g[2][e], g[3][e]);
            const size_t off = (size_t)t * kCols + so * kWidth + c;
            *reinterpret_cast<float4*>(out_f32 + off) = make_float4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint2*>(out_bf16 + off) =
                make_uint2((uint32_t)to_bf16_bits(o[0]) | ((uint32_t)to_bf16_bits(o[1]) << 16),
                           (uint32_t)to_bf16_bits(o[2]) | ((uint32_t)to_bf16_bits(o[3]) << 16));
            *reinterpret_cast<uint2*>(out_fp16 + off) =
                make_uint2((uint32_t)to_fp16_bits(o[0]) | ((uint32_t)to_fp16_bits(o[1]) << 16),
                           (uint32_t)to_fp16_bits(o[2]) | ((uint32_t)to_fp16_bits(o[3]) << 16));
        }
    }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool encode_map(CUtensorMap* map, CUtensorMapDataType dt, const void* base, int rank,
                const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                CUtensorMapSwizzle swz) {
    auto enc = get_encoder();
    if (enc == nullptr) return false;
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return enc(map, dt, rank, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A [T][4][2560] activation or output tensor seen as 3D (c, stream, token), in tiles
// of `cols` columns x 1 stream x `rows` tokens (TMA clips and zero-fills past T).
bool encode_act(CUtensorMap* map, CUtensorMapDataType dt, int esize, const void* base, int T,
                int cols, int rows) {
    const cuuint64_t dims[3] = {kWidth, kStreams, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)kWidth * esize, (cuuint64_t)kCols * esize};
    const cuuint32_t box[3] = {(cuuint32_t)cols, 1, (cuuint32_t)rows};
    return encode_map(map, dt, base, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// R [T][4][2560] fp32 seen as (column, stream, token), in boxes of 32 columns x 1
// stream x 128 tokens, 128-byte swizzled (a box row is 128 bytes); TMA zero-fills the
// rows past T of a last partial tile.
bool encode_down_r(CUtensorMap* map, const float* R, int T) {
    const cuuint64_t dims[3] = {kWidth, kStreams, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)kWidth * 4, (cuuint64_t)kCols * 4};
    const cuuint32_t box[3] = {kDownBK, 1, kTileM};
    return encode_map(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, R, 3, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B);
}

// The caller's W_down [kRank][kCols] bf16 in boxes of 32 K x 160 rows, 64-byte
// swizzled: one N half of a down tile's B operand per box.
bool encode_w_down_bf16(CUtensorMap* map, const uint16_t* W_down) {
    const cuuint64_t dims[2] = {kCols, kRank};
    const cuuint64_t strides[1] = {kCols * 2};
    const cuuint32_t box[2] = {kDownBK, kDownN / 2};
    return encode_map(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W_down, 2, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_64B);
}

// The caller's W_up [kCols][kRank] bf16 in boxes of 32 K x 64 rows, 64-byte swizzled:
// one stream's part of an up tile's B operand per box.
bool encode_w_up_sw64(CUtensorMap* map, const uint16_t* W_up) {
    const cuuint64_t dims[2] = {kRank, kCols};
    const cuuint64_t strides[1] = {kRank * 2};
    const cuuint32_t box[2] = {kUpBK, kUpCols};
    return encode_map(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W_up, 2, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_64B);
}

}  // namespace

bool encode_w_up_bf16(CUtensorMap* map, const uint16_t* W_up, int box_rows) {
    const cuuint64_t dims[2] = {kRank, kCols};
    const cuuint64_t strides[1] = {kRank * 2};
    const cuuint32_t box[2] = {kBK, (cuuint32_t)box_rows};
    return encode_map(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W_up, 2, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B);
}

cudaError_t prefill_setup(Ctx& c) {
    // lo's three bf16 terms [3][max_tokens][kRank] in the library's scratch: the up
    // tile's A operand, in boxes of 32 K x 128 tokens x 1 term, 64-byte swizzled (fixed
    // for the context)
    {
        const cuuint64_t dims[3] = {kRank, (cuuint64_t)c.max_tokens, kTerms};
        const cuuint64_t strides[2] = {kRank * 2, (cuuint64_t)c.max_tokens * kRank * 2};
        const cuuint32_t box[3] = {kUpBK, kTileM, 1};
        if (!encode_map(&c.tm_lo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c.lo3, 3, dims, strides, box,
                        CU_TENSOR_MAP_SWIZZLE_64B))
            return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(down_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kDownSmem);
    if (e != cudaSuccess) return e;
    // the register split of the up tile assumes the launch register count it was
    // written for: refuse to run a build whose count differs (the epilogue's
    // setmaxnreg.inc would wait for registers that are never given up)
    const void* ks[] = {reinterpret_cast<const void*>(upmix_tile_kernel<kOutMix, kTerms>),
                        reinterpret_cast<const void*>(upmix_tile_kernel<kOutMix, 1>),
                        reinterpret_cast<const void*>(upmix_tile_kernel<kOutY, kTerms>),
                        reinterpret_cast<const void*>(upmix_tile_kernel<kOutGated, kTerms>)};
    for (const void* k : ks) {
        cudaFuncAttributes fa;
        if ((e = cudaFuncGetAttributes(&fa, k)) != cudaSuccess) return e;
        if (fa.numRegs != kUpRegsLaunch) return cudaErrorInvalidConfiguration;
        if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kUpSmem)) !=
            cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

cudaError_t launch_prefill_down(const Ctx& c, const ReadArgs& a, cudaStream_t st) {
    const int n_tt = (a.T + kTileM - 1) / kTileM;
    const int down_tiles = n_tt * kStreams * kDownKSplit;
    const int down_grid = down_tiles < c.sm_count ? down_tiles : c.sm_count;
    CUtensorMap tm_r, tm_wd;
    if (!encode_down_r(&tm_r, a.R, a.T) || !encode_w_down_bf16(&tm_wd, a.W_down))
        return cudaErrorInvalidValue;
    // an ordinary launch: the first kernel of the read reads R and P, which the kernel
    // before it on the stream may have written
    down_tile_kernel<<<down_grid, kDownThreads, kDownSmem, st>>>(
        a.P, a.w_norm, tm_wd, tm_r, c.partials, c.ssq, a.T, c.s.status,
        c.s.sched + 2 * kSchedDown);
    const int rgrid = n_tt * (kRank / kLoCols);
    lo_split_kernel<<<rgrid, kLoThreads, 0, st>>>(c.partials, c.ssq, c.lo3, a.T, c.max_tokens,
                                                  c.eps, c.s.status);
    return cudaGetLastError();
}

namespace {
// An up tile launch, with programmatic stream serialisation when `pdl`.
template <typename... KArgs, typename... Args>
cudaError_t launch_up(void (*kernel)(KArgs...), int grid, bool pdl, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kUpThreads);
    cfg.dynamicSmemBytes = kUpSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}
}  // namespace

cudaError_t launch_prefill_upmix(const Ctx& c, const ReadArgs& a, PrefillMode mode, cudaStream_t st,
                                 bool pdl) {
    const int n_tt = (a.T + kTileM - 1) / kTileM;
    const int up_tiles = n_tt * kUpColTiles;
    const int up_grid = up_tiles < c.sm_count ? up_tiles : c.sm_count;
    EpiMaps em;
    CUtensorMap tm_wu;
    bool ok = encode_w_up_sw64(&tm_wu, a.W_up);
    ok = ok && encode_act(&em.R, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.R, a.T, kEpiCols, kTileM);
    ok = ok && encode_act(&em.P, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.P ? a.P : a.R, a.T,
                          kEpiCols, kTileM);
    // the mix's fp32 output (any [T][4][2560] fp32 tensor for the other epilogues)
    const bool mix = mode == PrefillMode::kFused || mode == PrefillMode::kFusedBf16Lo;
    ok = ok && encode_act(&em.out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, mix ? a.out_f32 : a.R, a.T,
                          kEpiCols, kEpiRows);
    if (!ok) return cudaErrorInvalidValue;
    const int has_P = a.P != nullptr;
    int* sched = c.s.sched + 2 * kSchedUp;
    cudaError_t e = cudaSuccess;
    switch (mode) {
        case PrefillMode::kFused:
            e = launch_up(upmix_tile_kernel<kOutMix, kTerms>, up_grid, pdl, st, a.Rmix, c.tm_lo,
                          tm_wu, em, a.out_f32, a.out_bf16, a.out_fp16, has_P, a.T, c.s.status,
                          sched, (int)pdl);
            break;
        case PrefillMode::kFusedBf16Lo:
            e = launch_up(upmix_tile_kernel<kOutMix, 1>, up_grid, pdl, st, a.Rmix, c.tm_lo, tm_wu,
                          em, a.out_f32, a.out_bf16, a.out_fp16, has_P, a.T, c.s.status, sched,
                          (int)pdl);
            break;
        case PrefillMode::kReadoutY:
            e = launch_up(upmix_tile_kernel<kOutY, kTerms>, up_grid, pdl, st, (const float*)nullptr,
                          c.tm_lo, tm_wu, em, a.out_f32, a.out_bf16, a.out_fp16, has_P, a.T,
                          c.s.status, sched, (int)pdl);
            break;
        case PrefillMode::kUnfused: {
            e = launch_up(upmix_tile_kernel<kOutGated, kTerms>, up_grid, pdl, st, a.Rmix, c.tm_lo,
                          tm_wu, em, c.gated, (uint16_t*)nullptr, (uint16_t*)nullptr, has_P, a.T,
                          c.s.status, sched, (int)pdl);
            if (e != cudaSuccess) return e;
            const int n = a.T * (kWidth / 4);
            const int mgrid = (n + 255) / 256 < 8 * c.sm_count ? (n + 255) / 256 : 8 * c.sm_count;
            mix_gated_kernel<<<mgrid, 256, 0, st>>>(c.gated, a.Rmix, a.out_f32, a.out_bf16,
                                                    a.out_fp16, a.T, c.s.status);
            break;
        }
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_prefill(const Ctx& c, const ReadArgs& a, PrefillMode mode, cudaStream_t st) {
    cudaError_t e = launch_prefill_down(c, a, st);
    if (e != cudaSuccess) return e;
    return launch_prefill_upmix(c, a, mode, st, true);
}

}  // namespace hc
