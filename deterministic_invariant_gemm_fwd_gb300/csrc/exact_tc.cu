// exact_tc.cu - exact tier for bf16 operands on the tensor cores.
//
// Same result as exact_kbn.cu and exact_int.cu, bit for bit: the fixed-order
// KBN sum of the float64 products (256-wide chunks left to right, chunk values
// fl(s + c) combined left to right with KBN), bias in float64, one RNE
// rounding (Carbon README, "How It Works"; sgemm-bi "Determinism contracts"
// for the downcast).
//
// Why integer sums give the literal algorithm's bits.  Over one chunk, row i
// of A is X[k] * 2^bx(i) and column j of B is W[k] * 2^bw(j) with integers
// |X| < 2^wx, |W| < 2^ww (the statistics of exact_bf16.cuh).  In the chunk's
// KBN loop every product, partial sum and correction is a multiple of
// 2^(bx + bw).  Each step's rounding error is recovered exactly (the larger
// magnitude goes first, as in Fast2Sum), and the errors also add up exactly:
// each is at most half an ulp of a partial sum below 2^(wx + ww + 8) grain
// units, so 256 of them stay below 2^(wx + ww - 37) grain units, which is
// representable while wx + ww < 90.  Then s + c equals the exact chunk sum and
// the chunk value fl(s + c) is the exact sum I * 2^(bx + bw) rounded once to
// float64.  The outer KBN over the chunk values behaves the same way (at most
// 65535 chunk values, each a multiple of the output grain), so the result
// before the bias is the exact sum of the chunk values rounded once.
//
// Chunk sums on the tensor cores.  I is computed exactly:
//  * every X is written in base-256 digits, X = sum_a d_a 256^a with
//    |d_a| <= 128: X = m * 2^s (|m| < 2^8) has two, lo = v mod 256 in
//    [-128, 127] at a = s / 8 and (v - lo) / 256 at a + 1, v = m * 2^(s % 8);
//    likewise W = sum_b e_b 256^b; a digit is an integer of at most 8
//    significant bits, so it is exact in bf16;
//  * for one digit pair (a, b) the 256 products d_a e_b are integers of
//    magnitude <= 2^14, their sum is at most 2^22 in magnitude, and the
//    tensor core accumulates it in an fp32 accumulator that starts at
//    1.5 * 2^23: every partial sum stays in [2^23, 2^24], where fp32 spacing
//    is 1, so the accumulation is exact for any order of addition, and the
//    accumulator's bit pattern minus that of 1.5 * 2^23 is the pair sum;
//  * I = sum_{a,b} 256^(a+b) (pair sum), assembled modulo 2^64: the sums of
//    B digits 2p and 2p + 1 combine exactly in 32 bits (|s + 256 s'| < 2^31,
//    the starting values taken out by one constant), then one 64-bit
//    multiply-add per combined pair; I is exact when the statistics bound
//    |I| below 2^62.
// A line of width w <= 31 needs ceil((w + 1) / 8) digits (trailing zero bits
// of the significands are moved into the exponents first, so the base is as
// high as the values allow); a tile uses the most any of its lines needs in
// the chunk, nx (1..4) A planes and nb (1..4) B planes.  One tcgen05.mma of
// M = 128, N = 64 nb, K = 16 multiplies one A digit plane of 128 rows with the
// nb B digit planes of 64 columns at once, so one "k-group" (the four K=16
// slices of each of four 64-deep blocks) yields the pair sums of nb digit
// pairs for a 128 x 64 output tile.  Rows that need four digits in some chunk
// are placed after the others within groups of 1024 rows, so that most row
// tiles get by with three.
//
// Outer sum.  The chunk values (I rounded to 53 significant bits when it is
// larger) are added exactly in the integer grain 2^(Gx(i) + Gw(j)), the
// smallest bases of row i and column j over all chunks: T += I << shift.  At
// the end T * 2^grain is rounded once to float64, the bias added in float64,
// and the result rounded once to bf16.  Outputs with a line wider than 31 bits
// (or inf/NaN), a chunk sum that may reach 2^62, or a running sum that would
// leave 2^62 go to the fix-up kernel of exact_bf16.cuh, which recomputes them
// from the operands.
//
// Structure.
//  digit_prep_kernel: one warp per (line, chunk): statistics and digit planes
//    (bf16, reduction index contiguous, the four planes of a tile's lines
//    together), the plane count per (tile, chunk) of each side.
//  exact_tc_kernel: persistent, one CTA per SM, 128 x 64 output tiles taken
//    in turn (unit u: tile u / pieces, handed out at run time; consecutive
//    tiles share the operand whose planes are the larger).
//   warps 0, 2 TMA producers of A: four stages of A plane blocks (16 KiB
//              each, one k-group), signalled in pairs, alternate loads (one
//              thread's copies complete in turn)
//   warp 3     TMA producer of B: per chunk the four B planes of each 64-deep
//              block (4 x 32 KiB, resident for the chunk), signalled in pairs;
//              it also takes the work units and posts them to the others
//   warp 1     MMA issuer: two accumulators of 256 TMEM columns used in turn,
//              one per k-group, each k-group opened by one K = 16, N = 256 MMA
//              of two constant shared-memory tiles that sets the accumulator
//              to 1.5 * 2^23 (so the epilogue never writes tensor memory, and
//              the columns of B planes a chunk does not need read as 0)
//   warps 4-11 epilogue: warp w reads lanes 32 (w % 4) .. +31 and 32 of the 64
//              output columns; adds the pair sums into per-output int64 chunk
//              sums and releases the accumulator; at each chunk end checks the
//              chunk and adds it to the outer sum; at the tile end stores the
//              exact partial sums for the finalize kernel.  Each thread keeps
//              32 outputs' chunk and outer sums in registers, which is why
//              warpgroup 0 hands its registers to the epilogue (setmaxnreg).
// Every wait is bounded (device_sync.cuh); a wait that gives up records
// CARBON_ERR_TIMEOUT and raises a CTA-wide abort flag, and the CTA still waits
// for its copies and MMAs in flight and frees its tensor memory.
#include "carbon_internal.h"
#include "bounds.cuh"
#include "device_sync.cuh"
#include "exact_bf16.cuh"
#include "superacc.cuh"
#include "tcgen05.cuh"

#include <algorithm>
#include <mutex>
#include <utility>
#include <vector>
#include <cstring>

namespace carbon {
namespace {

__device__ unsigned int g_exact_tc_status = 0;

// Bounds check of elements [idx, idx + len) of a buffer of n elements (the
// bounds-checked build; always true otherwise).
#define CHK(idx, len, n) in_bounds(&g_exact_tc_status, (int64_t)(idx), (int64_t)(len), (int64_t)(n))
__device__ unsigned long long g_exact_tc_kgroups = 0;   // plane products issued (measurement)
__device__ unsigned long long g_exact_tc_repairs = 0;   // chunk repairs and fix-ups (measurement)
__device__ unsigned long long g_exact_tc_fixups = 0;

// Optional CUDA-event timing of the main kernel (carbon_debug_kernel_timing).
std::mutex g_timing_mu;
bool g_timing_on = false;
// One call's events: before its first device operation, around the main
// kernel, after its last kernel (pre-pass, main kernel, post-pass).
struct CallEvents {
    cudaEvent_t e[4];
};
std::vector<CallEvents> g_timing_events;

// Events of a call while timing is on and the stream is not being captured;
// all null otherwise.
CallEvents timing_events(cudaStream_t s) {
    CallEvents ev = {{nullptr, nullptr, nullptr, nullptr}};
    std::lock_guard<std::mutex> lk(g_timing_mu);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (!g_timing_on || cudaStreamIsCapturing(s, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone)
        return ev;
    for (int k = 0; k < 4; ++k)
        if (cudaEventCreate(&ev.e[k]) != cudaSuccess) {
            for (int m = 0; m < k; ++m) cudaEventDestroy(ev.e[m]);
            return CallEvents{{nullptr, nullptr, nullptr, nullptr}};
        }
    g_timing_events.push_back(ev);
    return ev;
}

constexpr int kRowTile = 128;                         // output rows per tile = MMA M = TMEM lanes
constexpr int kColTile = 64;                          // output columns per tile
constexpr int kPlanes = 4;                            // base-256 digits of a line of width <= 31
constexpr int kMmaN = kColTile * kPlanes;             // 256
constexpr int kKBlock = 64;                           // reduction indices per 128-byte swizzle row
constexpr int kKBlocks = kChunk / kKBlock;            // 4
constexpr int kUmmaK = 16;
constexpr int kAStages = 4;                           // one k-group of A plane blocks...
constexpr int kAPairs = kAStages / 2;                 // ...signalled in pairs (half a k-group each)
constexpr int kEpiWarps = 8;
constexpr int kTcxThreads = 384;                      // warpgroup 0: TMA + MMA; 1-2: epilogue
constexpr int kUnitSlots = 4;                         // work units handed from the B producer to the others
constexpr int kUnitReaders = 2 + 1 + kEpiWarps;       // A producers, MMA issuer, epilogue warps
// Register split (setmaxnreg): the block is launched at kLaunchRegs per
// thread; warpgroup 0 gives registers back, warpgroups 1-2 take them:
// 128 * kRegsLow + 256 * kRegsHigh must not exceed 384 * kLaunchRegs.
constexpr int kLaunchRegs = 168;
constexpr int kRegsLow = 56;
constexpr int kRegsHigh = 224;
static_assert(128 * kRegsLow + 256 * kRegsHigh <= kTcxThreads * kLaunchRegs, "register split");
constexpr uint32_t kMagicBits = 0x4B400000u;          // fp32 bits of 1.5 * 2^23
constexpr uint32_t kABytes = kRowTile * kKBlock * 2;  // 16 KiB
constexpr uint32_t kBPlaneBytes = kColTile * kKBlock * 2;   // 8 KiB
constexpr uint32_t kBBytes = kPlanes * kBPlaneBytes;        // 32 KiB
constexpr uint32_t kTmemCols = 2 * kMmaN;             // 512
constexpr int kGrainNone = 0x40404040;                // grain of a line with no nonzero chunk (byte fill)
constexpr long long kDeferredSum = (long long)0x8000000000000000ull;   // Tout of a deferred output

// Start tiles: every 16-byte piece holds one bf16 value x and seven zeros, so
// one K = 16 MMA of the A tile (x = 1) with the B tile (x = 1.5 * 2^22) writes
// 2 * 1.5 * 2^22 = 1.5 * 2^23 to every accumulator element, whatever the order
// in which the tensor core walks the pieces.
constexpr uint32_t kStartABytes = kRowTile * kUmmaK * 2;   // 4 KiB
constexpr uint32_t kStartBBytes = kMmaN * kUmmaK * 2;      // 8 KiB
constexpr uint32_t kStartABits = 0x3F80u;                 // bf16 1.0
constexpr uint32_t kStartBBits = 0x4AC0u;                 // bf16 1.5 * 2^22

struct __align__(1024) TcxSmem {
    uint8_t B[kKBlocks][kBBytes];                     // 128 KiB: the chunk's B planes
    uint8_t A[kAStages][kABytes];                     // 64 KiB: A plane blocks
    uint8_t SA0[kStartABytes], SB0[kStartBBytes];     // 12 KiB: the accumulators' start tiles
    uint32_t pk[kEpiWarps][32];                       // packed column words of the current chunk
    uint64_t afull[kAPairs], aempty[kAPairs], bfull[kKBlocks / 2], bempty[kKBlocks / 2];
    uint64_t tfull[2], tempty[2], mdone;
    uint64_t ufull[kUnitSlots], uempty[kUnitSlots];
    int unit_q[kUnitSlots];                           // work unit in each slot (-1: no more)
    uint32_t tmem_slot, abort;
};

static_assert(sizeof(TcxSmem) + 1024 <= 232448, "shared memory per block");

struct TcxArgs {
    const unsigned short *bias;                       // bf16 [cols] or null
    void *out;
    int64_t rows, cols, LpA, LpB;
    int tiles_m, tiles_n, nchunks;
    int row_fast;                                     // tile order: row tile fastest (else column tile)
    int splits, cps;                                  // chunk range split into pieces of cps chunks
    const int4 *SA, *SB;                              // statistics [chunk][Lp]
    const int *GA, *GB;                               // line grains (smallest base) [Lp]
    const int *cntA;                                  // A planes per (row tile, chunk)
    const int *invA;                                  // row of each place in the A planes
    const int *cntB;                                  // B planes per (column tile, chunk)
    unsigned int *work_count, *work_list;             // deferred outputs
    int64_t work_cap;                                 // entries work_list can hold
    long long *Tout;                                  // exact sums in the output grain [piece][cols][rows]
    unsigned int *chunk_count;                        // (output, chunk) pairs for the chunk repair
    uint2 *chunk_list;
    unsigned int chunk_cap;
    unsigned int *unit_counter;                       // next work unit (starts at 0)
};

// Row and column tile of tile t.  Consecutive tiles share the operand whose
// digit planes are the larger of the two (the column tile when the B planes
// are larger, e.g. dW of a 768 x 3072 weight: the 6 row tiles of each column
// tile run together, so the B planes are read from DRAM about once instead of
// once per row tile); the order does not change any result.
__device__ __forceinline__ void tile_of(const TcxArgs &p, int t, int &tm, int &tn) {
    if (p.row_fast) { tm = t % p.tiles_m; tn = t / p.tiles_m; }
    else            { tm = t / p.tiles_n; tn = t % p.tiles_n; }
}

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile uint32_t *flag) {
    if (mbar_wait(bar, parity)) return true;
    *flag = 1u;
    atomicExch(&g_exact_tc_status, (unsigned)CARBON_ERR_TIMEOUT);
    return false;
}

// Work units are handed out at run time: the B producer takes the next one
// from the launch's counter when it is ready for it and posts it in slot
// n % kUnitSlots (-1 once all are taken); the other roles read the slots in
// the same order, so every role of a CTA works through the same units.  A
// reader frees its slot as soon as it has read it.
__device__ __forceinline__ bool fetch_unit(TcxSmem &sm, uint32_t n, unsigned int *counter, int nunits,
                                           volatile uint32_t *flag, int &u) {
    const uint32_t slot = n % kUnitSlots, use = n / kUnitSlots;
    if (!wait_or_abort(smem_addr(&sm.uempty[slot]), (use & 1u) ^ 1u, flag)) return false;
    const unsigned int v = atomicAdd(counter, 1u);
    u = v < (unsigned int)nunits ? (int)v : -1;
    sm.unit_q[slot] = u;
    mbar_arrive(smem_addr(&sm.ufull[slot]));              // release: the slot's value is visible
    return true;
}

__device__ __forceinline__ bool read_unit(TcxSmem &sm, uint32_t n, volatile uint32_t *flag, int &u) {
    const uint32_t slot = n % kUnitSlots, use = n / kUnitSlots;
    if (!wait_or_abort(smem_addr(&sm.ufull[slot]), use & 1u, flag)) return false;
    u = *reinterpret_cast<volatile int *>(&sm.unit_q[slot]);
    return true;
}

__device__ __forceinline__ void free_unit_slot(TcxSmem &sm, uint32_t n) {
    mbar_arrive(smem_addr(&sm.uempty[n % kUnitSlots]));
}

// ---- pre-pass: statistics and digit planes ------------------------------------

// bf16 bits of two integers of magnitude <= 256 (exact), hi in the upper
// half of the word and lo in the lower.
__device__ __forceinline__ uint32_t small_int_bf16_pair(int hi, int lo) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"((float)hi), "f"((float)lo));
    return r;
}

// Digits a line of this width needs (0: all zero, or not representable).
__device__ __forceinline__ int digits_for_width(int w) {
    return (w > 0 && w <= 31) ? (w + 8) / 8 : 0;
}

constexpr int kPrepThreads = 256;
constexpr int kPrepLines = 32;                        // lines per block (4 per warp)
constexpr int kRawPitch = kChunk + 8;                 // bf16 per staged line (16-byte rows)

// One block: 32 lines x one chunk; one warp per line at a time, lane t taking
// the reduction indices 8t .. 8t+7.  The source element (line, r) is
// src[line * ls + r * rs]; RCONTIG says rs == 1 (lines are read directly),
// otherwise the block's lines are staged in shared memory first (coalesced
// along the lines).  vec says 16-byte loads are aligned: 8 reduction indices
// of a line (RCONTIG), or 8 lines at one reduction index (ls == 1).
// Writes stats[chunk * Lp + line] and the line's digits (two per value, zeros
// elsewhere) tile by tile: plane a of the line placed at P goes to row
// (P / tg) 4 tg + a tg + P % tg of the [4 Lp][Rp] array (tg = tile lines,
// P = pos[line], or the line itself when pos is null); raises
// cnt[(P / tg) * nchunks + chunk] to the line's digit count n when cnt is not
// null; and lowers grain[line] (preset to kGrainNone) to the line's smallest
// base over the chunks where it is nonzero and finite with width <= 62 (the
// chunk repair adds the wider chunks in it).  FLAG_ONLY: only sets
// flag[line] when some chunk of the line needs four digits.
struct PrepArgs {
    const unsigned short *src;
    int64_t ls, rs, nlines, R, Lp, Rp;
    int tg;
    unsigned short *planes;
    int4 *stats;
    int *grain, *cnt;
    int nchunks, vec;
    const int *pos;
    int *flag;
};

// One block's work: lines bx * 32 .. + 31 of chunk by (see above).
template <bool RCONTIG, bool FLAG_ONLY>
__device__ __forceinline__ void prep_block(const PrepArgs &pa, int bx, int by) {
    const unsigned short *__restrict__ src = pa.src;
    const int64_t ls = pa.ls, rs = pa.rs, nlines = pa.nlines, R = pa.R, Lp = pa.Lp, Rp = pa.Rp;
    const int tg = pa.tg, nchunks = pa.nchunks, vec = pa.vec;
    unsigned short *__restrict__ planes = pa.planes;
    int4 *__restrict__ stats = pa.stats;
    int *__restrict__ grain = pa.grain;
    int *__restrict__ cnt = pa.cnt;
    const int *__restrict__ pos = pa.pos;
    int *__restrict__ flag = pa.flag;
    __shared__ __align__(16) unsigned short raw[RCONTIG ? 1 : kPrepLines * kRawPitch];
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int64_t line0 = (int64_t)bx * kPrepLines;
    const int q = by;
    const int64_t q0 = (int64_t)q * kChunk;
    // extents for the bounds-checked build: the operand, the planes, the
    // statistics, the per-line arrays and the per-(tile, chunk) counts
    const int64_t n_src = (nlines > 0 && R > 0) ? (nlines - 1) * ls + (R - 1) * rs + 1 : 0;
    const int64_t n_planes = (int64_t)kPlanes * Lp * Rp, n_stats = (int64_t)nchunks * Lp;
    const int64_t n_cnt = (Lp / tg) * nchunks;
    if (!RCONTIG) {
        if (vec && line0 + kPrepLines <= nlines && q0 + kChunk <= R) {
            // 8 lines at one reduction index per 16-byte load
            for (int e = tid; e < kPrepLines / 8 * kChunk; e += kPrepThreads) {
                const int lg = e % (kPrepLines / 8), r = e / (kPrepLines / 8);
                const int64_t at = (line0 + 8 * lg) + (q0 + r) * rs;
                if (!CHK(at, 8, n_src)) continue;
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src + at));
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int t = 0; t < 8; ++t)
                    raw[(8 * lg + t) * kRawPitch + r] = (unsigned short)(w[t / 2] >> (16 * (t & 1)));
            }
        } else {
            for (int e = tid; e < kPrepLines * kChunk; e += kPrepThreads) {
                const int l = e % kPrepLines, r = e / kPrepLines;
                const int64_t line = line0 + l, rr = q0 + r;
                raw[l * kRawPitch + r] = (line < nlines && rr < R && CHK(line * ls + rr * rs, 1, n_src))
                                             ? src[line * ls + rr * rs] : (unsigned short)0;
            }
        }
        __syncthreads();
    }
    // a warp's lines are l = warp, warp + 8, ...: their loads are all issued
    // before the first line is worked on (the loads' latency, not the
    // arithmetic, bounds this kernel)
    constexpr int kLinesPerWarp = kPrepLines / (kPrepThreads / 32);
    uint4 pre[kLinesPerWarp];
    int64_t places[kLinesPerWarp];
#pragma unroll
    for (int it = 0; it < kLinesPerWarp; ++it) {
        const int64_t L = line0 + warp + (kPrepThreads / 32) * it;
        places[it] = (pos != nullptr && CHK(L, 1, Lp)) ? (int64_t)__ldg(&pos[L]) : L;
        if (RCONTIG) {
            const int64_t r0 = q0 + 8 * lane;
            if (vec && L < nlines && r0 + 8 <= R && CHK(L * ls + r0, 8, n_src)) {
                pre[it] = __ldg(reinterpret_cast<const uint4 *>(src + L * ls + r0));
            } else {
                uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int64_t rr = r0 + e;
                    const uint32_t v = (L < nlines && rr < R && CHK(L * ls + rr, 1, n_src))
                                           ? (uint32_t)__ldg(src + L * ls + rr) : 0u;
                    w[e / 2] |= v << (16 * (e & 1));
                }
                pre[it] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        } else {
            pre[it] = *reinterpret_cast<const uint4 *>(&raw[(warp + (kPrepThreads / 32) * it) * kRawPitch + 8 * lane]);
        }
    }
#pragma unroll
    for (int it = 0; it < kLinesPerWarp; ++it) {
        const int64_t L = line0 + warp + (kPrepThreads / 32) * it;
        const int64_t LP = places[it];                       // the line's place in the planes
        uint32_t h[8];
        {
            const uint4 v = pre[it];
            h[0] = v.x & 0xffffu; h[1] = v.x >> 16; h[2] = v.y & 0xffffu; h[3] = v.y >> 16;
            h[4] = v.z & 0xffffu; h[5] = v.z >> 16; h[6] = v.w & 0xffffu; h[7] = v.w >> 16;
        }
        // values m * 2^e with the trailing zero bits of m moved into e, so the
        // base (the smallest such e) is as high as the values allow; the
        // width bound keeps the unstripped exponent (|m| < 2^8 there)
        int m[8], ex[8], lo = 1 << 20, hi = -(1 << 20), bad = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            bool b;
            decode(h[e], m[e], ex[e], b);
            if (m[e] != 0) {
                hi = max(hi, ex[e]);
                const int tz = __ffs(m[e]) - 1;
                m[e] >>= tz;                                  // exact: m is a multiple of 2^tz
                ex[e] += tz;
                lo = min(lo, ex[e]);
            }
            bad |= (int)b;
        }
        lo = __reduce_min_sync(0xffffffffu, lo);
        hi = __reduce_max_sync(0xffffffffu, hi);
        bad = (int)__reduce_or_sync(0xffffffffu, (unsigned)bad);
        const bool zero = hi == -(1 << 20);                   // no nonzero value
        const int base = zero ? 0 : lo;
        const int width = bad ? kWidthBad : (zero ? 0 : hi + 8 - lo);
        const bool use = width > 0 && width <= 31;
        const int n = digits_for_width(width);
        if (FLAG_ONLY) {                                  // the line needs four digits somewhere
            if (lane == 0 && n == kPlanes && L < nlines && CHK(L, 1, Lp)) atomicOr(&flag[L], 1);
            continue;
        }
        unsigned long long sum = 0ull;
        unsigned int mx = 0u;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            // (m = 0 gives 0 whatever its exponent: the shift is masked into range)
            const int X = use ? m[e] * (1 << ((ex[e] - base) & 31)) : 0;   // |X| < 2^31
            const unsigned int a = (unsigned int)abs(X);
            sum += a;
            mx = max(mx, a);
        }
        // the line's sum (below 2^39) from two 32-bit warp sums of its 16-bit
        // halves (each below 2^24)
        sum = ((unsigned long long)__reduce_add_sync(0xffffffffu, (unsigned)(sum >> 16)) << 16) +
              __reduce_add_sync(0xffffffffu, (unsigned)(sum & 0xffffu));
        mx = __reduce_max_sync(0xffffffffu, mx);
        if (lane == 0) {
            if (CHK((int64_t)q * Lp + L, 1, n_stats))
                stats[(int64_t)q * Lp + L] = make_int4(base, width, bit_count(sum), bit_count(mx));
            // the grain also covers finite lines too wide for the digits,
            // whose chunks the chunk repair adds in the same grain
            if (width > 0 && width <= 62 && CHK(L, 1, Lp)) atomicMin(&grain[L], base);
            if (use && cnt != nullptr && CHK((LP / tg) * nchunks + q, 1, n_cnt))
                atomicMax(&cnt[(LP / tg) * nchunks + q], n);
        }
        // X = v * 256^a with v = m << (s % 8), a = s / 8 (s = e - base): two
        // balanced digits, lo = v mod 256 in [-128, 127] at plane a and
        // hi = (v - lo) / 256 (|hi| <= 128) at plane a + 1; hi is 0 when a is
        // the line's top plane (then |v| < 2^(width % 8) <= 128)
        // The pair (hi, lo) of a value, as bf16 bits in one word, is moved to
        // the 16-bit fields a and a + 1 of a 64-bit word of the four planes
        // (a = 3 only when hi is 0, so nothing is shifted out); plane p of two
        // neighbouring values is then field p of their words, one byte
        // permute per plane and pair.
        static_assert(kPlanes == 4, "four 16-bit plane fields per 64-bit word");
        uint32_t wlo[8], whi[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int sh = ex[e] - base;
            const int v = use ? m[e] * (1 << (sh & 7)) : 0;             // |v| < 2^15; m = 0: 0
            const int lo = (int)(int8_t)v;                         // v mod 256 in [-128, 127]
            const unsigned long long w = (unsigned long long)small_int_bf16_pair((v - lo) >> 8, lo)
                                         << (16 * ((sh >> 3) & 3));            // v = 0: all zero
            wlo[e] = (uint32_t)w;
            whi[e] = (uint32_t)(w >> 32);
        }
        uint32_t packed[kPlanes][4];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            packed[0][w] = __byte_perm(wlo[2 * w], wlo[2 * w + 1], 0x5410);
            packed[1][w] = __byte_perm(wlo[2 * w], wlo[2 * w + 1], 0x7632);
            packed[2][w] = __byte_perm(whi[2 * w], whi[2 * w + 1], 0x5410);
            packed[3][w] = __byte_perm(whi[2 * w], whi[2 * w + 1], 0x7632);
        }
        const int64_t row = (LP / tg) * kPlanes * tg + LP % tg;
#pragma unroll
        for (int a = 0; a < kPlanes; ++a) {
            const int64_t at = (row + (int64_t)a * tg) * Rp + q0 + 8 * lane;
            if (CHK(at, 8, n_planes))
                *reinterpret_cast<uint4 *>(planes + at) =
                    make_uint4(packed[a][0], packed[a][1], packed[a][2], packed[a][3]);
        }
    }
}

template <bool RCONTIG, bool FLAG_ONLY>
__global__ void __launch_bounds__(kPrepThreads) digit_prep_kernel(const PrepArgs pa) {
    wait_prior_grid();
    allow_next_grid();
    prep_block<RCONTIG, FLAG_ONLY>(pa, blockIdx.x, blockIdx.y);
}

// Two independent passes in one launch (the A side's flag pass and the B
// side's digit planes): blocks [0, nx1) take the first, the rest the second.
template <bool RC1, bool FO1, bool RC2, bool FO2>
__global__ void __launch_bounds__(kPrepThreads)
digit_prep_pair_kernel(const PrepArgs p1, int nx1, const PrepArgs p2) {
    wait_prior_grid();
    allow_next_grid();
    if ((int)blockIdx.x < nx1) prep_block<RC1, FO1>(p1, blockIdx.x, blockIdx.y);
    else prep_block<RC2, FO2>(p2, blockIdx.x - nx1, blockIdx.y);
}

// ---- main kernel ----------------------------------------------------------------

// I += v * mul * 2^32 modulo 2^64 (mul = 256^(c - 4), c >= 4).
__device__ __forceinline__ void acc_hi(unsigned long long &I, uint32_t v, uint32_t mul) {
    asm("{\n\t.reg .u32 lo, hi;\n\t"
        "mov.b64 {lo, hi}, %0;\n\t"
        "mad.lo.u32 hi, %1, %2, hi;\n\t"
        "mov.b64 %0, {lo, hi};\n\t}"
        : "+l"(I) : "r"(v), "r"(mul));
}

// I += P * mul, P a signed 32-bit value, mul = 256^c (c <= 3), 32 x 32 -> 64-bit.
__device__ __forceinline__ void acc_pair_lo(unsigned long long &I, uint32_t P, uint32_t mul) {
    asm("mad.wide.s32 %0, %1, %2, %0;" : "+l"(I) : "r"(P), "r"(mul));
}

// Two accumulators a, b of planes 2 pp and 2 pp + 1 (bits = 1.5 * 2^23 + u,
// |u| <= 2^22): (bits_b << 8) + bits_a + kPairFix = u_a + 256 u_b modulo 2^32,
// which fits a signed 32-bit value.
constexpr uint32_t kPairFix = 0u - 257u * kMagicBits;

// Output bits the long way: float64 value, bias in float64, one rounding.
__device__ __noinline__ uint32_t out_bits_f64(long long T, int G, const unsigned short *bias, int64_t j) {
    double y = round_int_to_double(T, G);
    if (bias != nullptr) y = __dadd_rn(y, widen_bf16(ld_bits(bias, j)));
    return exact_round_bf16(y);
}

// v * 2^sh as a 64-bit two's complement pattern (the shift of the bits, which
// signed arithmetic leaves undefined for negative v or a result out of range;
// the callers check the range themselves).
__device__ __forceinline__ long long shl64(long long v, uint32_t sh) {
    return (long long)((unsigned long long)v << (sh & 63u));
}

// -2^k <= v < 2^k for a signed 64-bit v (0 < k < 63), tested in unsigned
// arithmetic so that no addition can overflow.
__device__ __forceinline__ bool below_pow2(long long v, int k) {
    return (unsigned long long)v + (1ull << k) < (2ull << k);
}

// I rounded to 53 significant bits, ties to even (|I| > 2^53 - 1, |I| < 2^63).
__device__ __forceinline__ long long round_to_53_bits(long long I) {
    const bool neg = I < 0;
    const unsigned long long mag = neg ? 0ull - (unsigned long long)I : (unsigned long long)I;
    const int sh = 11 - __clzll((long long)mag);           // 1 .. 10 low bits to drop
    const unsigned long long rem = mag & ((1ull << sh) - 1ull), half = 1ull << (sh - 1);
    unsigned long long m = mag >> sh;
    m += (rem > half || (rem == half && (m & 1ull))) ? 1ull : 0ull;
    const unsigned long long r = m << sh;
    return neg ? -(long long)r : (long long)r;
}

// bf16 bits of RN_bf16(V * 2^s) (nearest even), |V| <= 2^53: V truncated to
// float32 (one conversion), the lowest bit set when the truncation dropped a
// set bit (the low nb - 24 bits of |V|, nb its bit length, tested on the
// integer) - rounding to odd at 24 bits -, scaled by 2^s in the exponent
// field, and rounded to nearest even to bf16.  Rounding to odd at p + 2 or
// more bits and then to nearest at p bits gives the one rounding to nearest
// at p bits (Boldo and Melquiond, "Emulation of FMA and correctly rounded
// sums: proved algorithms using rounding to odd", IEEE Trans. Computers
// 57(4), 2008); here p = 8.  (The 64-bit conversion runs on the float64 pipe,
// hence one, not a conversion back.)  False when the value or the result is
// not a bf16 normal number (the caller then takes the float64 route).
__device__ __forceinline__ bool round_small_int_to_bf16(long long V, int s, uint32_t &bits) {
    float f;
    asm("cvt.rz.f32.s64 %0, %1;" : "=f"(f) : "l"(V));
    uint32_t fb = __float_as_uint(f);
    if (fb == 0u) { bits = 0u; return true; }               // V == 0
    const int e = (int)((fb >> 23) & 0xffu);                // 127 + nb - 1 (truncation keeps it)
    const int ef = e + s;                                   // biased exponent of the result
    if (ef < 1 || ef > 254) return false;
    // nb - 24 bits truncated, at most 30 (nb <= 54): all in the low word of
    // |V|, which is minus the low word of V when V < 0
    const int drop = e - 150;
    if (drop > 0) {
        const uint32_t lo = (uint32_t)(unsigned long long)V;
        if (((V < 0 ? 0u - lo : lo) & ((1u << drop) - 1u)) != 0u) fb |= 1u;
    }
    fb += (uint32_t)s << 23;
    unsigned short h;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(__uint_as_float(fb)));
    if ((h & 0x7fffu) >= 0x7f80u) return false;             // rounded past the largest finite
    bits = h;
    return true;
}

// bf16 bits of RN_bf16(RN_float64(V * 2^s)) (both nearest even), |V| < 2^63:
// V is first rounded to 53 significant bits when wider (the float64
// rounding; exact otherwise), and its zero low bits moved into the scale, so
// that what is rounded to bf16 is below 2^54 (2^53 after a rounding carry).
// False as above.
__device__ __forceinline__ bool round_int_to_bf16(long long V, int s, uint32_t &bits) {
    if (!below_pow2(V, 53)) {
        const unsigned long long mag = V < 0 ? 0ull - (unsigned long long)V : (unsigned long long)V;
        const int sh = 11 - __clzll((long long)mag);        // bits below the 53 kept ones
        V = round_to_53_bits(V) >> sh;                      // exact: those bits are now zero
        s += sh;
    }
    return round_small_int_to_bf16(V, s, bits);
}

// SUPER: the correctly rounded tier (chunk sums are added exactly, never
// rounded to 53 bits; the finalize rounds the exact total once).
template <bool SUPER>
__global__ void __launch_bounds__(kTcxThreads, 1)
exact_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                const TcxArgs p) {
    extern __shared__ uint8_t smem_raw[];
    TcxSmem &sm = *reinterpret_cast<TcxSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    volatile uint32_t *abort_flag = &sm.abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kAPairs; ++s) {
            mbar_init(smem_addr(&sm.afull[s]), 2);           // both A producers arrive
            mbar_init(smem_addr(&sm.aempty[s]), 1);
        }
        for (int pr = 0; pr < kKBlocks / 2; ++pr) {
            mbar_init(smem_addr(&sm.bfull[pr]), 1);
            mbar_init(smem_addr(&sm.bempty[pr]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_addr(&sm.tfull[b]), 1);
            mbar_init(smem_addr(&sm.tempty[b]), kEpiWarps);
        }
        mbar_init(smem_addr(&sm.mdone), 1);
        for (int u = 0; u < kUnitSlots; ++u) {
            mbar_init(smem_addr(&sm.ufull[u]), 1);
            mbar_init(smem_addr(&sm.uempty[u]), kUnitReaders);
        }
        *abort_flag = 0u;
        fence_mbar_init();
        if (p.nchunks > 0) {                                // maps are blank for an empty reduction
            prefetch_map(&map_a);
            prefetch_map(&map_b);
        }
    }
    for (uint32_t o = threadIdx.x * 16u; o < kStartABytes + kStartBBytes; o += kTcxThreads * 16u) {
        const uint32_t x = o < kStartABytes ? kStartABits : kStartBBits;
        uint8_t *dst = o < kStartABytes ? &sm.SA0[o] : &sm.SB0[o - kStartABytes];
        *reinterpret_cast<uint4 *>(dst) = make_uint4(x, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
    if (warp == 1) tmem_alloc(smem_addr(&sm.tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    wait_prior_grid();                                   // the digit planes and counters are written
    allow_next_grid();
    const uint32_t tmem = sm.tmem_slot;
    const int nunits = p.tiles_m * p.tiles_n * p.splits;   // (tile, chunk piece) work units
    const int nchunks = p.nchunks;

    if (warp < 4) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
      if (warp == 0 || warp == 2) {
        // ------------------------------------------------------------ A producers
        // The A loads of the CTA: k-group kg (counted over the CTA's units)
        // puts its 64-deep block kb in stage kb; stages 0-1 and 2-3 form the
        // pairs the MMA issuer waits for and releases together (two waits and
        // two commits per k-group instead of four each).  Warp 0 issues blocks
        // 0 and 2, warp 2 blocks 1 and 3 (one thread's copies complete one
        // after another, so two threads double the rate); both arrive on the
        // pair's barrier.
        if (lane == 0) {
            const uint32_t mine = warp == 0 ? 0u : 1u;
            uint32_t g = 0, n = 0;
            bool ok = true;
            while (ok) {
                int u;
                if (!(ok = read_unit(sm, n, abort_flag, u))) break;
                free_unit_slot(sm, n++);
                if (u < 0 || *abort_flag) break;
                const int t = u / p.splits, qlo = (u % p.splits) * p.cps;
                const int qhi = min(nchunks, qlo + p.cps);
                int tm, tn;
                tile_of(p, t, tm, tn);
                for (int q = qlo; ok && q < qhi; ++q) {
                    const int nx = CHK((int64_t)tm * nchunks + q, 1, (int64_t)p.tiles_m * nchunks)
                                       ? p.cntA[(int64_t)tm * nchunks + q] : 0;
                    for (int k = 0; ok && k < nx; ++k) {
                        for (int kb = 0; kb < kKBlocks; ++kb) {
                            if ((uint32_t)(kb & 1) != mine) continue;
                            const uint32_t pr = (uint32_t)kb >> 1;
                            // pair 0 is freed by its own commit; pair 1 when the
                            // previous k-group has finished, which its accumulator's
                            // commit (tfull) already signals
                            if (pr == 0) {
                                if (!(ok = wait_or_abort(smem_addr(&sm.aempty[0]), (g & 1u) ^ 1u, abort_flag))) break;
                            } else if (g > 0) {
                                if (!(ok = wait_or_abort(smem_addr(&sm.tfull[(g - 1u) & 1u]), ((g - 1u) >> 1) & 1u,
                                                         abort_flag)))
                                    break;
                            }
                            const uint32_t fa = smem_addr(&sm.afull[pr]);
                            mbar_arrive_expect_tx(fa, kABytes);
                            tma_load_2d(smem_addr(&sm.A[kb][0]), &map_a, fa, q * kChunk + kb * kKBlock,
                                        tm * kPlanes * kRowTile + k * kRowTile);
                        }
                        if (ok) ++g;                                // k-groups issued
                    }
                }
            }
            // the last use of each pair lands before the CTA may exit (an
            // earlier use was consumed, hence landed, before the pair was reused)
            if (g > 0)
                for (uint32_t pr = 0; pr < (uint32_t)kAPairs; ++pr)
                    if (!mbar_wait(smem_addr(&sm.afull[pr]), (g - 1u) & 1u)) break;
        }
      } else if (warp == 3) {
        // ------------------------------------------------------------ B producer
        // per chunk the four planes of each 64-deep block, 256 rows in one box
        if (lane == 0) {
            uint32_t bu = 0, n = 0, kg = 0;                  // chunks and k-groups loaded
            bool ok = true;
            while (ok) {
                int u;
                if (!(ok = fetch_unit(sm, n++, p.unit_counter, nunits, abort_flag, u))) break;
                if (u < 0 || *abort_flag) break;
                const int t = u / p.splits, qlo = (u % p.splits) * p.cps;
                const int qhi = min(nchunks, qlo + p.cps);
                int tm, tn;
                tile_of(p, t, tm, tn);
                for (int q = qlo; ok && q < qhi; ++q) {
                    if (!CHK((int64_t)tm * nchunks + q, 1, (int64_t)p.tiles_m * nchunks) ||
                        p.cntA[(int64_t)tm * nchunks + q] == 0)
                        continue;
                    // blocks 0-1 and 2-3 in pairs, one barrier each; pair 1 is
                    // free once the previous chunk's last k-group has finished
                    // (its accumulator's commit, tfull, signals that)
                    for (int pr = 0; pr < kKBlocks / 2; ++pr) {
                        if (pr == 0) {
                            if (!(ok = wait_or_abort(smem_addr(&sm.bempty[0]), (bu & 1u) ^ 1u, abort_flag))) break;
                        } else if (kg > 0) {
                            if (!(ok = wait_or_abort(smem_addr(&sm.tfull[(kg - 1u) & 1u]), ((kg - 1u) >> 1) & 1u,
                                                     abort_flag)))
                                break;
                        }
                        const uint32_t fb = smem_addr(&sm.bfull[pr]);
                        mbar_arrive_expect_tx(fb, 2 * kBBytes);
                        for (int kb = 2 * pr; kb < 2 * pr + 2; ++kb)
                            tma_load_2d(smem_addr(&sm.B[kb][0]), &map_b, fb, q * kChunk + kb * kKBlock,
                                        tn * kPlanes * kColTile);
                    }
                    if (ok) {
                        ++bu;
                        kg += (uint32_t)p.cntA[(int64_t)tm * nchunks + q];   // this chunk's k-groups
                    }
                }
            }
            if (bu > 0)
                for (int pr = 0; pr < kKBlocks / 2; ++pr)
                    if (!mbar_wait(smem_addr(&sm.bfull[pr]), (bu - 1u) & 1u)) break;
        }
      } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            // instruction descriptor: fp32 accumulate, bf16 A and B, both
            // K-major, M = 128; N = 256 for the start MMA, 64 per B plane the
            // column tile needs in the chunk for the others (the columns past
            // them keep the start value, a pair sum of 0)
            constexpr uint32_t idesc0 = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kRowTile >> 4) << 24);
            constexpr uint32_t idesc = idesc0 | ((uint32_t)(kMmaN >> 3) << 17);
            const uint64_t sdesc_a0 = smem_desc_noswizzle(smem_addr(&sm.SA0[0]), 128, 256);
            const uint64_t sdesc_b0 = smem_desc_noswizzle(smem_addr(&sm.SB0[0]), 128, 256);
            int acc = 0;
            uint32_t ph = 0, bu = 0, aph = 0;
            unsigned long long kgroups = 0;
            uint32_t n = 0;
            bool ok = true;
            while (ok) {
                int u;
                if (!(ok = read_unit(sm, n, abort_flag, u))) break;
                free_unit_slot(sm, n++);
                if (u < 0 || *abort_flag) break;
                const int t = u / p.splits, qlo = (u % p.splits) * p.cps;
                const int qhi = min(nchunks, qlo + p.cps);
                int tm, tn;
                tile_of(p, t, tm, tn);
                for (int q = qlo; ok && q < qhi; ++q) {
                    const int nx = CHK((int64_t)tm * nchunks + q, 1, (int64_t)p.tiles_m * nchunks)
                                       ? p.cntA[(int64_t)tm * nchunks + q] : 0;
                    if (nx == 0) continue;
                    const int nb = CHK((int64_t)tn * nchunks + q, 1, (int64_t)p.tiles_n * nchunks)
                                       ? max(1, p.cntB[(int64_t)tn * nchunks + q]) : 1;
                    const uint32_t idesc_q = idesc0 | ((uint32_t)(kColTile * nb >> 3) << 17);
                    for (int k = 0; ok && k < nx; ++k) {
                        if (!(ok = wait_or_abort(smem_addr(&sm.tempty[acc]), aph, abort_flag))) break;
                        tc_fence_after();
                        const uint32_t d = tmem + (uint32_t)(acc * kMmaN);
                        mma_bf16(d, sdesc_a0, sdesc_b0, idesc, 0u);    // every element 1.5 * 2^23
                        for (int kb = 0; kb < kKBlocks; ++kb) {
                            if ((kb & 1) == 0) {                     // a pair of A (and B) blocks
                                if (k == 0 && !(ok = wait_or_abort(smem_addr(&sm.bfull[kb >> 1]), bu & 1u, abort_flag)))
                                    break;
                                if (!(ok = wait_or_abort(smem_addr(&sm.afull[kb >> 1]), ph, abort_flag))) break;
                                tc_fence_after();
                            }
                            const uint32_t sa = smem_addr(&sm.A[kb][0]), sb = smem_addr(&sm.B[kb][0]);
#pragma unroll
                            for (int kk = 0; kk < kKBlock / kUmmaK; ++kk)
                                mma_bf16(d, smem_desc(sa + kk * (kUmmaK * 2), 16, 1024),
                                         smem_desc(sb + kk * (kUmmaK * 2), 16, 1024), idesc_q, 1u);
                            if (kb == 1) {                          // pair 1 is signalled by tfull
                                mma_commit(smem_addr(&sm.aempty[0]));
                                if (k == nx - 1) mma_commit(smem_addr(&sm.bempty[0]));
                            }
                        }
                        ph ^= 1u;                                   // the next k-group's pair phase
                        if (!ok) break;
                        mma_commit(smem_addr(&sm.tfull[acc]));          // k-group done
                        kgroups += (unsigned long long)nb;              // A plane x nb B planes
                        if (++acc == 2) { acc = 0; aph ^= 1u; }
                    }
                    ++bu;
                }
            }
            // every MMA issued so far has finished before the CTA frees TMEM
            mma_commit(smem_addr(&sm.mdone));
            mbar_wait(smem_addr(&sm.mdone), 0);
            atomicAdd(&g_exact_tc_kgroups, kgroups);
        }
      }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
        // ------------------------------------------------------------ epilogue
        const int ew = warp - 4;                             // 0..7
        const int quarter = warp % 4;                        // TMEM lanes 32 quarter .. +31
        const int half = ew / 4;                             // output columns 32 half .. +31
        const int rl = quarter * 32 + lane;                  // row within the tile
        const uint32_t tlane = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(half * 32);
        // both accumulators are free (each k-group's first MMA sets them to
        // 1.5 * 2^23)
        if (lane == 0) {
            mbar_arrive(smem_addr(&sm.tempty[0]));
            mbar_arrive(smem_addr(&sm.tempty[1]));
        }
        int acc = 0;
        uint32_t aph = 0, n = 0;
        bool ok = true;
        while (ok) {
            // lane 0 reads the unit and the warp follows its view, so that the
            // warp never splits here
            int u = -1, got = 0;
            if (lane == 0) {
                got = read_unit(sm, n, abort_flag, u) ? 1 : 0;
                if (got) free_unit_slot(sm, n);
                got |= (got && u >= 0 && !*abort_flag) ? 2 : 0;
            }
            got = __shfl_sync(0xffffffffu, got, 0);
            u = __shfl_sync(0xffffffffu, u, 0);
            ++n;
            if (!(ok = (got & 1) != 0)) break;
            if (!(got & 2)) break;
            const int t = u / p.splits, piece = u % p.splits, qlo = piece * p.cps;
            const int qhi = min(nchunks, qlo + p.cps);
            int tm, tn;
            tile_of(p, t, tm, tn);
            const int64_t ia_at = (int64_t)tm * kRowTile + rl;
            const int64_t i = CHK(ia_at, 1, p.LpA) ? (int64_t)__ldg(&p.invA[ia_at]) : 0;   // the row's own index
            const int64_t jw = (int64_t)tn * kColTile + half * 32;   // this warp's first column
            const int *cnt = p.cntA + (int64_t)tm * nchunks;
            const int Gx = CHK(i, 1, p.LpA) ? __ldg(&p.GA[i]) : 0;      // output grain: 2^(Gx + Gw)
            const int Gwl = CHK(jw + lane, 1, p.LpB) ? __ldg(&p.GB[jw + lane]) : 0;
            const int64_t n_cnt = (int64_t)(p.tiles_m - tm) * nchunks;    // cnt's extent from here
            const int64_t n_sa = (int64_t)nchunks * p.LpA, n_sb = (int64_t)nchunks * p.LpB;
            __syncwarp();                                    // last tile's reads are done
            // I, the chunk sum, starts at 0 (each plane pair's starting values
            // are taken out as it is added); T, the exact sum, too
            int nx = (qlo < qhi && CHK(qlo, 1, n_cnt)) ? cnt[qlo] : 0;
            unsigned long long I[32], T[32];
            {
#pragma unroll
                for (int c = 0; c < 32; ++c) { I[c] = 0ull; T[c] = 0ull; }
            }
            uint32_t defer = 0u;
            int4 rs = make_int4(0, 0, 0, 0), cl = rs;        // this chunk's statistics, loaded ahead
            if (qlo < qhi) {
                if (CHK((int64_t)qlo * p.LpA + i, 1, n_sa)) rs = __ldg(&p.SA[(int64_t)qlo * p.LpA + i]);
                if (CHK((int64_t)qlo * p.LpB + jw + lane, 1, n_sb)) cl = __ldg(&p.SB[(int64_t)qlo * p.LpB + jw + lane]);
            }

            for (int q = qlo; ok && q < qhi; ++q) {
                const int nx_next = (q + 1 < qhi && CHK(q + 1, 1, n_cnt)) ? cnt[q + 1] : 0;   // loaded a chunk ahead
                for (int k = 0; k < nx; ++k) {
                    if (!(ok = wait_or_abort(smem_addr(&sm.tfull[acc]), aph, abort_flag))) break;
                    tc_fence_after();
                    const uint32_t ta = tlane + (uint32_t)(acc * kMmaN);
                    // 8 units: planes (2 pp, 2 pp + 1) of 8 columns (group g), two
                    // 8-column loads each, issued before the previous unit's values
                    // are added in (planes past the chunk's nb hold the start value,
                    // a pair sum of 0).  The two planes' sums combine exactly in 32
                    // bits (|u_a + 256 u_b| < 2^31), on the integer ALUs, before one
                    // 64-bit multiply-add per pair.  Planes (0, 1) of every group
                    // first (weight 256^k, k <= 3), then planes (2, 3) (weight
                    // 256^(k+2)), whose two forms are chosen once per k-group.
                    uint32_t va[16], vb[16];
                    tmem_ld8x2_issue(ta, ta + (uint32_t)kColTile, va);
                    const uint32_t mul0 = 1u << (8 * k);
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        uint32_t(&cur)[16] = (g & 1) ? vb : va;
                        uint32_t(&nxt)[16] = (g & 1) ? va : vb;
                        tmem_wait_ld16(cur);
                        const uint32_t an = g < 3 ? ta + (uint32_t)(8 * (g + 1)) : ta + (uint32_t)(2 * kColTile);
                        tmem_ld8x2_issue(an, an + (uint32_t)kColTile, nxt);
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj)
                            acc_pair_lo(I[8 * g + jj], (cur[8 + jj] << 8) + cur[jj] + kPairFix, mul0);
                    }
                    if (k <= 1) {
                        const uint32_t mul = 1u << (8 * (k + 2));
#pragma unroll
                        for (int g = 0; g < 4; ++g) {
                            uint32_t(&cur)[16] = (g & 1) ? vb : va;
                            uint32_t(&nxt)[16] = (g & 1) ? va : vb;
                            tmem_wait_ld16(cur);
                            if (g < 3) {
                                const uint32_t an = ta + (uint32_t)(2 * kColTile + 8 * (g + 1));
                                tmem_ld8x2_issue(an, an + (uint32_t)kColTile, nxt);
                            }
#pragma unroll
                            for (int jj = 0; jj < 8; ++jj)
                                acc_pair_lo(I[8 * g + jj], (cur[8 + jj] << 8) + cur[jj] + kPairFix, mul);
                        }
                    } else {
                        const uint32_t mul = 1u << (8 * (k - 2));
#pragma unroll
                        for (int g = 0; g < 4; ++g) {
                            uint32_t(&cur)[16] = (g & 1) ? vb : va;
                            uint32_t(&nxt)[16] = (g & 1) ? va : vb;
                            tmem_wait_ld16(cur);
                            if (g < 3) {
                                const uint32_t an = ta + (uint32_t)(2 * kColTile + 8 * (g + 1));
                                tmem_ld8x2_issue(an, an + (uint32_t)kColTile, nxt);
                            }
#pragma unroll
                            for (int jj = 0; jj < 8; ++jj)
                                acc_hi(I[8 * g + jj], (cur[8 + jj] << 8) + cur[jj] + kPairFix, mul);
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_addr(&sm.tempty[acc]));
                    if (++acc == 2) { acc = 0; aph ^= 1u; }
                }
                if (!ok) break;
                // ---- chunk end: T += (chunk value in units of the output grain)
                const int bx = rs.x, wx = rs.y, lsx = rs.z, lmx = rs.w;
                const int shr = (wx > 0 && wx <= 31) ? bx - Gx : 0;
                const int shc = (cl.y > 0 && cl.y <= 31) ? min(cl.x - Gwl, 255) : 0;
                // bounds over the warp's 32 x 32 outputs (its rows and columns are
                // the lanes' rows and columns)
                const int wxm = (int)__reduce_max_sync(0xffffffffu, (unsigned)wx);
                const int wwm = (int)__reduce_max_sync(0xffffffffu, (unsigned)cl.y);
                const int shcm = (int)__reduce_max_sync(0xffffffffu, (unsigned)shc);
                const int bndm = min(min((int)__reduce_max_sync(0xffffffffu, (unsigned)lsx) +
                                             (int)__reduce_max_sync(0xffffffffu, (unsigned)cl.w),
                                         (int)__reduce_max_sync(0xffffffffu, (unsigned)lmx) +
                                             (int)__reduce_max_sync(0xffffffffu, (unsigned)cl.z)),
                                     wxm + wwm + 8);         // every |I| < 2^bndm
                __syncwarp();                                // last chunk's words are read
                // this lane's column in one word: bits 0-7 shift to the column grain
                // (255 when larger), 8-14 width, 15-20 bits of sum |W|, 21-26 of max |W|
                sm.pk[ew][lane] = (uint32_t)shc | ((uint32_t)min(cl.y, 127) << 8) |
                                  ((uint32_t)cl.z << 15) | ((uint32_t)cl.w << 21);
                __syncwarp();
                if (q + 1 < qhi) {                           // next chunk's statistics
                    if (CHK((int64_t)(q + 1) * p.LpA + i, 1, n_sa)) rs = __ldg(&p.SA[(int64_t)(q + 1) * p.LpA + i]);
                    if (CHK((int64_t)(q + 1) * p.LpB + jw + lane, 1, n_sb))
                        cl = __ldg(&p.SB[(int64_t)(q + 1) * p.LpB + jw + lane]);
                }
                // I is exact (modulo 2^64, and below 2^62) when every line fits.
                // Then all 32 outputs take T += I << sh at once while the checks
                // gather: the shifts lose no bit (and are below 64), no chunk
                // value rounds (|I| < 2^53) and T stays below 2^62 (the sum of
                // |T| < 2^62 and a lossless shift cannot wrap past that test).
                // A row that fails takes its additions back (exact, modulo 2^64)
                // and each of its outputs goes the long way.
                uint32_t redo = 0xffffffffu;                 // outputs for the per-output path
                bool added = false;                          // T holds this chunk's additions
                if (wxm <= 31 && wwm <= 31 && bndm <= 62) {
                    uint32_t lost = 0u, shs = 0u, ah = 0u, th = 0u;
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) {
                        const uint32_t sh = (uint32_t)shr + (sm.pk[ew][jj] & 0xffu);
                        const long long Ij = (long long)I[jj];
                        const long long v = shl64(Ij, sh);
                        const long long back = (v >> (sh & 63u)) ^ Ij;
                        lost |= (uint32_t)back | (uint32_t)(back >> 32);
                        shs |= sh;
                        const uint32_t ih = (uint32_t)(Ij >> 32);
                        ah |= ih ^ (uint32_t)((int)ih >> 31);
                        T[jj] += (unsigned long long)v;
                        const uint32_t t = (uint32_t)(T[jj] >> 32);
                        th |= t ^ (uint32_t)((int)t >> 31);
                    }
                    // a row that fails redoes its outputs one by one (its additions
                    // are still in T; each output keeps or takes back its own)
                    added = !(lost == 0u && shs < 64u && (SUPER || ah < (1u << 21)) && th < (1u << 30));
                    redo = added ? 0xffffffffu : 0u;
                }
                if (redo != 0u) {
                    // per output: the chunk value is the exact chunk sum rounded
                    // once to float64 (KBN recovers every rounding error of its
                    // loop exactly while wx + ww < 90), i.e. I itself when |I| < 2^53;
                    // the correctly rounded tier adds I itself
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) {
                        const uint32_t bit = 1u << jj;
                        if (!(redo & bit)) continue;
                        if (added) {
                            // this output's own checks: keep the addition when they pass
                            const uint32_t sh = (uint32_t)shr + (sm.pk[ew][jj] & 0xffu);
                            const long long I0 = (long long)I[jj];
                            const long long v = shl64(I0, sh);
                            // |I| < 2^53 and |T| < 2^62, tested in unsigned arithmetic
                            // (T may have wrapped: a signed test could overflow)
                            if ((v >> (sh & 63u)) == I0 && sh < 64u && (SUPER || below_pow2(I0, 53)) &&
                                below_pow2((long long)T[jj], 62))
                                continue;
                            T[jj] -= (unsigned long long)v;
                        }
                        long long Ij = (long long)I[jj];
                        const uint32_t w = sm.pk[ew][jj];
                        const int ww = (int)((w >> 8) & 0x7fu);
                        const int bnd = min(min(lsx + (int)((w >> 21) & 0x3fu), lmx + (int)((w >> 15) & 0x3fu)),
                                            wx + ww + 8);                   // |I| < 2^bnd
                        const bool fits = wx <= 31 && ww <= 31 && bnd <= 62;
                        if (!SUPER && bnd > 53 && !below_pow2(Ij, 53))
                            Ij = round_to_53_bits(Ij);                      // |result| <= 2^bnd
                        const int sh = shr + (int)(w & 0xffu);
                        const long long Tn = (long long)(T[jj] + (unsigned long long)shl64(Ij, (uint32_t)sh));
                        const int ib = 64 - __clzll(Ij ^ (Ij >> 63));          // |Ij| <= 2^ib
                        // no bit of I << sh lost, and the running sum stays below 2^62
                        const bool ok_add = ib + sh <= 61 && below_pow2(Tn, 62);
                        // a zero line (wx or ww 0) adds +0, which changes nothing
                        const bool live = fits && !(defer & bit) && wx != 0 && ww != 0;
                        T[jj] = (live && ok_add) ? (unsigned long long)Tn : T[jj];
                        bool bad = !(fits && (live ? ok_add : true));
                        // a finite line too wide for the digits: only this chunk is
                        // recomputed (and added to T) by the chunk repair kernel
                        if (!fits && !(defer & bit) && wx > 0 && ww > 0 && wx <= 62 && ww <= 62 &&
                            wx + ww < 90 && i < p.rows && jw + jj < p.cols) {
                            const unsigned int e = atomicAdd(p.chunk_count, 1u);
                            if (e < p.chunk_cap && CHK(e, 1, p.chunk_cap)) {
                                p.chunk_list[e] = make_uint2((unsigned int)(i * p.cols + jw + jj), (unsigned int)q);
                                bad = false;
                            }
                        }
                        defer |= bad ? bit : 0u;
                        T[jj] = bad ? 0ull : T[jj];
                    }
                }
                nx = nx_next;
#pragma unroll
                for (int c = 0; c < 32; ++c) I[c] = 0ull;
            }
            if (!ok) break;

            // ---- this piece's exact partial sums go to the finalize kernel
            // (deferred outputs: a sentinel no sum reaches, |T| < 2^62), stored
            // column-major so that a warp's 32 rows make one contiguous store
            if (i < p.rows) {
                const int64_t t0 = (int64_t)piece * p.rows * p.cols + jw * p.rows + i;
                const int64_t n_t = (int64_t)p.splits * p.rows * p.cols;
#pragma unroll
                for (int jj = 0; jj < 32; ++jj)
                    if (jw + jj < p.cols && CHK(t0 + (int64_t)jj * p.rows, 1, n_t))
                        p.Tout[t0 + (int64_t)jj * p.rows] = ((defer >> jj) & 1u) ? kDeferredSum : (long long)T[jj];
            }
            // outputs for the fix-up pass
            for (uint32_t dm = defer; dm != 0u; dm &= dm - 1u) {
                const int jj = __ffs((int)dm) - 1;
                if (i < p.rows && jw + jj < p.cols) {
                    const unsigned int at = atomicAdd(p.work_count, 1u);
                    if (CHK(at, 1, p.work_cap)) p.work_list[at] = (unsigned int)(i * p.cols + jw + jj);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---- chunk repair: single chunks with a line too wide for the digits ----------
//
// One warp per listed (output, chunk): the lanes load the chunk's 256 operand
// pairs, reduce the exact chunk sum I in 128-bit integers, and lane 0 rounds
// it once to 53 significant bits (the chunk value, as the KBN argument shows)
// and adds it, shifted to the output grain, into the output's piece sum with
// an integer atomic (exact, so the order of the additions does not matter).
// A value that does not fit, or an addition that overflows, lists the output
// for the full fix-up instead.
__device__ __forceinline__ __int128 round_i128_to_53_bits(__int128 I) {
    const bool neg = I < 0;
    const unsigned __int128 mag = neg ? (unsigned __int128)0 - (unsigned __int128)I : (unsigned __int128)I;
    const unsigned long long hi = (unsigned long long)(mag >> 64), lo = (unsigned long long)mag;
    const int nb = hi ? 128 - __clzll((long long)hi) : 64 - __clzll((long long)lo);
    if (nb <= 53) return I;
    const int sh = nb - 53;
    const unsigned __int128 rem = mag & (((unsigned __int128)1 << sh) - 1), half = (unsigned __int128)1 << (sh - 1);
    unsigned __int128 m = mag >> sh;
    m += (rem > half || (rem == half && (m & 1))) ? 1 : 0;
    const __int128 r = (__int128)(m << sh);
    return neg ? -r : r;
}

// One listed (output, chunk): its operand bits as loaded by the lanes.
struct RepairItem {
    int64_t o, q;
    int4 sa, sb;
    uint32_t hx[kChunk / 32], hw[kChunk / 32];
    bool valid;
};

// Loads list entry e (every lane: 8 of the chunk's 256 operand pairs).
__device__ __forceinline__ void repair_load(const IArgs &p, const int4 *__restrict__ SA,
                                            const int4 *__restrict__ SB, int64_t LpA, int64_t LpB,
                                            const uint2 *__restrict__ chunk_list, unsigned int chunk_cap,
                                            int64_t e, int lane, int64_t nq, int64_t n_a, int64_t n_b,
                                            RepairItem &it) {
    it.valid = CHK(e, 1, chunk_cap);
    if (!it.valid) return;
    const uint2 en = chunk_list[e];
    it.o = en.x;
    it.q = en.y;
    const int64_t i = it.o / p.cols, j = it.o % p.cols;
    it.valid = CHK(it.q * LpA + i, 1, nq * LpA) && CHK(it.q * LpB + j, 1, nq * LpB);
    if (!it.valid) return;
    it.sa = SA[it.q * LpA + i];
    it.sb = SB[it.q * LpB + j];
    const int64_t q0 = it.q * kChunk, qend = (p.R - q0 > kChunk) ? q0 + kChunk : p.R;
#pragma unroll
    for (int t = 0; t < kChunk / 32; ++t) {
        const int64_t r = q0 + lane + 32 * t;
        const bool in = r < qend && CHK(i * p.a_si + r * p.a_sr, 1, n_a) && CHK(r * p.b_sr + j * p.b_sj, 1, n_b);
        it.hx[t] = in ? ld_bits(p.A, i * p.a_si + r * p.a_sr) : 0u;
        it.hw[t] = in ? ld_bits(p.B, r * p.b_sr + j * p.b_sj) : 0u;
    }
}

template <bool SUPER>
__global__ void __launch_bounds__(256)
exact_chunk_repair_kernel(const IArgs p, const int4 *__restrict__ SA, const int4 *__restrict__ SB,
                          int64_t LpA, int64_t LpB, const int *__restrict__ GA,
                          const int *__restrict__ GB, const unsigned int *__restrict__ chunk_count,
                          const uint2 *__restrict__ chunk_list, unsigned int chunk_cap,
                          long long *Tout, int cps, unsigned int *work_count, unsigned int *work_list,
                          int64_t n_tout, int64_t work_cap) {
    wait_prior_grid();
    allow_next_grid();
    const int lane = threadIdx.x % 32;
    const int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) / 32;
    const int64_t nw = (int64_t)gridDim.x * blockDim.x / 32;
    const int64_t count = min(*chunk_count, chunk_cap);
    const int64_t nq = (p.R + kChunk - 1) / kChunk;
    const int64_t n_a = (p.rows > 0 && p.R > 0) ? (p.rows - 1) * p.a_si + (p.R - 1) * p.a_sr + 1 : 0;
    const int64_t n_b = (p.cols > 0 && p.R > 0) ? (p.R - 1) * p.b_sr + (p.cols - 1) * p.b_sj + 1 : 0;
    // the next entry's loads are issued before this one is reduced
    RepairItem cur, nxt;
    cur.valid = false;
    nxt.valid = false;
    if (gw < count) repair_load(p, SA, SB, LpA, LpB, chunk_list, chunk_cap, gw, lane, nq, n_a, n_b, cur);
    for (int64_t e = gw; e < count; e += nw) {
        if (e + nw < count) repair_load(p, SA, SB, LpA, LpB, chunk_list, chunk_cap, e + nw, lane, nq, n_a, n_b, nxt);
        if (cur.valid) {
            const int64_t o = cur.o, q = cur.q;
            const int64_t i = o / p.cols, j = o % p.cols;
            const int4 sa = cur.sa, sb = cur.sb;
            __int128 I = 0;
#pragma unroll
            for (int t = 0; t < kChunk / 32; ++t) {
                int mx, ex, mw, ew;
                bool bx_, bw_;
                decode(cur.hx[t], mx, ex, bx_);
                decode(cur.hw[t], mw, ew, bw_);
                if (mx == 0 || mw == 0) continue;
                const long long X = line_int(mx, ex, sa.x);                       // |X| < 2^62
                const long long W = line_int(mw, ew, sb.x);
                I += (__int128)X * W;                                             // |X W| < 2^90
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const long long lo = __shfl_xor_sync(0xffffffffu, (long long)(unsigned long long)I, off);
                const long long hi = __shfl_xor_sync(0xffffffffu, (long long)(I >> 64), off);
                I += ((__int128)hi << 64) | (__int128)(unsigned long long)lo;
            }
            if (lane == 0) {
                const __int128 J = SUPER ? I : round_i128_to_53_bits(I);
                const int sh = (CHK(i, 1, LpA) && CHK(j, 1, LpB)) ? (sa.x - __ldg(&GA[i])) + (sb.x - __ldg(&GB[j])) : -1;
                bool ok = sh >= 0 && sh < 62;
                __int128 v = 0;
                if (ok) {
                    v = (__int128)((unsigned __int128)J << sh);
                    ok = (v >> sh) == J && v >= -((__int128)1 << 61) && v < ((__int128)1 << 61);
                }
                if (ok && !CHK((q / cps) * p.rows * p.cols + j * p.rows + i, 1, n_tout)) ok = false;
                if (ok) {
                    long long *slot = Tout + (q / cps) * p.rows * p.cols + j * p.rows + i;
                    const long long add = (long long)v;
                    const long long old = (long long)atomicAdd(reinterpret_cast<unsigned long long *>(slot),
                                                               (unsigned long long)add);
                    const long long sum = (long long)((unsigned long long)old + (unsigned long long)add);
                    ok = !((old >= 0) == (add >= 0) && (sum >= 0) != (old >= 0));
                }
                if (!ok) {
                    const unsigned int at = atomicAdd(work_count, 1u);
                    if (CHK(at, 1, work_cap)) work_list[at] = (unsigned int)o;
                }
            }
        }
        cur = nxt;
    }
}

// Adds one call's chunk-repair and fix-up list lengths to the measurement
// counters (launched only while kernel timing is on).
__global__ void exact_count_kernel(const unsigned int *chunk_count, unsigned int chunk_cap,
                                   const unsigned int *work_count) {
    wait_prior_grid();
    allow_next_grid();
    atomicAdd(&g_exact_tc_repairs, (unsigned long long)min(*chunk_count, chunk_cap));
    atomicAdd(&g_exact_tc_fixups, (unsigned long long)*work_count);
}

// ---- finalize: bias and the two roundings ------------------------------------
//
// KBN over the chunk values is exact in the same way as inside a chunk: the
// value before the bias is the exact total T * 2^G rounded once to float64.
// That rounding is done on the integer, the bias (m * 2^e) joins it exactly,
// and the sum is rounded once more, to float64 and then to bf16 (both nearest
// even), all on integers; values outside those fast ranges take the float64
// route.  The chunk range of an output may have been split into pieces whose
// partial sums T add exactly.
//
// Layout of the work: a block takes 256 consecutive rows (a thread each) and
// a group of 8 consecutive columns (a two-dimensional grid, no division).  T
// is stored column-major, so each of a warp's loads is 256 contiguous bytes
// (32 rows of one column); the 8 columns' grains and biases are decoded once
// per block into one shared 16-byte word per column (one broadcast load per
// output); a thread's 8 outputs are 16 contiguous bytes of its row.
// Output modes of the finalize: the KBN tier's bf16 outputs, its float64
// values (inspection), and the correctly rounded tier's bf16 outputs (the
// exact total and the bias rounded once, never through float64).
constexpr int kFinBf16 = 0, kFinF64 = 1, kFinSuper = 2;
constexpr int kFinCols = 8;

// Output bits (KBN tier, bf16) of one output: exact sum T in grain 2^G, bias
// bm * 2^be (bm = 0: none; bad: inf/NaN) of column j.  Every case.
__device__ __noinline__ uint32_t kbn_bits_general(long long T, int G, int bm, int be, bool bad,
                                                  const unsigned short *bias, int64_t j) {
    long long Tv = T;
    int gs = G;
    bool fused = !bad;
    if (fused && bm != 0) {
        // the exact sum stays below 2^63: |T| < 2^61 and the bias term below
        // 2^62, or |T| < 2^53 shifted by at most 9
        if (be >= G && be - G <= 54 && below_pow2(T, 61)) {
            Tv = (below_pow2(T, 53) ? T : round_to_53_bits(T)) + shl64(bm, (uint32_t)(be - G));
        } else if (be < G && G - be <= 9 && below_pow2(T, 53)) {
            Tv = shl64(T, (uint32_t)(G - be)) + bm;
            gs = be;
        } else {
            fused = false;
        }
    }
    uint32_t bits = 0u;
    if (!(fused && round_int_to_bf16(Tv, gs, bits))) bits = out_bits_f64(T, G, bias, j);
    return bits;
}

// The same bits, with the common case inline: |T| < 2^53 (its float64 value
// is exact), no bias or one at or above the grain, and a sum below 2^53 that
// rounds to a bf16 normal number; the rest (rarely taken) in the general
// function, out of line.
__device__ __forceinline__ uint32_t kbn_bits(long long T, int G, int bm, int be, bool bad,
                                             const unsigned short *bias, int64_t j) {
    bool fast = !bad && below_pow2(T, 53);
    long long Tv = T;
    if (bm != 0) {
        fast = fast && be >= G && be - G <= 54;             // T + the bias term stays below 2^63
        Tv = T + shl64(bm, (uint32_t)(be - G) & 63u);
    }
    uint32_t bits = 0u;
    if (fast && below_pow2(Tv, 53) && round_small_int_to_bf16(Tv, G, bits)) return bits;
    return kbn_bits_general(T, G, bm, be, bad, bias, j);
}

template <int MODE>
__global__ void __launch_bounds__(256, 4)                  // 4 blocks per SM: at most 64 registers
exact_finalize_kernel(const long long *__restrict__ Tout, int pieces, const int *__restrict__ GA,
                      const int *__restrict__ GB, const unsigned short *__restrict__ bias, void *out,
                      int64_t rows, int64_t cols, int vec_out) {
    // the block's columns: grain of the column line, bias significand and
    // exponent, and the bias bits with an inf/NaN flag in bit 16
    __shared__ int4 s_col[kFinCols];
    wait_prior_grid();
    allow_next_grid();
    const int64_t plane = rows * cols, n_t = (int64_t)pieces * plane;
    const int64_t cgroups = (cols + kFinCols - 1) / kFinCols;
    const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
    const int gx = (i < rows && CHK(i, 1, rows)) ? __ldg(&GA[i]) : 0;
    for (int64_t cgi = blockIdx.y; cgi < cgroups; cgi += gridDim.y) {
        const int64_t j0 = cgi * kFinCols;
        if (cgi != (int64_t)blockIdx.y) __syncthreads();   // the previous columns' data is read
        if (threadIdx.x < kFinCols) {
            const int64_t j = j0 + threadIdx.x;
            int gw = 0, bm = 0, be = 0;
            bool bad = false;
            uint32_t hb = 0u;
            if (j < cols && CHK(j, 1, cols)) {
                gw = __ldg(&GB[j]);
                if (bias != nullptr) { hb = ld_bits(bias, j); decode(hb, bm, be, bad); }
            }
            s_col[threadIdx.x] = make_int4(gw, bm, be, (int)(hb | (bad ? 0x10000u : 0u)));
        }
        __syncthreads();
        if (i >= rows) continue;
        const int ncol = (int)min((int64_t)kFinCols, cols - j0);
        const long long *tp = Tout + j0 * rows + i;
        // the pieces' partial sums: in 64 bits with an overflow bit per output
        // (bf16 outputs; an overflowing output adds its pieces again in 128
        // bits), in 128 bits for the other modes
        long long sum[kFinCols];
        __int128 acc[MODE == kFinBf16 ? 1 : kFinCols];
        uint32_t deferred = 0u, ovf = 0u;
        for (int k = 0; k < pieces; ++k) {
            long long t[kFinCols];
#pragma unroll
            for (int e = 0; e < kFinCols; ++e) {
                const int64_t off = k * plane + e * rows;
                t[e] = (e < ncol && CHK(j0 * rows + i + off, 1, n_t)) ? __ldg(tp + off) : 0ll;
            }
#pragma unroll
            for (int e = 0; e < kFinCols; ++e) {
                // the sentinel's high word alone: a sum's is within +-2^30
                deferred |= ((uint32_t)((unsigned long long)t[e] >> 32) == 0x80000000u ? 1u : 0u) << e;
                if constexpr (MODE == kFinBf16) {
                    if (k == 0) {
                        sum[e] = t[e];
                    } else {
                        // two's complement sum; it overflowed when both terms
                        // have one sign and the sum the other
                        const long long v = (long long)((unsigned long long)sum[e] + (unsigned long long)t[e]);
                        ovf |= ((((sum[e] ^ v) & (t[e] ^ v)) < 0) ? 1u : 0u) << e;
                        sum[e] = v;
                    }
                } else {
                    acc[e] = (k == 0 ? (__int128)0 : acc[e]) + (__int128)t[e];
                }
            }
        }
        uint32_t packed[kFinCols / 2];
#pragma unroll
        for (int e = 0; e < kFinCols / 2; ++e) packed[e] = 0u;
#pragma unroll
        for (int e = 0; e < kFinCols; ++e) {
            if (e >= ncol || ((deferred >> e) & 1u)) continue;
            const int64_t j = j0 + e;
            const int4 c = s_col[e];
            const int G = gx + c.x;
            const int bm = c.y, be = c.z;
            const bool bad = (c.w >> 16) != 0;
            const uint32_t hb = (uint32_t)c.w & 0xffffu;
            uint32_t bits = 0u;
            if constexpr (MODE == kFinBf16) {
                if (!((ovf >> e) & 1u)) {
                    bits = kbn_bits(sum[e], G, bm, be, bad, bias, j);
                } else {                                    // the pieces' sum needs 128 bits
                    __int128 a = 0;
                    for (int k = 0; k < pieces; ++k) {
                        const int64_t at = k * plane + j * rows + i;
                        if (CHK(at, 1, n_t)) a += __ldg(&Tout[at]);
                    }
                    double y = round_i128_to_double(a, G);
                    if (bias != nullptr) y = __dadd_rn(y, widen_bf16(hb));
                    bits = exact_round_bf16(y);
                }
            } else if constexpr (MODE == kFinSuper) {
                bits = sacc::exact_sum_bf16(acc[e], G, bm, be, bad, hb);
            } else {                                        // float64 value (inspection)
                const bool small = acc[e] >= -((__int128)1 << 62) && acc[e] < ((__int128)1 << 62);
                double y = small ? round_int_to_double((long long)acc[e], G) : round_i128_to_double(acc[e], G);
                if (bias != nullptr) y = __dadd_rn(y, widen_bf16(hb));
                if (CHK(i * cols + j, 1, plane)) static_cast<double *>(out)[i * cols + j] = y;
            }
            packed[e / 2] |= bits << (16 * (e & 1));
        }
        if constexpr (MODE == kFinF64) continue;
        unsigned short *orow = static_cast<unsigned short *>(out) + i * cols + j0;
        if (!CHK(i * cols + j0, ncol, plane)) continue;
        if (deferred == 0u && ncol == kFinCols && vec_out) {
            *reinterpret_cast<uint4 *>(orow) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        } else {
#pragma unroll
            for (int e = 0; e < kFinCols; ++e)
                if (e < ncol && !((deferred >> e) & 1u)) orow[e] = (unsigned short)(packed[e / 2] >> (16 * (e & 1)));
        }
    }
}

// Blocks of the post-pass kernels that stride over the repair and fix-up
// lists (GPT-2 data lists thousands of chunk repairs on some weight
// gradients: fewer blocks cost more than their launch saves).
constexpr int kPostBlocks = kFixBlocks;

template <int MODE>
cudaError_t launch_tc_main(const CUtensorMap &ma, const CUtensorMap &mb, const TcxArgs &a, int grid,
                           const Problem &prob, const IArgs &ia, const int4 *SA, const int4 *SB,
                           int64_t LpA, int64_t LpB, unsigned int *work, const CallEvents &ev,
                           cudaStream_t s) {
    constexpr bool SUPER = MODE == kFinSuper;
    auto kern = exact_tc_kernel<SUPER>;
    const int smem = (int)sizeof(TcxSmem) + 1024;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    if (ev.e[1]) cudaEventRecord(ev.e[1], s);
    err = launch_k(kern, dim3(grid), dim3(kTcxThreads), (size_t)smem, s, 1, ma, mb, a);
    count_launch();
    if (ev.e[2]) cudaEventRecord(ev.e[2], s);
    if (err != cudaSuccess) return err;
    err = launch_k(exact_chunk_repair_kernel<SUPER>, dim3(kPostBlocks), dim3(256), 0, s, 1,
                   ia, SA, SB, LpA, LpB, a.GA, a.GB, (const unsigned int *)a.chunk_count,
                   (const uint2 *)a.chunk_list, a.chunk_cap, a.Tout, a.cps, work, work + 1,
                   (int64_t)a.splits * a.rows * a.cols, a.work_cap);
    count_launch();
    if (err != cudaSuccess) return err;
    if (ev.e[0]) {
        err = launch_k(exact_count_kernel, dim3(1), dim3(1), 0, s, 1,
                       (const unsigned int *)a.chunk_count, a.chunk_cap, (const unsigned int *)work);
        count_launch();
        if (err != cudaSuccess) return err;
    }
    {
        // a block per 256 rows and group of 8 columns (groups past 65535 taken
        // in turn by the blocks of the same rows)
        const int64_t cgroups = (a.cols + kFinCols - 1) / kFinCols;
        const dim3 grid((unsigned)((a.rows + 255) / 256), (unsigned)(cgroups < 65535 ? cgroups : 65535));
        const int vec_out = ((reinterpret_cast<uintptr_t>(a.out) & 15u) == 0 && (a.cols % 8) == 0) ? 1 : 0;
        err = launch_k(exact_finalize_kernel<MODE>, grid, dim3(256), 0, s, 1,
                       (const long long *)a.Tout, a.splits, a.GA, a.GB, a.bias, a.out, a.rows, a.cols,
                       vec_out);
        count_launch();
        if (err != cudaSuccess) return err;
    }
    if (SUPER) {
        err = superacc_fixup_bf16(prob, work, work + 1, kPostBlocks, s);
    } else {
        err = launch_k(exact_fixup_kernel<MODE == kFinF64>, dim3(kPostBlocks), dim3(kFixWarps * 32), 0, s, 1,
                       ia, SA, SB, LpA, LpB, (const unsigned int *)work, (const unsigned int *)(work + 1));
        count_launch();
    }
    if (ev.e[3]) cudaEventRecord(ev.e[3], s);
    return err;
}

// Pieces the chunk range of each output tile is cut into: the smallest count
// in {1, 2, 4, 8} (at most half the chunks, unless 1) that gives the launch at
// least four work units per SM and work units of at most 8 chunks, so that
// the units handed out last are short and the SMs finish close together.  The
// result does not depend on it: the pieces' integer sums add exactly.
int choose_pieces(int64_t tiles, int64_t nchunks, int sms) {
    int s = 1;
    while (s < 8 && 2 * s <= nchunks &&
           (tiles * s < 4 * (int64_t)sms || (nchunks + s - 1) / s > 8))
        s *= 2;
    return s;
}

PrepArgs prep_args(const unsigned short *src, int64_t ls, int64_t rs, int64_t nlines, int64_t R,
                   int64_t Lp, int64_t Rp, int tg, unsigned short *planes, int4 *stats, int *grain,
                   int *cnt, int nchunks, const int *pos, int *flag, bool rcontig) {
    PrepArgs a;
    a.src = src; a.ls = ls; a.rs = rs; a.nlines = nlines; a.R = R; a.Lp = Lp; a.Rp = Rp; a.tg = tg;
    a.planes = planes; a.stats = stats; a.grain = grain; a.cnt = cnt; a.nchunks = nchunks;
    const bool aligned = (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
    a.vec = rcontig ? (aligned && ls % 8 == 0) : (aligned && ls == 1 && rs % 8 == 0);
    a.pos = pos; a.flag = flag;
    return a;
}

template <bool RCONTIG, bool FLAG_ONLY>
cudaError_t launch_prep(const PrepArgs &a, cudaStream_t s) {
    const dim3 grid((unsigned)(a.Lp / kPrepLines), (unsigned)a.nchunks);
    const cudaError_t err = launch_k(digit_prep_kernel<RCONTIG, FLAG_ONLY>, grid, dim3(kPrepThreads), 0, s, 1, a);
    count_launch();
    return err;
}

// The A side's flag pass and the B side's planes, in one launch.
template <bool RCA, bool RCB>
cudaError_t launch_flag_and_prep_b(const PrepArgs &fa, const PrepArgs &pb, cudaStream_t s) {
    const int nx1 = (int)(fa.Lp / kPrepLines);
    const dim3 grid((unsigned)(nx1 + pb.Lp / kPrepLines), (unsigned)fa.nchunks);
    const cudaError_t err = launch_k(digit_prep_pair_kernel<RCA, true, RCB, false>, grid, dim3(kPrepThreads),
                                     0, s, 1, fa, nx1, pb);
    count_launch();
    return err;
}

// Workspace set-up of one call, in place of separate memsets: the line grains
// start at kGrainNone (n_grain ints from grain), the row flags, plane counts
// and counters at 0 (n_zero ints from zero, n_cnt from counters).
__global__ void __launch_bounds__(256)
exact_init_kernel(int *__restrict__ grain, int64_t n_grain, int *__restrict__ zero, int64_t n_zero,
                  unsigned int *__restrict__ counters, int n_cnt) {
    wait_prior_grid();
    allow_next_grid();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t t0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    for (int64_t k = t0; k < n_grain; k += stride) grain[k] = kGrainNone;
    for (int64_t k = t0; k < n_zero; k += stride) zero[k] = 0;
    if (t0 < n_cnt) counters[t0] = 0u;
}

// Places of the A rows in the digit planes: within each group of 1024 rows
// (8 row tiles) the rows whose chunks all fit three digits come first, in
// order, then the others, in order; places past the last row keep their own
// index.  Tiles then mostly hold rows of one kind, so fewer of them need the
// fourth digit plane (about 15% fewer MMAs on the GPT-2 operands).  The sums
// are exact, so the placement does not change any result.
constexpr int kOrderGroup = 1024;

__global__ void __launch_bounds__(kOrderGroup)
row_order_kernel(const int *__restrict__ flag, int64_t rows, int64_t Lp, int *__restrict__ pos,
                 int *__restrict__ inv) {
    __shared__ int wz[kOrderGroup / 32], wv[kOrderGroup / 32];
    wait_prior_grid();
    allow_next_grid();
    const int t = threadIdx.x, warp = t / 32, lane = t % 32;
    const int64_t base = (int64_t)blockIdx.x * kOrderGroup, i = base + t;
    const bool valid = i < rows;
    const bool z = valid && CHK(i, 1, Lp) && flag[i] == 0;   // three digits suffice everywhere
    const uint32_t below = (1u << lane) - 1u;
    const uint32_t bz = __ballot_sync(0xffffffffu, z), bv = __ballot_sync(0xffffffffu, valid);
    if (lane == 0) { wz[warp] = __popc(bz); wv[warp] = __popc(bv); }
    __syncthreads();
    int pz = 0, pv = 0, tz = 0;                      // rows of each kind before this warp; all z rows
    for (int w = 0; w < kOrderGroup / 32; ++w) {
        if (w < warp) { pz += wz[w]; pv += wv[w]; }
        tz += wz[w];
    }
    if (!valid) {
        if (i < Lp) { pos[i] = (int)i; inv[i] = (int)i; }
        return;
    }
    const int rz = pz + __popc(bz & below);          // z rows before this one
    const int rv = pv + __popc(bv & below);          // valid rows before this one
    const int64_t place = base + (z ? rz : tz + (rv - rz));
    if (CHK(i, 1, Lp)) pos[i] = (int)place;
    if (CHK(place, 1, Lp)) inv[place] = (int)i;
}

}  // namespace

carbon_status_t exact_tc_launch(const Problem &p, bool out_f64, bool super, cudaStream_t stream) {
    if (p.rows == 0 || p.cols == 0) return CARBON_OK;
    // deferred outputs are listed by 32-bit index; larger outputs take the
    // float64 kernel (or the warp-per-output superaccumulator), which compute
    // the same bits
    if (p.rows * p.cols >= ((int64_t)1 << 32))
        return super ? superacc_launch(p, stream) : exact_launch(p, out_f64, stream);
    int dev = 0, sms = 0;
    carbon_status_t st = current_device(&dev, &sms);
    if (st != CARBON_OK) return st;

    IArgs ia;
    ia.A = static_cast<const unsigned short *>(p.A);
    ia.B = static_cast<const unsigned short *>(p.B);
    ia.bias = static_cast<const unsigned short *>(p.bias);
    ia.out = p.out;
    ia.rows = p.rows; ia.cols = p.cols; ia.R = p.R;
    switch (p.pass) {
    case CARBON_PASS_FWD: ia.a_si = p.K; ia.a_sr = 1; ia.b_sr = p.N; ia.b_sj = 1; break;
    case CARBON_PASS_DX:  ia.a_si = p.N; ia.a_sr = 1; ia.b_sr = 1;   ia.b_sj = p.N; break;
    default:              ia.a_si = 1;   ia.a_sr = p.K; ia.b_sr = p.N; ia.b_sj = 1; break;
    }
    const int64_t tiles_m = (p.rows + kRowTile - 1) / kRowTile;
    const int64_t tiles_n = (p.cols + kColTile - 1) / kColTile;
    ia.tiles_n = tiles_n;
    const int64_t LpA = tiles_m * kRowTile, LpB = tiles_n * kColTile;
    const int64_t nchunks = (p.R + kChunk - 1) / kChunk;
    const int64_t Rp = nchunks * kChunk;
    if (tiles_m * tiles_n > 0x7fffffff || nchunks > 65535 || 4 * LpA > 0x7fffffff ||
        4 * LpB > 0x7fffffff || Rp > 0x7fffffff)
        return CARBON_ERR_INVALID_ARG;

    // workspace (stream-ordered, released at the end of this call): digit
    // planes of A and B, statistics, A plane counts, the deferral counter and list
    const size_t pA = (size_t)kPlanes * LpA * Rp, pB = (size_t)kPlanes * LpB * Rp;
    const size_t sA = (size_t)nchunks * LpA, sB = (size_t)nchunks * LpB;
    const size_t cntBytes = ((4 * (size_t)(tiles_m + tiles_n) * nchunks) + 15) & ~(size_t)15;
    const int pieces = choose_pieces(tiles_m * tiles_n, nchunks, sms);
    const size_t outs = (size_t)p.rows * (size_t)p.cols;
    const size_t tBytes = (8 * outs * pieces + 255) & ~(size_t)255;   // keeps the planes aligned
    // chunk repair list (capacity capped; an output that does not get a slot is
    // listed for the full fix-up instead); each piece and each repaired chunk
    // may list an output for the fix-up
    const size_t ccap = std::min<size_t>(outs * (size_t)nchunks, (size_t)1 << 22);
    const size_t bytes = tBytes + 2 * (pA + pB) + 16 * (sA + sB) + 4 * (size_t)(LpA + LpB) +
                         12 * (size_t)LpA + cntBytes + 8 * ccap + 16 + 4 * (outs * pieces + ccap + 1);
    char *ws = nullptr;
    cudaError_t err = cudaMallocAsync(reinterpret_cast<void **>(&ws), bytes, stream);
    if (err != cudaSuccess) return note_cuda(err);
    long long *Tout = reinterpret_cast<long long *>(ws);
    unsigned short *PA = reinterpret_cast<unsigned short *>(ws + tBytes);
    unsigned short *PB = PA + pA;
    int4 *SA = reinterpret_cast<int4 *>(PB + pB);
    int4 *SB = SA + sA;
    int *GA = reinterpret_cast<int *>(SB + sB);
    int *GB = GA + LpA;
    int *flagA = GB + LpB;                               // rows needing four digits somewhere
    int *posA = flagA + LpA;                             // place of each row in the A planes
    int *invA = posA + LpA;                              // row at each place
    int *cntA = invA + LpA;                              // planes per (row tile, chunk)
    int *cntB = cntA + tiles_m * nchunks;                // planes per (column tile, chunk)
    uint2 *clist = reinterpret_cast<uint2 *>(reinterpret_cast<char *>(cntA) + cntBytes);
    unsigned int *ccount = reinterpret_cast<unsigned int *>(clist + ccap);   // chunk repairs, work units
    unsigned int *work = ccount + 4;

    const CallEvents ev = timing_events(stream);
    if (ev.e[0]) cudaEventRecord(ev.e[0], stream);
    // the line grains start at kGrainNone; the row flags, the plane counts,
    // the chunk-repair and unit counters and the deferral counter at 0 (the
    // plane counts follow the row flags, place and row arrays: one zeroed
    // range covers flags .. counts, the place and row arrays being written
    // in full by the row order anyway)
    {
        const int64_t n_zero = (int64_t)(cntA - flagA) + (int64_t)(cntBytes / 4);
        const int64_t n_max = (LpA + LpB) > n_zero ? (LpA + LpB) : n_zero;
        const int64_t want = (n_max + 255) / 256;
        const unsigned blocks = (unsigned)(want < 1024 ? (want > 0 ? want : 1) : 1024);
        err = launch_k(exact_init_kernel, dim3(blocks), dim3(256), 0, stream, 1, GA,
                       (int64_t)(LpA + LpB), flagA, n_zero, ccount, 5);
        count_launch();
    }
    const bool a_rc = (p.pass != CARBON_PASS_DW), b_rc = (p.pass == CARBON_PASS_DX);
    const PrepArgs fa = prep_args(ia.A, ia.a_si, ia.a_sr, p.rows, p.R, LpA, Rp, kRowTile, PA, SA, GA,
                                  nullptr, (int)nchunks, nullptr, flagA, a_rc);
    const PrepArgs pa = prep_args(ia.A, ia.a_si, ia.a_sr, p.rows, p.R, LpA, Rp, kRowTile, PA, SA, GA,
                                  cntA, (int)nchunks, posA, nullptr, a_rc);
    const PrepArgs pb = prep_args(ia.B, ia.b_sj, ia.b_sr, p.cols, p.R, LpB, Rp, kColTile, PB, SB, GB,
                                  cntB, (int)nchunks, nullptr, nullptr, b_rc);
    // the A rows' four-digit flags and the B planes (independent) in one
    // launch, then the row order, then the A planes at the ordered places
    if (err == cudaSuccess && nchunks > 0)
        err = a_rc ? (b_rc ? launch_flag_and_prep_b<true, true>(fa, pb, stream)
                           : launch_flag_and_prep_b<true, false>(fa, pb, stream))
                   : (b_rc ? launch_flag_and_prep_b<false, true>(fa, pb, stream)
                           : launch_flag_and_prep_b<false, false>(fa, pb, stream));
    if (err == cudaSuccess) {
        err = launch_k(row_order_kernel, dim3((unsigned)((LpA + kOrderGroup - 1) / kOrderGroup)),
                       dim3(kOrderGroup), 0, stream, 1, flagA, p.rows, LpA, posA, invA);
        count_launch();
    }
    if (err == cudaSuccess && nchunks > 0)
        err = a_rc ? launch_prep<true, false>(pa, stream) : launch_prep<false, false>(pa, stream);
    // planes as 2-D [4 Lp][Rp] bf16 maps, 64-deep boxes, 128-byte swizzle:
    // one A plane of a row tile (128 rows), all four B planes of a column tile
    // (256 rows) per box
    CUtensorMap ma, mb;
    std::memset(&ma, 0, sizeof ma);
    std::memset(&mb, 0, sizeof mb);
    if (err == cudaSuccess && nchunks > 0) {
        err = encode_tensor_map_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, PA, (uint64_t)Rp,
                                   (uint64_t)(kPlanes * LpA), (uint64_t)Rp * 2, kKBlock, kRowTile,
                                   CU_TENSOR_MAP_SWIZZLE_128B);
        if (err == cudaSuccess)
            err = encode_tensor_map_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, PB, (uint64_t)Rp,
                                       (uint64_t)(kPlanes * LpB), (uint64_t)Rp * 2, kKBlock,
                                       kPlanes * kColTile, CU_TENSOR_MAP_SWIZZLE_128B);
    }
    if (err == cudaSuccess) {
        TcxArgs a;
        a.bias = ia.bias;
        a.out = p.out;
        a.rows = p.rows; a.cols = p.cols; a.LpA = LpA; a.LpB = LpB;
        a.tiles_m = (int)tiles_m; a.tiles_n = (int)tiles_n; a.nchunks = (int)nchunks;
        a.row_fast = LpB > LpA ? 1 : 0;                  // keep the larger planes' tiles together
        a.splits = pieces;
        a.cps = (int)((nchunks + pieces - 1) / pieces);
        a.SA = SA; a.SB = SB; a.GA = GA; a.GB = GB; a.cntA = cntA; a.invA = invA;
        a.cntB = cntB;
        a.work_count = work; a.work_list = work + 1;
        a.work_cap = (int64_t)(outs * pieces + ccap);
        a.Tout = Tout;
        a.chunk_count = ccount;
        a.chunk_list = clist;
        a.chunk_cap = (unsigned int)ccap;
        a.unit_counter = ccount + 1;
        const int64_t units = tiles_m * tiles_n * pieces;
        const int grid = (int)(units < sms ? units : sms);
        err = super ? launch_tc_main<kFinSuper>(ma, mb, a, grid, p, ia, SA, SB, LpA, LpB, work, ev, stream)
            : out_f64 ? launch_tc_main<kFinF64>(ma, mb, a, grid, p, ia, SA, SB, LpA, LpB, work, ev, stream)
                      : launch_tc_main<kFinBf16>(ma, mb, a, grid, p, ia, SA, SB, LpA, LpB, work, ev, stream);
    }
    const cudaError_t ferr = cudaFreeAsync(ws, stream);
    if (err == cudaSuccess) err = ferr;
    return note_cuda(err);
}

void exact_tc_timing(int enable) {
    std::lock_guard<std::mutex> lk(g_timing_mu);
    if (enable) {
        for (auto &c : g_timing_events)
            for (auto &e : c.e) cudaEventDestroy(e);
        g_timing_events.clear();
        const unsigned long long zero = 0;
        cudaMemcpyToSymbol(g_exact_tc_kgroups, &zero, sizeof zero);
        cudaMemcpyToSymbol(g_exact_tc_repairs, &zero, sizeof zero);
        cudaMemcpyToSymbol(g_exact_tc_fixups, &zero, sizeof zero);
    }
    g_timing_on = enable != 0;
}

// Milliseconds between events a and b of every recorded call, summed.
static cudaError_t sum_between(int a, int b, double *total) {
    *total = 0.0;
    for (auto &c : g_timing_events) {
        if (c.e[a] == nullptr || c.e[b] == nullptr) continue;
        cudaError_t err = cudaEventSynchronize(c.e[b]);
        float t = 0.0f;
        if (err == cudaSuccess) err = cudaEventElapsedTime(&t, c.e[a], c.e[b]);
        if (err != cudaSuccess) return err;
        *total += t;
    }
    return cudaSuccess;
}

carbon_status_t exact_tc_time(double *ms, int64_t *launches, int64_t *kgroups) {
    std::lock_guard<std::mutex> lk(g_timing_mu);
    double total = 0.0;
    const cudaError_t err = sum_between(1, 2, &total);
    if (err != cudaSuccess) return note_cuda(err);
    if (ms) *ms = total;
    if (launches) *launches = (int64_t)g_timing_events.size();
    if (kgroups) {
        unsigned long long v = 0;
        const cudaError_t e2 = cudaMemcpyFromSymbol(&v, g_exact_tc_kgroups, sizeof v);
        if (e2 != cudaSuccess) return note_cuda(e2);
        *kgroups = (int64_t)v;
    }
    return CARBON_OK;
}

carbon_status_t exact_tc_phase_time(double *pre_ms, double *main_ms, double *post_ms) {
    std::lock_guard<std::mutex> lk(g_timing_mu);
    double v[3];
    for (int k = 0; k < 3; ++k) {
        const cudaError_t err = sum_between(k, k + 1, &v[k]);
        if (err != cudaSuccess) return note_cuda(err);
    }
    if (pre_ms) *pre_ms = v[0];
    if (main_ms) *main_ms = v[1];
    if (post_ms) *post_ms = v[2];
    return CARBON_OK;
}

carbon_status_t exact_tc_path_counts(int64_t *repairs, int64_t *fixups) {
    std::lock_guard<std::mutex> lk(g_timing_mu);
    unsigned long long r = 0, f = 0;
    cudaError_t err = cudaDeviceSynchronize();
    if (err == cudaSuccess) err = cudaMemcpyFromSymbol(&r, g_exact_tc_repairs, sizeof r);
    if (err == cudaSuccess) err = cudaMemcpyFromSymbol(&f, g_exact_tc_fixups, sizeof f);
    if (err != cudaSuccess) return note_cuda(err);
    if (repairs) *repairs = (int64_t)r;
    if (fixups) *fixups = (int64_t)f;
    return CARBON_OK;
}

carbon_status_t exact_tc_take_device_status() {
    unsigned int v = 0, f = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_exact_tc_status, sizeof v) != cudaSuccess) return CARBON_OK;
    if (v != 0) cudaMemcpyToSymbol(g_exact_tc_status, &zero, sizeof zero);
    if (cudaMemcpyFromSymbol(&f, g_fixup_status, sizeof f) == cudaSuccess && f != 0)
        cudaMemcpyToSymbol(g_fixup_status, &zero, sizeof zero);
    return (carbon_status_t)(v != 0 ? v : f);
}

}  // namespace carbon
