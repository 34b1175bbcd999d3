// exact_int.cu - exact tier for bf16 operands on the integer pipes.
//
// Same result as exact_kbn.cu, bit for bit: the fixed-order KBN sum of the
// float64 products (256-wide chunks left to right, chunk values fl(s + c)
// combined left to right with KBN), bias in float64, one RNE rounding (Carbon
// README, "How It Works"; sgemm-bi "Determinism contracts" for the downcast).
//
// Why integers give the same bits.  Inside one chunk, if every partial sum of
// the products is exactly representable in float64, then every KBN step is
// exact: t = s + p, the correction is 0, c stays +0, and the chunk value
// fl(s + c) is the exact chunk sum.  The exact sum can then be computed by any
// exact method.  A bf16 value is m * 2^e with |m| < 2^8; over a chunk, row i
// of A is written as X[k] * 2^bx(i) with integers X[k] = m * 2^(e - bx(i))
// (bx = the smallest exponent of the row's significand units), |X| < 2^wx(i);
// likewise column j of B with bw(j), ww(j).  The chunk sum is then
// I * 2^(bx + bw) with I = sum_k X[k] * W[k], an integer dot product that
// IMAD.WIDE computes exactly in int64.  Every partial sum is bounded by
// sum_k |X W| < 256 * 2^(wx + ww) <= 2^53 when wx + ww <= 45, so then every
// partial sum is an integer below 2^53 times 2^(bx + bw): representable, every
// KBN step exact, chunk value = I * 2^(bx + bw).
//
// When that cheap bound fails for a (row, column, chunk), a precise check runs
// on the integer pipes (sum of |X W| below 2^(53 + the lowest set bit of any
// product), which again makes every partial sum representable); only if that
// fails too is the chunk summed with the float64 KBN step from the operands in
// global memory.  On the GPT-2 shapes the cheap bound holds for ~99.9% of
// (output, chunk) pairs.
//
// The outer sum over chunk values uses one DADD per chunk when an integer proof
// shows the addition is exact (both addends are multiples of ulp of the
// result, by the same grain argument as exact_kbn.cu), else the full KBN step.
//
// Structure.  int_prep_kernel converts each operand once into the int32
// operands of every (line, chunk) and that group's base and width (a
// stream-ordered workspace of 4 bytes per operand element, allocated and
// freed on the caller's stream).  exact_int_kernel computes one 64x64 output
// tile per CTA: a producer warp streams 64-deep int32 tiles of both operands
// by TMA into a 4-stage shared-memory ring (mbarrier transaction counts);
// eight consumer warps, 4x4 outputs per thread, run the IMAD.WIDE loop and
// release each stage through an mbarrier, with no CTA-wide barrier in the
// loop.  Every wait is bounded; a wait that gives up records
// CARBON_ERR_TIMEOUT and the CTA winds down.
#include "carbon_internal.h"
#include "device_sync.cuh"
#include "exact_common.cuh"
#include "exact_bf16.cuh"

#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

namespace carbon {
namespace {

__device__ unsigned int g_exact_status = 0;

constexpr int kTile = 64;                  // CTA output tile: 64 x 64
constexpr int kThreads = 256;              // 16 x 16 threads, 4 x 4 outputs each
constexpr int kGrainBad = -0x40000000;
constexpr int kGrainZero = 0x70000000;

// acc += a * b, 32 x 32 -> 64-bit signed multiply-add in one instruction
// (two's-complement wrap; callers only use sums they have bounded).
__device__ __forceinline__ void mad_wide(long long &acc, int a, int b) {
    asm("mad.wide.s32 %0, %1, %2, %0;" : "+l"(acc) : "r"(a), "r"(b));
}

// Precise exactness check of one (row, column, chunk), run by the whole warp
// for the output owned by lane `owner`: every lane loads its eight reduction
// indices up front (one memory latency), then the warp reduces sum |X W| and
// the fewest trailing zero bits t of a nonzero product; every partial sum is
// representable if sum |X W| < 2^(53 + t).  Requires wx, ww <= 31 and
// wx + ww <= 54 for the owner, so sum |X W| < 2^62.  Verdict to every lane.
__device__ __forceinline__ bool warp_exact_precise(const IArgs &p, int owner, int64_t i, int64_t j,
                                                   int64_t q0, int64_t qend, int bx, int bw) {
    const int lane = threadIdx.x % 32;
    i = __shfl_sync(0xffffffffu, i, owner);
    j = __shfl_sync(0xffffffffu, j, owner);
    bx = __shfl_sync(0xffffffffu, bx, owner);
    bw = __shfl_sync(0xffffffffu, bw, owner);
    uint32_t hx[kChunk / 32], hw[kChunk / 32];
#pragma unroll
    for (int t = 0; t < kChunk / 32; ++t) {
        const int64_t r = q0 + lane + 32 * t;
        hx[t] = r < qend ? ld_bits(p.A, i * p.a_si + r * p.a_sr) : 0u;
        hw[t] = r < qend ? ld_bits(p.B, r * p.b_sr + j * p.b_sj) : 0u;
    }
    unsigned long long abs_sum = 0;
    int tz = 1 << 20;
#pragma unroll
    for (int t = 0; t < kChunk / 32; ++t) {
        int mx, ex, mw, ew;
        bool bad_x, bad_w;
        decode(hx[t], mx, ex, bad_x);
        decode(hw[t], mw, ew, bad_w);
        if (mx == 0 || mw == 0) continue;
        const long long X = (long long)mx * (1ll << (ex - bx));      // |X| < 2^31
        const long long W = (long long)mw * (1ll << (ew - bw));
        const long long prod = X * W;
        abs_sum += (unsigned long long)(prod < 0 ? -prod : prod);
        tz = min(tz, __ffsll(prod) - 1);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) abs_sum += __shfl_xor_sync(0xffffffffu, abs_sum, off);
    tz = __reduce_min_sync(0xffffffffu, tz);
    if (abs_sum == 0) return true;
    return tz + 53 >= 64 || abs_sum < (1ull << (tz + 53));
}

// Per-chunk row/column statistics.  For the A tile the "lines" are rows i, for
// the B tile columns j.  Every line gets the minimum exponent of its nonzero
// significand units (base), the maximum, and a flag for inf/NaN.
struct LineStats {
    int emin[kTile], emax[kTile], bad[kTile];
};

template <bool LINE_CONTIG>
__device__ __forceinline__ void gather_stats(const unsigned short *base, int64_t line_stride,
                                             int64_t r_stride, int64_t line0, int64_t nlines,
                                             int64_t q0, int64_t qend, LineStats &st, int tid) {
    const int warp = tid / 32, lane = tid % 32;
    if (!LINE_CONTIG) {
        // reduction index contiguous in memory: warp w owns lines 8w .. 8w+7,
        // lanes walk the chunk 32 at a time (coalesced), then reduce
#pragma unroll 1
        for (int li = 0; li < 8; ++li) {
            const int l = warp * 8 + li;
            int lo = 1 << 20, hi = -(1 << 20), bad = 0;
            if (line0 + l < nlines) {
                for (int64_t r = q0 + lane; r < qend; r += 32) {
                    int m, e;
                    bool b;
                    decode(ld_bits(base, (line0 + l) * line_stride + r * r_stride), m, e, b);
                    if (m != 0) { lo = min(lo, e); hi = max(hi, e); }
                    bad |= (int)b;
                }
            }
            lo = __reduce_min_sync(0xffffffffu, lo);
            hi = __reduce_max_sync(0xffffffffu, hi);
            bad = __reduce_or_sync(0xffffffffu, (unsigned)bad);
            if (lane == 0) { st.emin[l] = lo; st.emax[l] = hi; st.bad[l] = bad; }
        }
    } else {
        // lines contiguous in memory: lane = line (two halves), warp w walks a
        // slice of the reduction; combine the 8 warps with shared atomics
        int lo[2], hi[2], bad[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) { lo[h] = 1 << 20; hi[h] = -(1 << 20); bad[h] = 0; }
        for (int64_t r = q0 + warp; r < qend; r += 8) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int l = lane + 32 * h;
                if (line0 + l < nlines) {
                    int m, e;
                    bool b;
                    decode(ld_bits(base, (line0 + l) * line_stride + r * r_stride), m, e, b);
                    if (m != 0) { lo[h] = min(lo[h], e); hi[h] = max(hi[h], e); }
                    bad[h] |= (int)b;
                }
            }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int l = lane + 32 * h;
            atomicMin(&st.emin[l], lo[h]);
            atomicMax(&st.emax[l], hi[h]);
            atomicOr(&st.bad[l], bad[h]);
        }
    }
}

// ---- pre-pass: int32 operands and per-(line, chunk) statistics --------------

// T[r * Lp + line] = m * 2^(e - base(line, chunk of r)) for lines whose width
// fits int32, else 0 (those outputs never use the integer sum).  Rows past R,
// up to the padded length Rp, and lines past nlines are 0.  stats[chunk * Lp +
// line] = (base, width, bits of sum |T|, bits of max |T|) over the chunk.
template <bool LINE_CONTIG>
__global__ void __launch_bounds__(kThreads)
int_prep_kernel(const unsigned short *src, int64_t line_stride, int64_t r_stride, int64_t nlines,
                int64_t R, int64_t Rp, int64_t Lp, int *T, int4 *stats) {
    __shared__ LineStats st;
    __shared__ int lbase[kTile], lwidth[kTile];
    __shared__ unsigned long long lsum[kTile];
    __shared__ unsigned int lmax[kTile];
    __shared__ unsigned short raw[kTile][kChunk + 2];     // transpose buffer (reduction-contiguous sources)
    const int tid = threadIdx.x;
    const int64_t line0 = (int64_t)blockIdx.x * kTile;
    const int64_t q0 = (int64_t)blockIdx.y * kChunk;
    const int64_t qend = (R - q0 > kChunk) ? q0 + kChunk : R;
    const int64_t rtop = (Rp - q0 > kChunk) ? q0 + kChunk : Rp;

    if (tid < kTile) {
        st.emin[tid] = 1 << 20; st.emax[tid] = -(1 << 20); st.bad[tid] = 0;
        lsum[tid] = 0ull; lmax[tid] = 0u;
    }
    __syncthreads();
    gather_stats<LINE_CONTIG>(src, line_stride, r_stride, line0, nlines, q0, qend, st, tid);
    __syncthreads();
    if (tid < kTile) {
        const int lo = st.emin[tid], hi = st.emax[tid];
        lbase[tid] = (lo > hi) ? 0 : lo;                        // all-zero line: base 0
        lwidth[tid] = st.bad[tid] ? kWidthBad : ((lo > hi) ? 0 : hi + 8 - lo);
    }
    if (!LINE_CONTIG) {
        // coalesced read along the reduction into shared memory
        for (int e = tid; e < kTile * kChunk; e += kThreads) {
            const int l = e / kChunk, rr = e % kChunk;
            const int64_t line = line0 + l, r = q0 + rr;
            raw[l][rr] = (line < nlines && r < qend) ? src[line * line_stride + r * r_stride] : 0;
        }
    }
    __syncthreads();
    const int rows_here = (int)(rtop - q0);
    // every thread keeps one line (kThreads is a multiple of kTile)
    unsigned long long my_sum = 0ull;
    unsigned int my_max = 0u;
    for (int e = tid; e < kTile * rows_here; e += kThreads) {
        const int l = e % kTile, rr = e / kTile;
        const int64_t line = line0 + l, r = q0 + rr;
        int v = 0;
        if (line < nlines && r < qend && lwidth[l] <= 31) {
            const uint32_t h = LINE_CONTIG ? (uint32_t)src[line * line_stride + r * r_stride]
                                           : (uint32_t)raw[l][rr];
            int m, ex;
            bool b;
            decode(h, m, ex, b);
            if (m != 0) v = m * (1 << (ex - lbase[l]));          // shift <= 23: |v| < 2^31
        }
        T[r * Lp + line] = v;
        const unsigned int av = (unsigned int)(v < 0 ? -v : v);
        my_sum += av;
        my_max = max(my_max, av);
    }
    atomicAdd(&lsum[tid % kTile], my_sum);
    atomicMax(&lmax[tid % kTile], my_max);
    __syncthreads();
    if (tid < kTile)
        stats[(int64_t)blockIdx.y * Lp + line0 + tid] =
            make_int4(lbase[tid], lwidth[tid], bit_count(lsum[tid]), bit_count(lmax[tid]));
}

// ---- main kernel --------------------------------------------------------------

constexpr int kStageK = 32;                          // reduction rows per ring stage
constexpr int kStages = 4;
constexpr int kStagesPerChunk = kChunk / kStageK;
constexpr int kConsumerWarps = 8;
constexpr int kMainThreads = (kConsumerWarps + 1) * 32;
constexpr uint32_t kTileBytes = kStageK * kTile * 4; // 8 KiB per operand per stage

struct __align__(1024) MainSmem {
    int X[kStages][kStageK][kTile];
    int W[kStages][kStageK][kTile];
    double C[16][kConsumerWarps * 32];               // outer KBN compensation, per output
    uint64_t full[kStages], empty[kStages];
    uint32_t abort;
};

template <int PASS, bool OUT_F64>
__global__ void __launch_bounds__(kMainThreads, 1)
exact_int_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                 const IArgs p, const int4 *__restrict__ SA, const int4 *__restrict__ SB,
                 int64_t LpA, int64_t LpB, int64_t Rp, unsigned int *__restrict__ work_count,
                 unsigned int *__restrict__ work_list) {
    extern __shared__ uint8_t smem_raw[];
    MainSmem &sm = *reinterpret_cast<MainSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x;
    const int warp = tid / 32, lane = tid % 32;
    const int64_t i0 = (blockIdx.x / p.tiles_n) * kTile;
    const int64_t j0 = (blockIdx.x % p.tiles_n) * kTile;
    const int nstages = (int)(Rp / kStageK);
    volatile uint32_t *abort_flag = &sm.abort;

    if (tid == 0) {
        for (int st = 0; st < kStages; ++st) {
            mbar_init(smem_addr(&sm.full[st]), 1);
            mbar_init(smem_addr(&sm.empty[st]), kConsumerWarps);
        }
        *abort_flag = 0u;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_map(&map_a);
            prefetch_map(&map_b);
            int issued = 0;
            for (int g = 0; g < nstages && !*abort_flag; ++g) {
                const int st = g % kStages;
                const uint32_t use = (uint32_t)(g / kStages);
                if (!mbar_wait(smem_addr(&sm.empty[st]), (use & 1u) ^ 1u)) {
                    *abort_flag = 1u;
                    atomicExch(&g_exact_status, (unsigned)CARBON_ERR_TIMEOUT);
                    break;
                }
                const uint32_t fb = smem_addr(&sm.full[st]);
                mbar_arrive_expect_tx(fb, 2 * kTileBytes);
                tma_load_2d(smem_addr(&sm.X[st][0][0]), &map_a, fb, (int)i0, g * kStageK);
                tma_load_2d(smem_addr(&sm.W[st][0][0]), &map_b, fb, (int)j0, g * kStageK);
                issued = g + 1;
            }
            // every issued load lands before the CTA may exit
            for (int g = (issued > kStages ? issued - kStages : 0); g < issued; ++g)
                if (!mbar_wait(smem_addr(&sm.full[g % kStages]), (uint32_t)(g / kStages) & 1u)) break;
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int tx = tid % 16, ty = tid / 16;               // 16 x 16 consumer threads
    double S[4][4];
    long long acc[4][4];
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int n = 0; n < 4; ++n) { S[m][n] = 0.0; acc[m][n] = 0ll; sm.C[4 * m + n][tid] = 0.0; }
    // Outer grain: the running sum S is a multiple of 2^(min over chunks of
    // rb + cb); (min rb) + (min cb) over the chunks with nonzero products is a
    // lower bound of that, kept per line (rows of this thread, columns of this
    // thread).  A line that held inf/NaN makes every later outer step take the
    // full KBN step.
    int rbmin[4], cbmin[4];
    bool rbad[4], cbad[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) { rbmin[m] = 1 << 20; cbmin[m] = 1 << 20; rbad[m] = false; cbad[m] = false; }
    // outputs with a chunk the bounds cannot prove: left to the fix-up pass
    unsigned int deferred = 0u;

    for (int g = 0; g < nstages; ++g) {
        const int st = g % kStages;
        if (!mbar_wait(smem_addr(&sm.full[st]), (uint32_t)(g / kStages) & 1u)) {
            *abort_flag = 1u;
            atomicExch(&g_exact_status, (unsigned)CARBON_ERR_TIMEOUT);
            break;
        }
#pragma unroll 8
        for (int k = 0; k < kStageK; ++k) {
            const int4 a4 = *reinterpret_cast<const int4 *>(&sm.X[st][k][4 * ty]);
            const int4 b4 = *reinterpret_cast<const int4 *>(&sm.W[st][k][4 * tx]);
            const int a[4] = {a4.x, a4.y, a4.z, a4.w};
            const int b[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
            for (int m = 0; m < 4; ++m)
#pragma unroll
                for (int n = 0; n < 4; ++n)
                    mad_wide(acc[m][n], a[m], b[n]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&sm.empty[st]));

        const bool chunk_end = ((g + 1) % kStagesPerChunk == 0) || (g == nstages - 1);
        if (!chunk_end) continue;
        // ---- chunk values and the outer KBN step
        const int q = g / kStagesPerChunk;
        int rbx[4], rwx[4], rsx[4], rmx[4], cbw[4], cww[4], csw[4], cmw[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int4 v = __ldg(&SA[(int64_t)q * LpA + i0 + 4 * ty + m]);
            rbx[m] = v.x; rwx[m] = v.y; rsx[m] = v.z; rmx[m] = v.w;
            if (v.y == kWidthBad) rbad[m] = true;
            else if (v.y > 0) rbmin[m] = min(rbmin[m], v.x);
        }
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            const int4 v = __ldg(&SB[(int64_t)q * LpB + j0 + 4 * tx + n]);
            cbw[n] = v.x; cww[n] = v.y; csw[n] = v.z; cmw[n] = v.w;
            if (v.y == kWidthBad) cbad[n] = true;
            else if (v.y > 0) cbmin[n] = min(cbmin[n], v.x);
        }
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                const int o = 4 * m + n;
                const int wx = rwx[m], ww = cww[n];
                const int64_t i = i0 + 4 * ty + m, j = j0 + 4 * tx + n;
                // every partial sum below 2^53 (in units of 2^(bx + bw)) if
                // sum_k |X W| < 256 * 2^(wx + ww) <= 2^53, or if
                // sum_k |X W| <= (sum |X|) (max |W|) or (max |X|) (sum |W|) < 2^53
                const bool fits = wx <= 31 && ww <= 31;
                bool proven = fits && (wx + ww <= 45 || min(rsx[m] + cmw[n], rmx[m] + csw[n]) <= 53);
                if (i >= p.rows || j >= p.cols) proven = true;        // padding output
                const bool checkable = !proven && fits && wx + ww <= 54;
                unsigned pending = __ballot_sync(0xffffffffu, checkable);
                while (pending) {                                      // the warp checks together
                    const int owner = __ffs(pending) - 1;
                    pending &= pending - 1;
                    const int64_t q0 = (int64_t)q * kChunk;
                    const int64_t qend = (p.R - q0 > kChunk) ? q0 + kChunk : p.R;
                    const bool ok = warp_exact_precise(p, owner, i, j, q0, qend, rbx[m], cbw[n]);
                    if (lane == owner) proven = ok;
                }
                if (!proven) deferred |= 1u << o;
                const double P = scaled_int_to_double(acc[m][n], rbx[m] + cbw[n]);
                acc[m][n] = 0ll;
                if (deferred & (1u << o)) continue;               // recomputed by the fix-up pass
                // P and S are multiples of 2^(rbmin + cbmin): if that is at least
                // ulp(S + P), the addition is exact and C is unchanged.
                const int G = (rbad[m] || cbad[n]) ? kGrainBad
                              : (rbmin[m] + cbmin[n] > (1 << 19)) ? kGrainZero
                              : (rbmin[m] + cbmin[n] + 1075) << 20;
                const double t = __dadd_rn(S[m][n], P);
                const bool inexact = (__double2hiint(t) & 0x7ff00000) > G;
                if (!inexact) {
                    S[m][n] = t;
                } else {
                    double c = sm.C[o][tid];
                    kbn_value_step(S[m][n], c, P);
                    sm.C[o][tid] = c;
                }
            }
    }

    // ---- bias, one rounding, store
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const int64_t i = i0 + 4 * ty + m;
        if (i >= p.rows) continue;
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            const int64_t j = j0 + 4 * tx + n;
            if (j >= p.cols) continue;
            const int64_t o = i * p.cols + j;
            if ((deferred >> (4 * m + n)) & 1u) {                // for the fix-up pass
                work_list[atomicAdd(work_count, 1u)] = (unsigned int)o;
                continue;
            }
            double y = __dadd_rn(S[m][n], sm.C[4 * m + n][tid]);
            if (p.bias) y = __dadd_rn(y, widen_bf16(ld_bits(p.bias, j)));
            if (OUT_F64) static_cast<double *>(p.out)[o] = y;
            else static_cast<unsigned short *>(p.out)[o] = exact_round_bf16(y);
        }
    }
}


template <int PASS, bool F64>
cudaError_t launch_main(const CUtensorMap &ma, const CUtensorMap &mb, const IArgs &a, int64_t tiles,
                        const int4 *SA, const int4 *SB, int64_t LpA, int64_t LpB, int64_t Rp,
                        unsigned int *work, cudaStream_t s) {
    // work[0] = number of deferred outputs, work[1..] = their indices
    cudaError_t err = cudaMemsetAsync(work, 0, sizeof(unsigned int), s);
    if (err != cudaSuccess) return err;
    auto kern = exact_int_kernel<PASS, F64>;
    const int smem = (int)sizeof(MainSmem) + 1024;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    kern<<<(unsigned)tiles, kMainThreads, smem, s>>>(ma, mb, a, SA, SB, LpA, LpB, Rp, work, work + 1);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    exact_fixup_kernel<F64><<<kFixBlocks, kFixWarps * 32, 0, s>>>(a, SA, SB, LpA, LpB, work, work + 1);
    count_launch();
    return cudaGetLastError();
}

template <int PASS>
cudaError_t launch_main_pass(bool f64, const CUtensorMap &ma, const CUtensorMap &mb, const IArgs &a,
                             int64_t tiles, const int4 *SA, const int4 *SB, int64_t LpA,
                             int64_t LpB, int64_t Rp, unsigned int *work, cudaStream_t s) {
    return f64 ? launch_main<PASS, true>(ma, mb, a, tiles, SA, SB, LpA, LpB, Rp, work, s)
               : launch_main<PASS, false>(ma, mb, a, tiles, SA, SB, LpA, LpB, Rp, work, s);
}

}  // namespace

carbon_status_t exact_int_launch(const Problem &p, bool out_f64, cudaStream_t stream) {
    if (p.rows == 0 || p.cols == 0) return CARBON_OK;
    // the deferral list holds 32-bit output indices; larger outputs run the
    // float64 kernel, which computes the same bits
    if (p.rows * p.cols >= ((int64_t)1 << 32)) return exact_launch(p, out_f64, stream);
    IArgs a;
    a.A = static_cast<const unsigned short *>(p.A);
    a.B = static_cast<const unsigned short *>(p.B);
    a.bias = static_cast<const unsigned short *>(p.bias);
    a.out = p.out;
    a.rows = p.rows; a.cols = p.cols; a.R = p.R;
    switch (p.pass) {
    case CARBON_PASS_FWD: a.a_si = p.K; a.a_sr = 1; a.b_sr = p.N; a.b_sj = 1; break;
    case CARBON_PASS_DX:  a.a_si = p.N; a.a_sr = 1; a.b_sr = 1;   a.b_sj = p.N; break;
    default:              a.a_si = 1;   a.a_sr = p.K; a.b_sr = p.N; a.b_sj = 1; break;
    }
    a.tiles_n = (p.cols + kTile - 1) / kTile;
    const int64_t tiles_m = (p.rows + kTile - 1) / kTile;
    const int64_t tiles = tiles_m * a.tiles_n;
    if (tiles > 0x7fffffff) return CARBON_ERR_INVALID_ARG;
    const int64_t LpA = tiles_m * kTile, LpB = a.tiles_n * kTile;
    const int64_t Rp = ((p.R + 63) / 64) * 64;
    const int64_t nchunks = (p.R + kChunk - 1) / kChunk;
    if (nchunks > 65535) return CARBON_ERR_INVALID_ARG;

    // workspace: int32 operands [Rp][Lp] of A and B, the statistics of every
    // (chunk, line), one deferral flag per output; stream-ordered, released at
    // the end of this call
    const size_t tA = (size_t)Rp * LpA, tB = (size_t)Rp * LpB;
    const size_t bytes = 4 * (tA + tB) + 16 * (size_t)nchunks * (LpA + LpB) +
                         4 * ((size_t)p.rows * (size_t)p.cols + 1);
    char *ws = nullptr;
    cudaError_t err = cudaSuccess;
    if (bytes > 0) {
        err = cudaMallocAsync(reinterpret_cast<void **>(&ws), bytes, stream);
        if (err != cudaSuccess) return note_cuda(err);
    }
    int *TA = reinterpret_cast<int *>(ws);
    int *TB = TA + tA;
    int4 *SA = reinterpret_cast<int4 *>(TB + tB);
    int4 *SB = SA + (size_t)nchunks * LpA;
    unsigned int *work = reinterpret_cast<unsigned int *>(SB + (size_t)nchunks * LpB);

    const bool a_contig = (p.pass == CARBON_PASS_DW), b_contig = (p.pass != CARBON_PASS_DX);
    if (nchunks > 0) {
        const dim3 ga((unsigned)tiles_m, (unsigned)nchunks), gb((unsigned)a.tiles_n, (unsigned)nchunks);
        if (a_contig) int_prep_kernel<true><<<ga, kThreads, 0, stream>>>(a.A, a.a_si, a.a_sr, p.rows, p.R, Rp, LpA, TA, SA);
        else int_prep_kernel<false><<<ga, kThreads, 0, stream>>>(a.A, a.a_si, a.a_sr, p.rows, p.R, Rp, LpA, TA, SA);
        if (b_contig) int_prep_kernel<true><<<gb, kThreads, 0, stream>>>(a.B, a.b_sj, a.b_sr, p.cols, p.R, Rp, LpB, TB, SB);
        else int_prep_kernel<false><<<gb, kThreads, 0, stream>>>(a.B, a.b_sj, a.b_sr, p.cols, p.R, Rp, LpB, TB, SB);
        count_launch(2);
        err = cudaGetLastError();
    }
    // int32 tiles: 64 lines x 64 reduction rows per TMA box, no swizzle
    CUtensorMap ma, mb;
    if (err == cudaSuccess && nchunks > 0) {
        err = encode_tensor_map_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_INT32, TA, (uint64_t)LpA, (uint64_t)Rp,
                                   (uint64_t)LpA * 4, kTile, kStageK, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (err == cudaSuccess)
            err = encode_tensor_map_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_INT32, TB, (uint64_t)LpB,
                                       (uint64_t)Rp, (uint64_t)LpB * 4, kTile, kStageK,
                                       CU_TENSOR_MAP_SWIZZLE_NONE);
    } else {
        std::memset(&ma, 0, sizeof ma);
        std::memset(&mb, 0, sizeof mb);
    }
    if (err == cudaSuccess) {
        switch (p.pass) {
        case CARBON_PASS_FWD: err = launch_main_pass<CARBON_PASS_FWD>(out_f64, ma, mb, a, tiles, SA, SB, LpA, LpB, Rp, work, stream); break;
        case CARBON_PASS_DX:  err = launch_main_pass<CARBON_PASS_DX>(out_f64, ma, mb, a, tiles, SA, SB, LpA, LpB, Rp, work, stream); break;
        default:              err = launch_main_pass<CARBON_PASS_DW>(out_f64, ma, mb, a, tiles, SA, SB, LpA, LpB, Rp, work, stream); break;
        }
        count_launch();
    }
    if (ws) {
        const cudaError_t ferr = cudaFreeAsync(ws, stream);
        if (err == cudaSuccess) err = ferr;
    }
    return note_cuda(err);
}

carbon_status_t exact_take_device_status() {
    unsigned int v = 0, f = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_exact_status, sizeof v) != cudaSuccess) return CARBON_OK;
    if (v != 0) cudaMemcpyToSymbol(g_exact_status, &zero, sizeof zero);
    if (cudaMemcpyFromSymbol(&f, g_fixup_status, sizeof f) == cudaSuccess && f != 0)
        cudaMemcpyToSymbol(g_fixup_status, &zero, sizeof zero);
    return (carbon_status_t)(v != 0 ? v : f);
}

}  // namespace carbon

// ---- bf16 exact tier without any device allocation ----------------------------
//
// Some callers cannot allocate device memory while they run: code inside a
// framework whose allocator owns every byte of the GPU, code on a path that
// must never block on or fail in an allocator (a latency-critical serving
// loop, a watchdog), or a process where the stream-ordered pool is
// unavailable.  For them carbon_gemm_exact_bf16_noalloc runs the same two
// kernels as the bf16 exact tier above, with the workspace taken from a
// fixed array in device memory.  The array belongs to this file's module,
// which CUDA loads onto a device (reserving the array there) the first time
// the module is used on that device -- under the default lazy module loading
// that is the first no-allocation call on that device.  Callers whose
// allocator later takes all free memory, or who capture streams, should make
// one small call on each device beforehand.

namespace carbon {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)64 << 20;   // 64 MiB per device

// Fixed workspace of the no-allocation entry point.  Every GPU on which the
// module has been loaded holds it until the process exits.  Host code must not use the
// symbol as an address (it is a host-side stand-in); the device address comes
// from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Driver calls that identify the current context, fetched through the
// runtime (the library does not link libcuda).
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_once;

void find_context_calls() {
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
        g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
        g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
}

struct ScratchSlot {
    unsigned long long ctx_id;   // context the address belongs to (0 = none yet)
    void *ptr;
};
std::mutex g_noalloc_mu;
ScratchSlot g_noalloc_slot[128];

// Unique id of the calling thread's current context, or 0 if none is current
// or the driver cannot say.
unsigned long long current_context_id() {
    std::call_once(g_ctx_once, find_context_calls);
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (g_ctx_current && g_ctx_id && g_ctx_current(&ctx) == CUDA_SUCCESS && ctx != nullptr &&
        g_ctx_id(ctx, &id) == CUDA_SUCCESS)
        return id;
    return 0;
}

// Device address of g_noalloc_scratch in the current device's current
// context.  It is looked up with cudaGetSymbolAddress once per device and
// context: the first call on a device loads this file's module there (under
// CUDA's default lazy loading), which is when the 64 MiB array is reserved,
// and a new context (after cudaDeviceReset, say) gets a fresh lookup rather
// than a stale address.  If the context cannot be identified the address is
// looked up on every call (cheap once the module is loaded).
cudaError_t noalloc_scratch(void **ptr) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    unsigned long long id = current_context_id();
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    ScratchSlot &slot = g_noalloc_slot[dev];
    if (id == 0 || slot.ctx_id != id || slot.ptr == nullptr) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess) return err;
        // the lookup makes the device's primary context current if no
        // context was, so ask again for the identity to cache it under
        if (id == 0) id = current_context_id();
        slot.ptr = p;
        slot.ctx_id = id;
    }
    *ptr = slot.ptr;
    return cudaSuccess;
}

}  // namespace
}  // namespace carbon

extern "C" carbon_status_t carbon_gemm_exact_bf16_noalloc(carbon_pass_t pass, void *out,
                                                          const void *A, const void *B,
                                                          const void *bias, int64_t M, int64_t K,
                                                          int64_t N, carbon_stream_t stream) {
    using namespace carbon;
    if (pass < CARBON_PASS_FWD || pass > CARBON_PASS_DW) return CARBON_ERR_INVALID_ARG;
    if (M < 0 || K < 0 || N < 0) return CARBON_ERR_INVALID_ARG;
    int64_t mk, kn, mn;
    if (__builtin_mul_overflow(M, K, &mk) || __builtin_mul_overflow(K, N, &kn) ||
        __builtin_mul_overflow(M, N, &mn))
        return CARBON_ERR_INVALID_ARG;
    int64_t bytes;   // byte counts must fit as well, as in the other entry points
    if (__builtin_mul_overflow(mk, 8, &bytes) || __builtin_mul_overflow(kn, 8, &bytes) ||
        __builtin_mul_overflow(mn, 8, &bytes))
        return CARBON_ERR_INVALID_ARG;
    const Problem p = make_problem(pass, CARBON_BF16, out, A, B, bias, M, K, N);
    const int64_t a_elems = (pass == CARBON_PASS_DX) ? mn : mk;
    const int64_t b_elems = (pass == CARBON_PASS_DW) ? mn : kn;
    const int64_t out_elems = p.rows * p.cols;
    if (out_elems == 0) return CARBON_OK;
    if (out == nullptr || (a_elems > 0 && A == nullptr) || (b_elems > 0 && B == nullptr))
        return CARBON_ERR_INVALID_ARG;

    // the same workspace layout as exact_int_launch, checked against the array
    const int64_t tiles_m = (p.rows + kTile - 1) / kTile, tiles_n = (p.cols + kTile - 1) / kTile;
    const int64_t LpA = tiles_m * kTile, LpB = tiles_n * kTile;
    const int64_t Rp = ((p.R + 63) / 64) * 64;
    const int64_t nchunks = (p.R + kChunk - 1) / kChunk;
    if (tiles_m * tiles_n > 0x7fffffff || nchunks > 65535) return CARBON_ERR_INVALID_ARG;
    if (out_elems >= ((int64_t)1 << 32)) return CARBON_ERR_SCRATCH_LIMIT;
    const double need = 4.0 * (double)Rp * (double)(LpA + LpB) +
                        16.0 * (double)nchunks * (double)(LpA + LpB) + 4.0 * ((double)out_elems + 1.0);
    if (need > (double)kNoAllocScratchBytes) return CARBON_ERR_SCRATCH_LIMIT;

    carbon_status_t st = injected_launch_failure();
    if (st != CARBON_OK) return st;
    st = current_device(nullptr, nullptr);
    if (st != CARBON_OK) return st;
    void *scratch = nullptr;
    cudaError_t err = noalloc_scratch(&scratch);
    if (err != cudaSuccess) return note_cuda(err);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    IArgs a;
    a.A = static_cast<const unsigned short *>(p.A);
    a.B = static_cast<const unsigned short *>(p.B);
    a.bias = static_cast<const unsigned short *>(p.bias);
    a.out = p.out;
    a.rows = p.rows; a.cols = p.cols; a.R = p.R;
    switch (p.pass) {
    case CARBON_PASS_FWD: a.a_si = p.K; a.a_sr = 1; a.b_sr = p.N; a.b_sj = 1; break;
    case CARBON_PASS_DX:  a.a_si = p.N; a.a_sr = 1; a.b_sr = 1;   a.b_sj = p.N; break;
    default:              a.a_si = 1;   a.a_sr = p.K; a.b_sr = p.N; a.b_sj = 1; break;
    }
    a.tiles_n = tiles_n;
    const size_t tA = (size_t)Rp * LpA, tB = (size_t)Rp * LpB;
    int *TA = static_cast<int *>(scratch);
    int *TB = TA + tA;
    int4 *SA = reinterpret_cast<int4 *>(TB + tB);
    int4 *SB = SA + (size_t)nchunks * LpA;
    unsigned int *work = reinterpret_cast<unsigned int *>(SB + (size_t)nchunks * LpB);

    // Only the deferral counter has to start at zero; it is cleared on the
    // stream before the main kernel.  The pre-pass writes every operand word
    // and statistic, and the main kernel every list entry it counts, before
    // they are read in this same call.
    CUtensorMap ma, mb;
    std::memset(&ma, 0, sizeof ma);
    std::memset(&mb, 0, sizeof mb);
    if (nchunks > 0) {
        const dim3 ga((unsigned)tiles_m, (unsigned)nchunks), gb((unsigned)tiles_n, (unsigned)nchunks);
        if (p.pass == CARBON_PASS_DW) int_prep_kernel<true><<<ga, kThreads, 0, s>>>(a.A, a.a_si, a.a_sr, p.rows, p.R, Rp, LpA, TA, SA);
        else int_prep_kernel<false><<<ga, kThreads, 0, s>>>(a.A, a.a_si, a.a_sr, p.rows, p.R, Rp, LpA, TA, SA);
        if (p.pass != CARBON_PASS_DX) int_prep_kernel<true><<<gb, kThreads, 0, s>>>(a.B, a.b_sj, a.b_sr, p.cols, p.R, Rp, LpB, TB, SB);
        else int_prep_kernel<false><<<gb, kThreads, 0, s>>>(a.B, a.b_sj, a.b_sr, p.cols, p.R, Rp, LpB, TB, SB);
        count_launch(2);
        err = cudaGetLastError();
        if (err == cudaSuccess)
            err = encode_tensor_map_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_INT32, TA, (uint64_t)LpA, (uint64_t)Rp,
                                       (uint64_t)LpA * 4, kTile, kStageK, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (err == cudaSuccess)
            err = encode_tensor_map_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_INT32, TB, (uint64_t)LpB, (uint64_t)Rp,
                                       (uint64_t)LpB * 4, kTile, kStageK, CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    if (err == cudaSuccess) {
        const int64_t tiles = tiles_m * tiles_n;
        switch (p.pass) {
        case CARBON_PASS_FWD: err = launch_main_pass<CARBON_PASS_FWD>(false, ma, mb, a, tiles, SA, SB, LpA, LpB, Rp, work, s); break;
        case CARBON_PASS_DX:  err = launch_main_pass<CARBON_PASS_DX>(false, ma, mb, a, tiles, SA, SB, LpA, LpB, Rp, work, s); break;
        default:              err = launch_main_pass<CARBON_PASS_DW>(false, ma, mb, a, tiles, SA, SB, LpA, LpB, Rp, work, s); break;
        }
        count_launch();
    }
    return note_cuda(err);
}
