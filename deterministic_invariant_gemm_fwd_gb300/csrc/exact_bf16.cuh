// exact_bf16.cuh - pieces shared by the two bf16 kernels of the exact tier
// (exact_int.cu on the integer pipes, exact_tc.cu on the tensor cores): the
// operand decoding, the per-(line, chunk) statistics format, and the fix-up
// kernel that recomputes an output whose chunks the fast paths could not prove.
//
// Statistics.  For a line (a row i of A or a column j of B) and a chunk of 256
// reduction indices, the bf16 values are m * 2^e with |m| < 2^8; the line's
// base is an exponent of which every value is an integer multiple (the
// integer-pipe kernel takes the smallest e of a nonzero value, the
// tensor-core kernel the smallest e + tz, tz the trailing zero bits of m) and
// its integers are X = m * 2^(e - base) (line_int).  stats[chunk * Lp + line] =
// (base, width, bits of sum |X|, bits of max |X|) with |X| < 2^width; width 0
// for an all-zero line, kWidthBad for a line holding inf or NaN.
#pragma once

#include "bounds.cuh"
#include "carbon_internal.h"
#include "device_sync.cuh"
#include "exact_common.cuh"

namespace carbon {
namespace {

constexpr int kChunk = 256;
constexpr int kWidthBad = 99;              // width of a row/column holding inf/NaN

struct IArgs {
    const unsigned short *A, *B, *bias;
    void *out;
    int64_t rows, cols, R;
    int64_t a_si, a_sr, b_sr, b_sj;
    int64_t tiles_n;
};

// bf16 bits -> value = m * 2^e with m a signed integer, |m| < 2^8 (subnormals
// share the scale of the smallest normal binade).  Flags inf/NaN.
__device__ __forceinline__ void decode(uint32_t h, int &m, int &e, bool &bad) {
    const int e8 = (int)((h >> 7) & 0xffu);
    const int mag = (e8 ? 128 : 0) | (int)(h & 0x7fu);
    m = (h & 0x8000u) ? -mag : mag;
    e = (e8 ? e8 : 1) - 134;
    bad = (e8 == 0xff);
}

// The integer X = m * 2^(e - base) of a value on its line's grid.  A line's
// base may lie above e when m has trailing zero bits (m * 2^e is still a
// multiple of 2^base), then the shift is a right shift that drops only zeros.
__device__ __forceinline__ long long line_int(int m, int e, int base) {
    const int d = e - base;
    return d >= 0 ? (long long)m * (1ll << d) : (long long)(m >> -d);
}

__device__ __forceinline__ uint32_t ld_bits(const unsigned short *base, int64_t idx) {
    return (uint32_t)__ldg(base + idx);
}

// Exact float64 of an integer with at most 53 significant bits, times 2^b.
__device__ __forceinline__ double scaled_int_to_double(long long I, int b) {
    if (I == 0) return 0.0;
    const unsigned long long sign = (unsigned long long)I & 0x8000000000000000ull;
    const unsigned long long mag = sign ? (unsigned long long)(-I) : (unsigned long long)I;
    const int lz = __clzll((long long)mag);
    const int exp2 = 63 - lz + b;                          // value in [2^exp2, 2^(exp2+1))
    const unsigned long long frac = ((mag << lz) << 1) >> 12;  // 52 stored bits (exact: <= 53 significant)
    return __longlong_as_double((long long)(sign | ((unsigned long long)(exp2 + 1023) << 52) | frac));
}

__device__ __forceinline__ double widen_bf16(uint32_t h) { return widen(h << 16); }

// Float64 nearest to mag * 2^b (ties to even), sign from neg; mag < 2^nbits,
// nbits = 0 for mag = 0.  The caller keeps the result inside the normal range.
__device__ __forceinline__ double round_mag_to_double(unsigned long long mag, int nbits, bool neg,
                                                      int b) {
    if (mag == 0ull) return 0.0;
    unsigned long long m = mag;
    int e = nbits - 1 + b;                                  // value in [2^e, 2^(e+1))
    if (nbits > 53) {
        const int sh = nbits - 53;
        const unsigned long long rem = mag & ((1ull << sh) - 1ull), half = 1ull << (sh - 1);
        m = mag >> sh;
        m += (rem > half || (rem == half && (m & 1ull))) ? 1ull : 0ull;
        if (m >> 53) { m >>= 1; ++e; }
    } else {
        m <<= 53 - nbits;
    }
    return __longlong_as_double((long long)((neg ? 0x8000000000000000ull : 0ull) |
                                            ((unsigned long long)(e + 1023) << 52) |
                                            (m & 0x000fffffffffffffull)));
}

// Float64 nearest to I * 2^b (ties to even).
__device__ __forceinline__ double round_int_to_double(long long I, int b) {
    const bool neg = I < 0;
    const unsigned long long mag = neg ? 0ull - (unsigned long long)I : (unsigned long long)I;
    return round_mag_to_double(mag, 64 - __clzll((long long)mag), neg, b);
}

// Float64 nearest to I * 2^b (ties to even) for a 128-bit integer: the top
// 64 significant bits with the rest folded into a sticky bit round the same.
__device__ __forceinline__ double round_i128_to_double(__int128 I, int b) {
    const bool neg = I < 0;
    const unsigned __int128 mag = neg ? (unsigned __int128)0 - (unsigned __int128)I : (unsigned __int128)I;
    const unsigned long long hi = (unsigned long long)(mag >> 64), lo = (unsigned long long)mag;
    if (hi == 0ull) return round_mag_to_double(lo, 64 - __clzll((long long)lo), neg, b);
    const int nbits = 128 - __clzll((long long)hi);         // 65 .. 128
    const int sh = nbits - 64;                              // keep 64 bits, sticky the rest
    const unsigned long long top = (unsigned long long)(mag >> sh);
    const unsigned long long sticky = (mag & (((unsigned __int128)1 << sh) - 1)) != 0 ? 1ull : 0ull;
    return round_mag_to_double(top | sticky, 64, neg, b + sh);
}

// Bits needed for an unsigned value (0 for 0): v < 2^bits.
__device__ __forceinline__ int bit_count(unsigned long long v) { return 64 - __clzll((long long)v); }

// ---- fix-up pass: outputs the fast kernels left undone ----------------------
//
// One block per listed output recomputes it from the bf16 operands.  Its 32
// warps take 32 chunks at a time (a 256-deep chunk of the literal loop below
// is a chain of 256 dependent steps, so chunks in separate warps rather than
// in turn): the 32 lanes of a warp load the chunk's
// 256 operand pairs at once and reduce the exact chunk sum in 128-bit
// integers; the chunk value is that sum rounded once to float64 (see the
// argument in the loop).  Chunks with inf or NaN operands, or of extreme
// width, run the float64 KBN loop on the warp's lane 0 from shared memory.
// Thread 0 then combines the chunk values in order with the full KBN step, and
// finally adds the bias and rounds.  Literal-algorithm bits throughout.
constexpr int kFixWarps = 32;
constexpr int kFixBlocks = 1024;

// Status word of the fix-up kernel in the bounds-checked build (one per
// translation unit that includes this header; read by its status function).
__device__ unsigned int g_fixup_status = 0;

template <bool OUT_F64>
__global__ void __launch_bounds__(kFixWarps * 32)
exact_fixup_kernel(const IArgs p, const int4 *__restrict__ SA, const int4 *__restrict__ SB,
                   int64_t LpA, int64_t LpB, const unsigned int *__restrict__ work_count,
                   const unsigned int *__restrict__ work_list) {
    __shared__ unsigned short xs[kFixWarps][kChunk], ws[kFixWarps][kChunk];   // bf16 bits
    __shared__ double Pq[kFixWarps];
    wait_prior_grid();
    allow_next_grid();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int64_t count = *work_count;
    const int64_t nq = (p.R + kChunk - 1) / kChunk;
    const int64_t n_a = (p.rows > 0 && p.R > 0) ? (p.rows - 1) * p.a_si + (p.R - 1) * p.a_sr + 1 : 0;
    const int64_t n_b = (p.cols > 0 && p.R > 0) ? (p.R - 1) * p.b_sr + (p.cols - 1) * p.b_sj + 1 : 0;
    for (int64_t item = blockIdx.x; item < count; item += gridDim.x) {
        const int64_t o = work_list[item];
        const int64_t i = o / p.cols, j = o % p.cols;
        if (!in_bounds(&g_fixup_status, o, 1, p.rows * p.cols)) continue;
        double S = 0.0, C = 0.0;                        // thread 0's outer KBN state
        for (int64_t qb = 0; qb < nq; qb += kFixWarps) {
            const int64_t q = qb + warp;
            if (q < nq) {
                const int64_t q0 = q * kChunk;
                const int64_t qend = (p.R - q0 > kChunk) ? q0 + kChunk : p.R;
                const bool sok = in_bounds(&g_fixup_status, q * LpA + i, 1, nq * LpA) &&
                                 in_bounds(&g_fixup_status, q * LpB + j, 1, nq * LpB);
                const int4 sa = sok ? SA[q * LpA + i] : make_int4(0, kWidthBad, 0, 0);
                const int4 sb = sok ? SB[q * LpB + j] : make_int4(0, kWidthBad, 0, 0);
                uint32_t hx[kChunk / 32], hw[kChunk / 32];
#pragma unroll
                for (int t = 0; t < kChunk / 32; ++t) {
                    const int64_t r = q0 + lane + 32 * t;
                    hx[t] = (r < qend && in_bounds(&g_fixup_status, i * p.a_si + r * p.a_sr, 1, n_a))
                                ? ld_bits(p.A, i * p.a_si + r * p.a_sr) : 0u;
                    hw[t] = (r < qend && in_bounds(&g_fixup_status, r * p.b_sr + j * p.b_sj, 1, n_b))
                                ? ld_bits(p.B, r * p.b_sr + j * p.b_sj) : 0u;
                }
                // KBN over a chunk captures every rounding error exactly and,
                // while wx + ww < 90, also sums them exactly (each error is a
                // multiple of 2^(bx + bw) below 2^(wx + ww - 45) of it), so the
                // chunk value fl(s + c) is the exact chunk sum rounded once to
                // float64; the exact sum is an integer dot product in 128 bits
                const bool exact = sa.y <= 62 && sb.y <= 62 && sa.y + sb.y < 90;   // no inf/NaN either
                double P;
                if (exact) {
                    __int128 I = 0;
#pragma unroll
                    for (int t = 0; t < kChunk / 32; ++t) {
                        int mx, ex, mw, ew;
                        bool bx_, bw_;
                        decode(hx[t], mx, ex, bx_);
                        decode(hw[t], mw, ew, bw_);
                        if (mx == 0 || mw == 0) continue;
                        const long long X = line_int(mx, ex, sa.x);   // |X| < 2^62
                        const long long W = line_int(mw, ew, sb.x);
                        I += (__int128)X * W;                                     // |X W| < 2^90
                    }
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) {
                        const long long lo = __shfl_xor_sync(0xffffffffu, (long long)(unsigned long long)I, off);
                        const long long hi = __shfl_xor_sync(0xffffffffu, (long long)(I >> 64), off);
                        I += ((__int128)hi << 64) | (__int128)(unsigned long long)lo;
                    }
                    P = round_i128_to_double(I, sa.x + sb.x);
                } else {                                   // inf/NaN or extreme widths: literal loop
#pragma unroll
                    for (int t = 0; t < kChunk / 32; ++t) {
                        xs[warp][lane + 32 * t] = (unsigned short)hx[t];
                        ws[warp][lane + 32 * t] = (unsigned short)hw[t];
                    }
                    __syncwarp();
                    double s_ = 0.0, c_ = 0.0;
                    if (lane == 0) {
                        const int len = (int)(qend - q0);
                        for (int k = 0; k < len; ++k) {
                            const double x = widen_bf16(xs[warp][k]), w = widen_bf16(ws[warp][k]);
                            kbn_product_step(s_, c_, x, w,
                                             ((uint32_t)__double2hiint(x) & 0x7ff00000u) +
                                             ((uint32_t)__double2hiint(w) & 0x7ff00000u));
                        }
                    }
                    __syncwarp();
                    P = __dadd_rn(s_, c_);
                }
                if (lane == 0) Pq[warp] = P;
            }
            __syncthreads();
            if (threadIdx.x == 0)
                for (int w = 0; w < kFixWarps && qb + w < nq; ++w) kbn_value_step(S, C, Pq[w]);
            __syncthreads();
        }
        if (threadIdx.x == 0) {
            double y = __dadd_rn(S, C);
            if (p.bias && in_bounds(&g_fixup_status, j, 1, p.cols)) y = __dadd_rn(y, widen_bf16(ld_bits(p.bias, j)));
            if (OUT_F64) static_cast<double *>(p.out)[o] = y;
            else static_cast<unsigned short *>(p.out)[o] = exact_round_bf16(y);
        }
    }
}

}  // namespace
}  // namespace carbon
