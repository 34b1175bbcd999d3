// exact_kbn.cu - exact tier: float64 products, fixed-order Kahan-Babushka-
// Neumaier summation, one round-to-nearest-even to the output type.
//
// What is computed (Carbon README, "How It Works"; sgemm-bi "Determinism
// contracts" for the downcast): for every output, the products a_r * b_r are
// formed in float64 (exact for fp32 and bf16 operands), summed with KBN in
// 256-wide chunks of the reduction index taken left to right, each chunk
// contributing fl(s + c), the chunk values combined left to right with KBN,
// the bias added once in float64 (forward pass), and the float64 value
// rounded once to fp32 or bf16.
//
// How it is computed on GB300.  GB300 issues float64 instructions at two
// lanes per SM per clock (1/64 of its fp32 rate); everything here is shaped
// to spend that pipe only on the additions the method names:
//  * Operands are widened to float64 with integer bit operations while they
//    are staged into shared memory (a hardware fp32->fp64 conversion would
//    run on the float64 pipe).
//  * One KBN step costs four float64 instructions instead of five:
//      t = fma(x, w, s)           == fl(s + p), since p = x*w is exact
//      d = fma(a1, a2, -t)        error, first half
//      e = fma(b1, b2, d)         error, second half
//      c = c + e
//    KBN's correction (a - t) + b with a the operand of larger magnitude
//    is Fast2Sum, whose result is the exact rounding error of s + p whenever
//    the exponent of a is at least that of b.  Which operand plays a is
//    chosen from exponent fields on the integer pipe: s is taken as a when
//    E(s) > E(x) + E(w) (then E(s) >= E(p)); otherwise p is (then
//    E(p) >= E(x) + E(w) >= E(s)).  Both choices give the exact error, which
//    is the value the literal |s| >= |p| test produces, so the bits equal the
//    plain algorithm's.  The choice is applied with predicated selects
//    (a1, a2) = (s, 1) or (x, w), never with a branch, so a warp whose lanes
//    disagree issues the four float64 instructions once.
//  * Most KBN steps on bf16 data do not round at all: a bf16 x bf16 product
//    has at most 16 significant bits, so s + p is usually representable and
//    the correction term is exactly 0.  The kernel first runs each 32-deep
//    slice of the reduction issuing only t = fma(x, w, s) per step, together
//    with an integer proof that the step was exact: s is always an integer
//    multiple of 2^L, where L is the lowest set-bit exponent over the chunk's
//    products so far (true for the sums of the plain algorithm too: rounding
//    to a coarser grid keeps multiples of 2^L), and the product is a multiple
//    of 2^(L(x) + L(w)); if both are multiples of ulp(t), then s + p = t
//    exactly, the correction is 0 and c is unchanged -- the same bits the
//    full step produces.  If any lane of the warp cannot prove every step of
//    the slice, the warp restores its state at the slice start and runs the
//    slice with the full four-instruction step.  Either way the bits are the
//    plain algorithm's.
//  * Every output is owned by one thread (output-stationary), so the
//    summation order is the documented one by construction, for every M.
// Zero padding of ragged tiles is exact: adding a +0 product leaves s and c
// unchanged (s is never -0: it starts at +0 and fl(a + b) is -0 only when
// both are -0).
#include "carbon_internal.h"
#include "bounds.cuh"
#include "device_sync.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "exact_common.cuh"

namespace carbon {
namespace {

// Status word: CARBON_ERR_OUT_OF_BOUNDS in the bounds-checked build.
__device__ unsigned int g_kbn_status = 0;
#define CHK(idx, len, n) in_bounds(&g_kbn_status, (int64_t)(idx), (int64_t)(len), (int64_t)(n))

constexpr int kChunk = 256;              // documented chunk width
constexpr int kBK = 32;                  // reduction slice staged per step (divides kChunk)
constexpr int kTX = 16, kTY = 16;        // thread grid of a CTA
constexpr int kTM = 2, kTN = 2;          // outputs per thread (rows x cols)
constexpr int kBM = kTY * kTM;           // CTA output tile rows
constexpr int kBN = kTX * kTN;           // CTA output tile cols
constexpr int kThreads = kTX * kTY;
static_assert(kChunk % kBK == 0, "a staged slice must not straddle chunks");

struct KArgs {
    const void *A, *B, *bias;
    void *out;
    int64_t rows, cols, R;
    int64_t a_si, a_sr, b_sr, b_sj;
    int64_t tiles_n;
    int64_t n_a, n_b;                    // operand extents (elements), for the bounds checks
};

// Grain keys for the exactness proof, kept shifted left by 20 so they compare
// directly with a double's exponent field (hi word & 0x7ff00000).
// For a nonzero finite operand v, L(v) is the exponent of its lowest set bit.
// A-side key: (L(x) + 1075) << 20; B-side key: L(w) << 20.  Their sum G is
// the biased exponent field of 2^(L(x) + L(w) + 52): the step is exact when
// the result's exponent field is <= min(G) over the chunk so far.
// Zeros get keys that never lower the minimum; non-finite operands get keys
// that always fail the proof (the full step then handles them).
constexpr int kGrainZeroA = 0x58000000;
constexpr int kGrainZeroB = 0x20000000;
constexpr int kGrainBad = -0x40000000;

__device__ __forceinline__ int lsb_exponent(double v) {
    const unsigned long long u = (unsigned long long)__double_as_longlong(v);
    const int f = (int)((u >> 52) & 0x7ffull);
    const unsigned long long mant = u & 0x000fffffffffffffull;
    return mant ? (f - 1023 - 52 + __ffsll((long long)mant) - 1) : (f - 1023);
}

// Zero test on the bit pattern: a float64 compare would run on the FP64 pipe.
__device__ __forceinline__ bool is_zero_bits(double v) {
    return (((uint32_t)__double2hiint(v) & 0x7fffffffu) | (uint32_t)__double2loint(v)) == 0u;
}

__device__ __forceinline__ int grain_key_a(double v) {
    const uint32_t f = ((uint32_t)__double2hiint(v) >> 20) & 0x7ffu;
    if (f == 0x7ffu) return kGrainBad;
    if (is_zero_bits(v)) return kGrainZeroA;
    return (lsb_exponent(v) + 1075) << 20;
}

__device__ __forceinline__ int grain_key_b(double v) {
    const uint32_t f = ((uint32_t)__double2hiint(v) >> 20) & 0x7ffu;
    if (f == 0x7ffu) return kGrainBad;
    if (is_zero_bits(v)) return kGrainZeroB;
    return lsb_exponent(v) << 20;
}

// float64 -> IEEE binary16, round to nearest even, one rounding: 11
// significant bits, normal exponents -14..15 (largest finite 65504),
// subnormal quantum 2^-24, on the integer fields of the float64.
__device__ __forceinline__ unsigned short exact_round_f16(double y) {
    const unsigned long long u = (unsigned long long)__double_as_longlong(y);
    const unsigned int sign = (unsigned int)(u >> 48) & 0x8000u;
    const unsigned long long mag = u & 0x7fffffffffffffffull;
    if (mag > 0x7ff0000000000000ull) return (unsigned short)(sign | 0x7e00u);  // NaN
    const int E = (int)(mag >> 52) - 1023;
    if (E >= 16) return (unsigned short)(sign | 0x7c00u);                     // |y| >= 2^16
    if (E >= -14) {                                                           // normal range
        const unsigned long long lsb = (mag >> 42) & 1ull;
        const unsigned long long r = (mag + 0x000001ffffffffffull + lsb) >> 42;
        const int Ed = (int)(r >> 10);                                        // biased, after carry
        if (Ed - 1023 >= 16) return (unsigned short)(sign | 0x7c00u);
        return (unsigned short)(sign | ((unsigned int)(Ed - 1023 + 15) << 10) | (unsigned int)(r & 0x3ff));
    }
    if (E < -25) return (unsigned short)sign;                                 // below half the quantum
    // subnormal range: n = RNE(|y| / 2^-24), 0 <= n <= 1024 (1024 = min normal)
    const unsigned long long sig = (mag & 0x000fffffffffffffull) | 0x0010000000000000ull;
    const int shift = 28 - E;                                                 // 43 .. 53
    const unsigned long long n = sig >> shift;
    const unsigned long long rem = sig & ((1ull << shift) - 1ull);
    const unsigned long long half = 1ull << (shift - 1);
    const unsigned long long nr = n + ((rem > half || (rem == half && (n & 1ull))) ? 1ull : 0ull);
    return (unsigned short)(sign | (unsigned int)nr);
}

// The fp32 bit pattern of an operand element (bf16 is the top half of an
// fp32; fp16 widens to fp32 exactly with the hardware conversion).
template <int DT>
__device__ __forceinline__ uint32_t load_bits(const void *base, int64_t idx) {
    if (DT == CARBON_F32) return __ldg(static_cast<const unsigned int *>(base) + idx);
    if (DT == CARBON_F16)
        return __float_as_uint(__half2float(__ushort_as_half(__ldg(static_cast<const unsigned short *>(base) + idx))));
    return (uint32_t)__ldg(static_cast<const unsigned short *>(base) + idx) << 16;
}

template <int DT, int PASS>
__device__ __forceinline__ void stage_slice(const KArgs &p, double (*As)[kBM + 1],
                                            double (*Bs)[kBN + 1], int (*Ag)[kBM + 1],
                                            int (*Bg)[kBN + 1], int64_t i0, int64_t j0,
                                            int64_t r0, int64_t rend, int tid) {
#pragma unroll
    for (int l = 0; l < (kBK * kBM) / kThreads; ++l) {
        const int e = tid + kThreads * l;
        int ii, rr;
        if (PASS == CARBON_PASS_DW) { ii = e % kBM; rr = e / kBM; }   // i contiguous in memory
        else                        { rr = e % kBK; ii = e / kBK; }   // r contiguous in memory
        const int64_t i = i0 + ii, r = r0 + rr;
        double v = 0.0;
        if (i < p.rows && r < rend && CHK(i * p.a_si + r * p.a_sr, 1, p.n_a))
            v = widen(load_bits<DT>(p.A, i * p.a_si + r * p.a_sr));
        As[rr][ii] = v;
        Ag[rr][ii] = grain_key_a(v);
    }
#pragma unroll
    for (int l = 0; l < (kBK * kBN) / kThreads; ++l) {
        const int e = tid + kThreads * l;
        int jj, rr;
        if (PASS == CARBON_PASS_DX) { rr = e % kBK; jj = e / kBK; }   // r contiguous in memory
        else                        { jj = e % kBN; rr = e / kBN; }   // j contiguous in memory
        const int64_t j = j0 + jj, r = r0 + rr;
        double v = 0.0;
        if (j < p.cols && r < rend && CHK(r * p.b_sr + j * p.b_sj, 1, p.n_b))
            v = widen(load_bits<DT>(p.B, r * p.b_sr + j * p.b_sj));
        Bs[rr][jj] = v;
        Bg[rr][jj] = grain_key_b(v);
    }
}

// Output modes: the rounded output, the float64 value before the rounding,
// or the chunk values fl(s + c) themselves (P[chunk][rows][cols], no outer
// sum and no bias), for reductions split across ranks on chunk boundaries.
constexpr int kOutRounded = 0, kOutF64 = 1, kOutChunks = 2;

template <int DT, int PASS, int OUT>
__global__ void __launch_bounds__(kThreads)
exact_kbn_kernel(const KArgs p) {
    __shared__ double As[kBK][kBM + 1];
    __shared__ double Bs[kBK][kBN + 1];
    __shared__ int Ag[kBK][kBM + 1];
    __shared__ int Bg[kBK][kBN + 1];
    wait_prior_grid();
    allow_next_grid();
    const int tid = threadIdx.x;
    const int tx = tid % kTX, ty = tid / kTX;
    const int64_t tile = blockIdx.x;
    const int64_t i0 = (tile / p.tiles_n) * kBM;
    const int64_t j0 = (tile % p.tiles_n) * kBN;

    double S[kTM][kTN], C[kTM][kTN];
#pragma unroll
    for (int m = 0; m < kTM; ++m)
#pragma unroll
        for (int n = 0; n < kTN; ++n) { S[m][n] = 0.0; C[m][n] = 0.0; }

    for (int64_t q0 = 0; q0 < p.R; q0 += kChunk) {
        const int64_t qend = (p.R - q0 > kChunk) ? q0 + kChunk : p.R;
        double s[kTM][kTN], c[kTM][kTN];
        int g[kTM][kTN];                     // min grain key over the chunk so far
#pragma unroll
        for (int m = 0; m < kTM; ++m)
#pragma unroll
            for (int n = 0; n < kTN; ++n) { s[m][n] = 0.0; c[m][n] = 0.0; g[m][n] = 0x7fffffff; }
        bool try_fast = true;                // warp-uniform

        for (int64_t r0 = q0; r0 < qend; r0 += kBK) {
            __syncthreads();
            stage_slice<DT, PASS>(p, As, Bs, Ag, Bg, i0, j0, r0, qend, tid);
            __syncthreads();

            bool slow = !try_fast;
            if (try_fast) {
                // fast attempt: one DFMA per step plus the integer exactness proof
                double s0[kTM][kTN];
                int g0[kTM][kTN];
#pragma unroll
                for (int m = 0; m < kTM; ++m)
#pragma unroll
                    for (int n = 0; n < kTN; ++n) { s0[m][n] = s[m][n]; g0[m][n] = g[m][n]; }
                int bad = 0;
#pragma unroll 4
                for (int k = 0; k < kBK; ++k) {
                    double a[kTM], b[kTN];
                    int ga[kTM], gb[kTN];
#pragma unroll
                    for (int m = 0; m < kTM; ++m) { a[m] = As[k][ty + kTY * m]; ga[m] = Ag[k][ty + kTY * m]; }
#pragma unroll
                    for (int n = 0; n < kTN; ++n) { b[n] = Bs[k][tx + kTX * n]; gb[n] = Bg[k][tx + kTX * n]; }
#pragma unroll
                    for (int m = 0; m < kTM; ++m)
#pragma unroll
                        for (int n = 0; n < kTN; ++n) {
                            s[m][n] = __fma_rn(a[m], b[n], s[m][n]);
                            g[m][n] = min(g[m][n], ga[m] + gb[n]);
                            bad |= (__double2hiint(s[m][n]) & 0x7ff00000) > g[m][n];
                        }
                }
                if (__any_sync(0xffffffffu, bad)) {
#pragma unroll
                    for (int m = 0; m < kTM; ++m)
#pragma unroll
                        for (int n = 0; n < kTN; ++n) { s[m][n] = s0[m][n]; g[m][n] = g0[m][n]; }
                    slow = true;
                    try_fast = false;        // rest of this chunk: straight to the full step
                }
            }
            if (slow) {
#pragma unroll 4
                for (int k = 0; k < kBK; ++k) {
                    double a[kTM], b[kTN];
                    uint32_t ak[kTM], bk[kTN];
                    int ga[kTM], gb[kTN];
#pragma unroll
                    for (int m = 0; m < kTM; ++m) {
                        a[m] = As[k][ty + kTY * m];
                        ak[m] = (uint32_t)__double2hiint(a[m]) & 0x7ff00000u;
                        ga[m] = Ag[k][ty + kTY * m];
                    }
#pragma unroll
                    for (int n = 0; n < kTN; ++n) {
                        b[n] = Bs[k][tx + kTX * n];
                        bk[n] = (uint32_t)__double2hiint(b[n]) & 0x7ff00000u;
                        gb[n] = Bg[k][tx + kTX * n];
                    }
#pragma unroll
                    for (int m = 0; m < kTM; ++m)
#pragma unroll
                        for (int n = 0; n < kTN; ++n) {
                            kbn_product_step(s[m][n], c[m][n], a[m], b[n], ak[m] + bk[n]);
                            g[m][n] = min(g[m][n], ga[m] + gb[n]);
                        }
                }
            }
        }
        if constexpr (OUT == kOutChunks) {
            double *P = static_cast<double *>(p.out) + (q0 / kChunk) * p.rows * p.cols;
#pragma unroll
            for (int m = 0; m < kTM; ++m)
#pragma unroll
                for (int n = 0; n < kTN; ++n) {
                    const int64_t i = i0 + ty + kTY * m, j = j0 + tx + kTX * n;
                    if (i < p.rows && j < p.cols &&
                        CHK((q0 / kChunk) * p.rows * p.cols + i * p.cols + j, 1,
                            ((p.R + kChunk - 1) / kChunk) * p.rows * p.cols))
                        P[i * p.cols + j] = __dadd_rn(s[m][n], c[m][n]);
                }
        } else {
#pragma unroll
            for (int m = 0; m < kTM; ++m)
#pragma unroll
                for (int n = 0; n < kTN; ++n)
                    kbn_value_step(S[m][n], C[m][n], __dadd_rn(s[m][n], c[m][n]));
        }
    }
    if constexpr (OUT != kOutChunks) {
#pragma unroll
    for (int m = 0; m < kTM; ++m) {
        const int64_t i = i0 + ty + kTY * m;
        if (i >= p.rows) continue;
#pragma unroll
        for (int n = 0; n < kTN; ++n) {
            const int64_t j = j0 + tx + kTX * n;
            if (j >= p.cols) continue;
            double y = __dadd_rn(S[m][n], C[m][n]);
            if (p.bias) y = __dadd_rn(y, widen(load_bits<DT>(p.bias, j)));
            const int64_t o = i * p.cols + j;
            if (!CHK(o, 1, p.rows * p.cols)) continue;
            if (OUT == kOutF64)
                static_cast<double *>(p.out)[o] = y;
            else if (DT == CARBON_F32)
                static_cast<float *>(p.out)[o] = __double2float_rn(y);
            else if (DT == CARBON_F16)
                static_cast<unsigned short *>(p.out)[o] = exact_round_f16(y);
            else
                static_cast<unsigned short *>(p.out)[o] = exact_round_bf16(y);
        }
    }
    }
}

__global__ void round_kernel(int dtype, void *out, const double *in, int64_t n) {
    wait_prior_grid();
    allow_next_grid();
    for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < n;
         k += (int64_t)gridDim.x * blockDim.x) {
        const double y = in[k];
        if (dtype == CARBON_F32) static_cast<float *>(out)[k] = __double2float_rn(y);
        else if (dtype == CARBON_F16) static_cast<unsigned short *>(out)[k] = exact_round_f16(y);
        else static_cast<unsigned short *>(out)[k] = exact_round_bf16(y);
    }
}

// Not scheduled early: blocks of a grid launched before its predecessor ends
// take whichever slots free up first, two to an SM where one would do, and
// this kernel is bound by each SM's float64 pipe (the fp32 toy MLP's nine
// GEMMs, grids of 128-256 blocks, took 9.0 ms that way instead of 6.9).
template <int DT, int PASS, int OUT>
cudaError_t launch_one(const KArgs &a, int64_t tiles, cudaStream_t stream) {
    return launch_kernel(false, exact_kbn_kernel<DT, PASS, OUT>, dim3((unsigned)tiles), dim3(kThreads), 0,
                         stream, 1, a);
}

template <int DT, int PASS>
cudaError_t launch_pass(const KArgs &a, int64_t tiles, int out, cudaStream_t stream) {
    return out == kOutChunks ? launch_one<DT, PASS, kOutChunks>(a, tiles, stream)
         : out == kOutF64    ? launch_one<DT, PASS, kOutF64>(a, tiles, stream)
                             : launch_one<DT, PASS, kOutRounded>(a, tiles, stream);
}

template <int DT>
cudaError_t launch_dtype(int pass, const KArgs &a, int64_t tiles, int out, cudaStream_t s) {
    switch (pass) {
    case CARBON_PASS_FWD: return launch_pass<DT, CARBON_PASS_FWD>(a, tiles, out, s);
    case CARBON_PASS_DX:  return launch_pass<DT, CARBON_PASS_DX>(a, tiles, out, s);
    default:              return launch_pass<DT, CARBON_PASS_DW>(a, tiles, out, s);
    }
}

// The outer KBN over chunk values in chunk order, the bias, one rounding: the
// steps the kernel above takes after its chunks, for chunk values that were
// computed elsewhere (P[q][rows][cols], q = 0 .. nchunks - 1).
template <int DT>
__global__ void __launch_bounds__(256)
combine_kernel(void *out, const double *__restrict__ P, int64_t nchunks, int64_t rows, int64_t cols,
               const void *bias) {
    wait_prior_grid();
    allow_next_grid();
    const int64_t n = rows * cols;
    for (int64_t o = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; o < n;
         o += (int64_t)gridDim.x * blockDim.x) {
        double S = 0.0, C = 0.0;
        for (int64_t q = 0; q < nchunks; ++q)
            if (CHK(q * n + o, 1, nchunks * n)) kbn_value_step(S, C, __ldg(&P[q * n + o]));
        double y = __dadd_rn(S, C);
        if (bias) y = __dadd_rn(y, widen(load_bits<DT>(bias, o % cols)));
        if (DT == CARBON_F32) static_cast<float *>(out)[o] = __double2float_rn(y);
        else if (DT == CARBON_F16) static_cast<unsigned short *>(out)[o] = exact_round_f16(y);
        else static_cast<unsigned short *>(out)[o] = exact_round_bf16(y);
    }
}

KArgs make_kargs(const Problem &p) {
    KArgs a;
    a.A = p.A; a.B = p.B; a.bias = p.bias; a.out = p.out;
    a.rows = p.rows; a.cols = p.cols; a.R = p.R;
    switch (p.pass) {
    case CARBON_PASS_FWD: a.a_si = p.K; a.a_sr = 1; a.b_sr = p.N; a.b_sj = 1; break;
    case CARBON_PASS_DX:  a.a_si = p.N; a.a_sr = 1; a.b_sr = 1;   a.b_sj = p.N; break;
    default:              a.a_si = 1;   a.a_sr = p.K; a.b_sr = p.N; a.b_sj = 1; break;
    }
    a.tiles_n = (p.cols + kBN - 1) / kBN;
    a.n_a = (p.rows > 0 && p.R > 0) ? (p.rows - 1) * a.a_si + (p.R - 1) * a.a_sr + 1 : 0;
    a.n_b = (p.cols > 0 && p.R > 0) ? (p.R - 1) * a.b_sr + (p.cols - 1) * a.b_sj + 1 : 0;
    return a;
}

carbon_status_t launch_kbn(const Problem &p, int out, cudaStream_t stream) {
    if (p.rows == 0 || p.cols == 0) return CARBON_OK;
    KArgs a = make_kargs(p);
    const int64_t tiles_m = (p.rows + kBM - 1) / kBM;
    const int64_t tiles = tiles_m * a.tiles_n;
    if (tiles > 0x7fffffff) return CARBON_ERR_INVALID_ARG;
    const cudaError_t err = (p.dtype == CARBON_F32)   ? launch_dtype<CARBON_F32>(p.pass, a, tiles, out, stream)
                          : (p.dtype == CARBON_F16) ? launch_dtype<CARBON_F16>(p.pass, a, tiles, out, stream)
                                                    : launch_dtype<CARBON_BF16>(p.pass, a, tiles, out, stream);
    count_launch();
    return note_cuda(err);
}

}  // namespace

carbon_status_t exact_chunk_values_launch(const Problem &p, cudaStream_t stream) {
    if (p.R == 0) return CARBON_OK;                       // no chunks: nothing to write
    return launch_kbn(p, kOutChunks, stream);
}

carbon_status_t exact_combine_launch(int dtype, void *out, const double *P, int64_t nchunks,
                                     int64_t rows, int64_t cols, const void *bias,
                                     cudaStream_t stream) {
    const int64_t n = rows * cols;
    if (n == 0) return CARBON_OK;
    const int64_t blocks = (n + 255) / 256 < 8192 ? (n + 255) / 256 : 8192;
    const dim3 g((unsigned)blocks), b(256);
    cudaError_t err;
    if (dtype == CARBON_F32) err = launch_k(combine_kernel<CARBON_F32>, g, b, 0, stream, 1, out, P, nchunks, rows, cols, bias);
    else if (dtype == CARBON_F16) err = launch_k(combine_kernel<CARBON_F16>, g, b, 0, stream, 1, out, P, nchunks, rows, cols, bias);
    else err = launch_k(combine_kernel<CARBON_BF16>, g, b, 0, stream, 1, out, P, nchunks, rows, cols, bias);
    count_launch();
    return note_cuda(err);
}

carbon_status_t exact_launch(const Problem &p, bool out_f64, cudaStream_t stream) {
    return launch_kbn(p, out_f64 ? kOutF64 : kOutRounded, stream);
}

carbon_status_t exact_round_launch(int dtype, void *out, const double *in, int64_t n,
                                   cudaStream_t stream) {
    if (n == 0) return CARBON_OK;
    const int64_t blocks = (n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096;
    const cudaError_t err = launch_k(round_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, 1,
                                     dtype, out, in, n);
    count_launch();
    return note_cuda(err);
}

carbon_status_t kbn_take_device_status() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_kbn_status, sizeof v) != cudaSuccess) return CARBON_OK;
    if (v != 0) cudaMemcpyToSymbol(g_kbn_status, &zero, sizeof zero);
    return (carbon_status_t)v;
}

}  // namespace carbon
