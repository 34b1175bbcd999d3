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
#include "carbon_internal.h"
#include "exact_common.cuh"

namespace carbon {
namespace {

constexpr int kChunk = 256;
constexpr int kHalf = 128;                 // reduction rows staged at a time
constexpr int kTile = 64;                  // CTA output tile: 64 x 64
constexpr int kThreads = 256;              // 16 x 16 threads, 4 x 4 outputs each
constexpr int kPitch = kTile + 4;          // int32 row pitch of the staged tiles
constexpr int kWidthBad = 99;              // width of a row/column holding inf/NaN
constexpr int kGrainBad = -0x40000000;
constexpr int kGrainZero = 0x70000000;

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

// Chunk value by the float64 KBN step, operands read from global memory.
__device__ __noinline__ double chunk_kbn_global(const IArgs &p, int64_t i, int64_t j, int64_t q0,
                                                int64_t qend) {
    double s = 0.0, c = 0.0;
    for (int64_t r = q0; r < qend; ++r) {
        const double x = widen_bf16(ld_bits(p.A, i * p.a_si + r * p.a_sr));
        const double w = widen_bf16(ld_bits(p.B, r * p.b_sr + j * p.b_sj));
        kbn_product_step(s, c, x, w,
                         ((uint32_t)__double2hiint(x) & 0x7ff00000u) +
                         ((uint32_t)__double2hiint(w) & 0x7ff00000u));
    }
    return __dadd_rn(s, c);
}

// Precise exactness check of one (row, column, chunk) on the integer pipes:
// with X, W the integer operands at bases bx, bw, every partial sum is
// representable if sum |X W| < 2^(53 + t), t the smallest number of trailing
// zero bits of a nonzero product X*W.  Needs wx, ww <= 31 and wx + ww <= 54
// (so sum |X W| < 2^62 cannot overflow).
__device__ __noinline__ bool chunk_exact_precise(const IArgs &p, int64_t i, int64_t j, int64_t q0,
                                                 int64_t qend, int bx, int bw) {
    unsigned long long abs_sum = 0;
    int tz = 1 << 20;
    for (int64_t r = q0; r < qend; ++r) {
        int mx, ex, mw, ew;
        bool bad_x, bad_w;
        decode(ld_bits(p.A, i * p.a_si + r * p.a_sr), mx, ex, bad_x);
        decode(ld_bits(p.B, r * p.b_sr + j * p.b_sj), mw, ew, bad_w);
        if (mx == 0 || mw == 0) continue;
        const long long X = (long long)mx * (1ll << (ex - bx));      // |X| < 2^31
        const long long W = (long long)mw * (1ll << (ew - bw));
        const long long prod = X * W;
        abs_sum += (unsigned long long)(prod < 0 ? -prod : prod);
        tz = min(tz, __ffsll(prod) - 1);
    }
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

// Integer operands of one staged half: T[r - r0][l] = m * 2^(e - base(l)),
// or 0 for lines too wide for int32 (those outputs never use the integer sum).
template <bool LINE_CONTIG>
__device__ __forceinline__ void stage_ints(const unsigned short *base, int64_t line_stride,
                                           int64_t r_stride, int64_t line0, int64_t nlines,
                                           int64_t r0, int64_t rend, const int *lbase,
                                           const int *lwidth, int (*T)[kPitch], int tid) {
#pragma unroll 4
    for (int l8 = 0; l8 < (kHalf * kTile) / kThreads; ++l8) {
        const int e = tid + kThreads * l8;
        int l, rr;
        if (LINE_CONTIG) { l = e % kTile; rr = e / kTile; }
        else             { rr = e % kHalf; l = e / kHalf; }
        const int64_t line = line0 + l, r = r0 + rr;
        int v = 0;
        if (line < nlines && r < rend && lwidth[l] <= 31) {
            int m, ex;
            bool b;
            decode(ld_bits(base, line * line_stride + r * r_stride), m, ex, b);
            if (m != 0) v = m * (1 << (ex - lbase[l]));          // shift <= 23: |v| < 2^31
        }
        T[rr][l] = v;
    }
}

template <int PASS, bool OUT_F64>
__global__ void __launch_bounds__(kThreads, 2)
exact_int_kernel(const IArgs p) {
    __shared__ __align__(16) int Xs[kHalf][kPitch];
    __shared__ __align__(16) int Ws[kHalf][kPitch];
    __shared__ LineStats rs, cs;
    __shared__ int rbase[kTile], rwidth[kTile], cbase[kTile], cwidth[kTile];

    const int tid = threadIdx.x;
    const int tx = tid % 16, ty = tid / 16;
    const int64_t i0 = (blockIdx.x / p.tiles_n) * kTile;
    const int64_t j0 = (blockIdx.x % p.tiles_n) * kTile;
    // A lines (rows i) are contiguous in memory for dW; B lines (cols j) for fwd and dW
    constexpr bool A_CONTIG = (PASS == CARBON_PASS_DW);
    constexpr bool B_CONTIG = (PASS != CARBON_PASS_DX);

    double S[4][4], C[4][4];
    int G[4][4];                               // outer grain: min over chunks of (base + 1075) << 20
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int n = 0; n < 4; ++n) { S[m][n] = 0.0; C[m][n] = 0.0; G[m][n] = 0x7fffffff; }

    for (int64_t q0 = 0; q0 < p.R; q0 += kChunk) {
        const int64_t qend = (p.R - q0 > kChunk) ? q0 + kChunk : p.R;

        // ---- per-line statistics of this chunk
        __syncthreads();
        if (tid < kTile) {
            rs.emin[tid] = 1 << 20; rs.emax[tid] = -(1 << 20); rs.bad[tid] = 0;
            cs.emin[tid] = 1 << 20; cs.emax[tid] = -(1 << 20); cs.bad[tid] = 0;
        }
        __syncthreads();
        gather_stats<A_CONTIG>(p.A, p.a_si, p.a_sr, i0, p.rows, q0, qend, rs, tid);
        gather_stats<B_CONTIG>(p.B, p.b_sj, p.b_sr, j0, p.cols, q0, qend, cs, tid);
        __syncthreads();
        if (tid < kTile) {
            const int lo = rs.emin[tid], hi = rs.emax[tid];
            rbase[tid] = (lo > hi) ? 0 : lo;                          // all-zero line: base 0
            rwidth[tid] = rs.bad[tid] ? kWidthBad : ((lo > hi) ? 0 : hi + 8 - lo);
        } else if (tid < 2 * kTile) {
            const int l = tid - kTile;
            const int lo = cs.emin[l], hi = cs.emax[l];
            cbase[l] = (lo > hi) ? 0 : lo;
            cwidth[l] = cs.bad[l] ? kWidthBad : ((lo > hi) ? 0 : hi + 8 - lo);
        }

        // ---- integer dot products over the chunk, two staged halves
        unsigned long long acc[4][4];
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int n = 0; n < 4; ++n) acc[m][n] = 0ull;
        for (int64_t r0 = q0; r0 < qend; r0 += kHalf) {
            const int64_t rend = (qend - r0 > kHalf) ? r0 + kHalf : qend;
            __syncthreads();
            stage_ints<A_CONTIG>(p.A, p.a_si, p.a_sr, i0, p.rows, r0, rend, rbase, rwidth, Xs, tid);
            stage_ints<B_CONTIG>(p.B, p.b_sj, p.b_sr, j0, p.cols, r0, rend, cbase, cwidth, Ws, tid);
            __syncthreads();
            const int kn = (int)(rend - r0);
#pragma unroll 4
            for (int k = 0; k < kn; ++k) {
                const int4 a4 = *reinterpret_cast<const int4 *>(&Xs[k][4 * ty]);
                const int4 b4 = *reinterpret_cast<const int4 *>(&Ws[k][4 * tx]);
                const int a[4] = {a4.x, a4.y, a4.z, a4.w};
                const int b[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                for (int m = 0; m < 4; ++m)
#pragma unroll
                    for (int n = 0; n < 4; ++n)
                        acc[m][n] += (unsigned long long)((long long)a[m] * (long long)b[n]);
            }
        }

        // ---- chunk values and the outer KBN step, one output at a time
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                const int li = 4 * ty + m, lj = 4 * tx + n;
                const int wx = rwidth[li], ww = cwidth[lj];
                const int b = rbase[li] + cbase[lj];
                const int64_t i = i0 + li, j = j0 + lj;
                double P;
                if (wx <= 31 && ww <= 31 && wx + ww <= 45) {
                    P = scaled_int_to_double((long long)acc[m][n], b);
                } else if (i < p.rows && j < p.cols) {
                    if (wx <= 31 && ww <= 31 && wx + ww <= 54 &&
                        chunk_exact_precise(p, i, j, q0, qend, rbase[li], cbase[lj]))
                        P = scaled_int_to_double((long long)acc[m][n], b);
                    else
                        P = chunk_kbn_global(p, i, j, q0, qend);
                } else {
                    P = 0.0;                                           // padding output
                }
                // P is a multiple of 2^b; S of 2^(min b so far).  If both are
                // multiples of ulp(S + P), the addition is exact and C is unchanged.
                const int g = (wx == kWidthBad || ww == kWidthBad) ? kGrainBad
                              : (wx == 0 || ww == 0) ? kGrainZero : (b + 1075) << 20;
                G[m][n] = min(G[m][n], g);
                const double t = __dadd_rn(S[m][n], P);
                const bool inexact = (__double2hiint(t) & 0x7ff00000) > G[m][n];
                if (!__any_sync(0xffffffffu, inexact)) S[m][n] = t;
                else kbn_value_step(S[m][n], C[m][n], P);
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
            double y = __dadd_rn(S[m][n], C[m][n]);
            if (p.bias) y = __dadd_rn(y, widen_bf16(ld_bits(p.bias, j)));
            const int64_t o = i * p.cols + j;
            if (OUT_F64) static_cast<double *>(p.out)[o] = y;
            else static_cast<unsigned short *>(p.out)[o] = exact_round_bf16(y);
        }
    }
}

template <int PASS>
cudaError_t launch_int_pass(const IArgs &a, int64_t tiles, bool out_f64, cudaStream_t s) {
    if (out_f64) exact_int_kernel<PASS, true><<<(unsigned)tiles, kThreads, 0, s>>>(a);
    else exact_int_kernel<PASS, false><<<(unsigned)tiles, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

carbon_status_t exact_int_launch(const Problem &p, bool out_f64, cudaStream_t stream) {
    if (p.rows == 0 || p.cols == 0) return CARBON_OK;
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
    const int64_t tiles = ((p.rows + kTile - 1) / kTile) * a.tiles_n;
    if (tiles > 0x7fffffff) return CARBON_ERR_INVALID_ARG;
    cudaError_t err;
    switch (p.pass) {
    case CARBON_PASS_FWD: err = launch_int_pass<CARBON_PASS_FWD>(a, tiles, out_f64, stream); break;
    case CARBON_PASS_DX:  err = launch_int_pass<CARBON_PASS_DX>(a, tiles, out_f64, stream); break;
    default:              err = launch_int_pass<CARBON_PASS_DW>(a, tiles, out_f64, stream); break;
    }
    count_launch();
    return note_cuda(err);
}

}  // namespace carbon
