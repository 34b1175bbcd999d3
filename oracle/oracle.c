/*
 * oracle.c - plain CPU oracle for the deterministic, batch-invariant
 * linear-layer GEMM (forward Y = X.W + b, dX = dY.W^T, dW = X^T.dY).
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library.  It shares no code, header, table
 * or helper with the CUDA library: it decodes its own inputs, runs its own
 * summation and rounds its own outputs.
 *
 * What it computes (Carbon README, "How It Works"): every product is taken
 * in float64, and products are accumulated with Kahan-Babushka-Neumaier
 * (KBN) compensation in a fixed order.  The fixed order is the one stated
 * for this library: the reduction index r runs in 256-wide chunks
 * [0,256), [256,512), ... summed left to right with KBN, each chunk yields
 * the single double fl(s + c), and the chunk values are combined left to
 * right with KBN again.  The forward pass then adds the bias in float64
 * (one rounded addition) and every pass rounds the float64 value once,
 * to nearest-even, to the output type (fp32, bf16 or fp16).  sgemm-bi's
 * "Determinism contracts" table describes the same final step as an RNE
 * downcast.
 *
 * A second mode computes the correctly rounded result that the README's
 * "Roadmap" superaccumulators stand for: the exact sum of the products and
 * the bias, rounded once to the output type, independent of any order.
 *
 * Layouts (weights stored [in, out], sgemm-bi "Use"): row-major X[M,K],
 * W[K,N], b[N], Y[M,N], dY[M,N], dX[M,K], dW[K,N].
 *   fwd : Y[i,j]  = sum_r X[i,r]  * W[r,j]   (R = K)
 *   dX  : dX[i,j] = sum_r dY[i,r] * W[j,r]   (R = N)
 *   dW  : dW[i,j] = sum_r X[r,i]  * dY[r,j]  (R = M)
 *
 * Build: -O2 -ffp-contract=off -fno-fast-math.  With contraction off every
 * `a * b` and `a + b` below is one IEEE-754 binary64 operation rounded to
 * nearest-even; products of two fp32 (or two bf16, or two fp16) values are exact in
 * binary64, so the only roundings are the additions the algorithm names.
 */
#include <float.h>
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the oracle needs FLT_EVAL_METHOD == 0 (no excess precision)"
#endif

#define ORACLE_CHUNK 256

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F16 = 2 };
enum { ORACLE_FWD = 0, ORACLE_DX = 1, ORACLE_DW = 2 };

/* ---- input decoding (exact widening to binary64) ------------------------ */

/* IEEE binary16 from its fields: 5 exponent bits (bias 15), 10 fraction
 * bits; exponent field 0 holds zeros and subnormals (quantum 2^-24), 31
 * infinities and NaNs. */
static double decode_f16(uint16_t h)
{
    int sign = (h >> 15) & 1, ex = (h >> 10) & 31, fr = h & 1023;
    double v;
    if (ex == 31)
        v = fr ? NAN : INFINITY;
    else if (ex == 0)
        v = ldexp((double)fr, -24);
    else
        v = ldexp((double)(1024 + fr), ex - 25);
    return sign ? -v : v;
}

static double decode(const void *base, int dtype, int64_t idx)
{
    float f;
    if (dtype == ORACLE_F16) {
        uint16_t h;
        memcpy(&h, (const char *)base + 2 * idx, 2);
        return decode_f16(h);          /* exact: binary16 is a subset of binary64 */
    }
    if (dtype == ORACLE_F32) {
        memcpy(&f, (const char *)base + 4 * idx, 4);
    } else {
        uint16_t h;
        uint32_t u;
        memcpy(&h, (const char *)base + 2 * idx, 2);
        u = (uint32_t)h << 16;          /* bf16 is the top half of an fp32 */
        memcpy(&f, &u, 4);
    }
    return (double)f;                   /* exact: binary32 is a subset of binary64 */
}

/* ---- output rounding ----------------------------------------------------- */

/* binary64 -> binary32, nearest-even: C's conversion in the default mode. */
static uint32_t round_to_f32_bits(double y)
{
    float f = (float)y;
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
}

/* binary64 -> bf16, nearest-even, in ONE rounding (never through fp32).
 * bf16 has 8 significant bits and the exponent range of fp32: normal
 * exponents -126..127, subnormal quantum 2^-133, largest finite
 * (2 - 2^-7) * 2^127.  The value is divided by its quantum (a power of two,
 * so exactly), rounded to an integer with ties to even, and scaled back. */
static uint16_t round_to_bf16_bits(double y)
{
    double a, quantum, n, r;
    int e, E;
    uint16_t sign = signbit(y) ? 0x8000u : 0u;
    float f;
    uint32_t u;

    if (isnan(y))
        return 0x7FC0u | sign;
    a = fabs(y);
    if (a >= 0x1p128)                   /* already beyond every finite bf16 */
        return 0x7F80u | sign;
    if (a == 0.0)
        return sign;
    (void)frexp(a, &e);                 /* a = m * 2^e, m in [0.5, 1) */
    E = e - 1;                          /* floor(log2(a)) */
    if (E < -126)
        E = -126;                       /* subnormal range: fixed quantum */
    quantum = ldexp(1.0, E - 7);
    n = nearbyint(a / quantum);         /* default mode: ties to even */
    r = n * quantum;
    if (r >= 0x1p128)                   /* rounded past the largest finite value */
        return 0x7F80u | sign;
    f = (float)r;                       /* exact: r has <= 8 significant bits */
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16) | sign;
}

/* binary64 -> binary16, nearest-even, in one rounding.  binary16 has 11
 * significant bits, normal exponents -14..15, subnormal quantum 2^-24 and
 * largest finite (2 - 2^-10) * 2^15 = 65504; the same quantum method as
 * for bf16, then the fields of the (exact) rounded value. */
static uint16_t round_to_f16_bits(double y)
{
    double a, quantum, n, r;
    int e, E;
    uint16_t sign = signbit(y) ? 0x8000u : 0u;

    if (isnan(y))
        return 0x7E00u | sign;
    a = fabs(y);
    if (a >= 0x1p16)                    /* beyond every finite binary16 */
        return 0x7C00u | sign;
    if (a == 0.0)
        return sign;
    (void)frexp(a, &e);
    E = e - 1;                          /* floor(log2(a)) */
    if (E < -14)
        E = -14;                        /* subnormal range: fixed quantum 2^-24 */
    quantum = ldexp(1.0, E - 10);
    n = nearbyint(a / quantum);         /* default mode: ties to even */
    r = n * quantum;
    if (r >= 65520.0)                   /* rounded past 65504 */
        return 0x7C00u | sign;
    if (r < 0x1p-14)                    /* subnormal (or zero): r = k * 2^-24 */
        return (uint16_t)(sign | (uint16_t)(r * 0x1p24));
    (void)frexp(r, &e);
    E = e - 1;
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(ldexp(r, 10 - E) - 1024.0));
}

/* ---- the summation ------------------------------------------------------- */

/* One step of Neumaier's improved Kahan-Babuska summation, as on the page
 * the Carbon README links: add x to (sum, comp). */
static void kbn_step(double *sum, double *comp, double x)
{
    double t = *sum + x;
    if (fabs(*sum) >= fabs(x))
        *comp += (*sum - t) + x;
    else
        *comp += (x - t) + *sum;
    *sum = t;
}

/* Fixed-order dot product of a[a0 + r*as] and b[b0 + r*bs], r = 0..R-1.
 * Returns the float64 value before the bias and the output rounding. */
static double fixed_order_dot(const void *A, int64_t a0, int64_t as,
                              const void *B, int64_t b0, int64_t bs,
                              int64_t R, int dtype)
{
    double S = 0.0, C = 0.0;            /* outer KBN over chunk values */
    int64_t q0;
    for (q0 = 0; q0 < R; q0 += ORACLE_CHUNK) {
        int64_t q1 = (R - q0 > ORACLE_CHUNK) ? q0 + ORACLE_CHUNK : R;
        double s = 0.0, c = 0.0;        /* KBN inside the chunk */
        int64_t r;
        for (r = q0; r < q1; ++r) {
            double p = decode(A, dtype, a0 + r * as) * decode(B, dtype, b0 + r * bs);
            kbn_step(&s, &c, p);
        }
        kbn_step(&S, &C, s + c);        /* chunk value fl(s + c) */
    }
    return S + C;
}

/* ---- the correctly rounded tier: a superaccumulator ---------------------- */

/* The Carbon README's "Roadmap" names superaccumulators, exact summation that
 * needs no fixed order.  The value such a sum stands for has a plain
 * definition: the exact sum of the products (each exact in float64) plus the
 * bias, rounded once, to nearest-even, to the output type.  Written out here
 * with a fixed-point accumulator wide enough for any product of two inputs:
 * 32-bit digits, each held in an int64 so that carries can wait, bit 0 of
 * the accumulator weighing 2^-SA_OFFSET.  Every product of two fp32 values
 * lies in [2^-298, 2^256) in magnitude, so as m * 2^e with |m| < 2^53 its
 * lowest bit is at e >= -350 and its highest below 2^256. */
#define SA_DIGITS 24                    /* 768 bits */
#define SA_OFFSET 360

typedef struct {
    int64_t d[SA_DIGITS];
    int nan, pinf, ninf;                /* non-finite terms seen */
    int64_t adds;                       /* additions since the last carry pass */
} superacc_t;

static void sa_carry(superacc_t *a)
{
    int k;
    for (k = 0; k + 1 < SA_DIGITS; ++k) {
        int64_t c = a->d[k] >> 32;      /* arithmetic shift: floor division by 2^32 */
        a->d[k] -= c * ((int64_t)1 << 32);
        a->d[k + 1] += c;
    }
    a->adds = 0;
}

/* Adds the float64 value x exactly. */
static void sa_add(superacc_t *a, double x)
{
    int e, k, s, neg;
    double f;
    uint64_t u;
    unsigned __int128 v;
    if (isnan(x)) { a->nan = 1; return; }
    if (isinf(x)) { if (x > 0) a->pinf = 1; else a->ninf = 1; return; }
    if (x == 0.0)
        return;
    f = frexp(x, &e);                   /* x = f * 2^e, 0.5 <= |f| < 1 */
    neg = f < 0;
    u = (uint64_t)ldexp(fabs(f), 53);   /* exact: an integer below 2^53 */
    e = e - 53 + SA_OFFSET;             /* x = +-u * 2^(e - SA_OFFSET), e >= 10 */
    k = e / 32;
    s = e % 32;
    v = (unsigned __int128)u << s;      /* below 2^85: three digits */
    if (neg) {
        a->d[k] -= (int64_t)(uint32_t)v;
        a->d[k + 1] -= (int64_t)(uint32_t)(v >> 32);
        a->d[k + 2] -= (int64_t)(v >> 64);
    } else {
        a->d[k] += (int64_t)(uint32_t)v;
        a->d[k + 1] += (int64_t)(uint32_t)(v >> 32);
        a->d[k + 2] += (int64_t)(v >> 64);
    }
    if (++a->adds == ((int64_t)1 << 28))
        sa_carry(a);
}

static int sa_bit(const superacc_t *a, int i)
{
    return i < 0 ? 0 : (int)((a->d[i / 32] >> (i % 32)) & 1);
}

/* Rounds the accumulated value once to the output type; returns its bits
 * (fp32 bits, or the 16-bit pattern of bf16 / fp16).  A NaN term, or both
 * infinities, gives NaN; otherwise an infinite term gives that infinity; an
 * exact sum of zero gives +0. */
static uint32_t sa_round(superacc_t *a, int dtype)
{
    int p, qmin, top, k, q, neg = 0;
    uint64_t n = 0;
    int half, sticky = 0;
    double v;
    if (a->nan || (a->pinf && a->ninf))
        v = NAN;
    else if (a->pinf || a->ninf)
        v = a->pinf ? INFINITY : -INFINITY;
    else {
        sa_carry(a);                    /* digits 0..SA_DIGITS-2 now in [0, 2^32) */
        if (a->d[SA_DIGITS - 1] < 0) {  /* negative: take the magnitude */
            neg = 1;
            for (k = 0; k < SA_DIGITS; ++k)
                a->d[k] = -a->d[k];
            sa_carry(a);
        }
        /* precision and the bit index of the smallest quantum (subnormals) */
        p = dtype == ORACLE_F32 ? 24 : (dtype == ORACLE_F16 ? 11 : 8);
        qmin = (dtype == ORACLE_F32 ? -149 : (dtype == ORACLE_F16 ? -24 : -133)) + SA_OFFSET;
        for (top = 32 * SA_DIGITS - 1; top >= 0 && !sa_bit(a, top); --top)
            ;
        if (top < 0)
            return 0u;                  /* exact zero: +0 */
        q = top - (p - 1) > qmin ? top - (p - 1) : qmin;   /* quantum bit */
        for (k = top; k >= q; --k)
            n = 2 * n + (uint64_t)sa_bit(a, k);
        half = sa_bit(a, q - 1);
        for (k = q - 2; k >= 0 && !sticky; --k)
            sticky = sa_bit(a, k);
        if (half && (sticky || (n & 1)))
            ++n;                        /* nearest, ties to even */
        v = ldexp((double)n, q - SA_OFFSET);   /* exact; may reach the overflow bound */
        if (neg)
            v = -v;
    }
    /* v is NaN, infinite, or exact in the output type except when it is the
     * power of two just past the largest finite value, which the routines
     * below send to infinity: no second rounding happens */
    if (dtype == ORACLE_F32)
        return round_to_f32_bits(v);
    return dtype == ORACLE_F16 ? round_to_f16_bits(v) : round_to_bf16_bits(v);
}

/* Correctly rounded a[a0 + r*as] . b[b0 + r*bs] (+ bias), r = 0..R-1. */
static uint32_t exact_dot_rounded(const void *A, int64_t a0, int64_t as,
                                  const void *B, int64_t b0, int64_t bs,
                                  int64_t R, int dtype, const void *bias, int64_t j)
{
    superacc_t acc;
    int64_t r;
    memset(&acc, 0, sizeof acc);
    for (r = 0; r < R; ++r)
        sa_add(&acc, decode(A, dtype, a0 + r * as) * decode(B, dtype, b0 + r * bs));
    if (bias)
        sa_add(&acc, decode(bias, dtype, j));
    return sa_round(&acc, dtype);
}

/* ---- one output element --------------------------------------------------- */

typedef struct {
    int pass, dtype;
    int superacc;       /* correctly rounded tier instead of fixed-order KBN */
    const void *A, *B, *bias;
    int64_t M, K, N;
    void *out;          /* output-typed array, or NULL */
    double *y64;        /* float64 value before output rounding, or NULL */
    /* either a dense range [first, last) of row-major output positions ... */
    int64_t first, last;
    /* ... or explicit coordinates (when rows != NULL) */
    const int64_t *rows, *cols;
    int64_t ncols_out;  /* row length of the output matrix */
} job_t;

static void one_output_rounded(const job_t *jb, int64_t i, int64_t j, int64_t slot)
{
    uint32_t u;
    switch (jb->pass) {
    case ORACLE_FWD:
        u = exact_dot_rounded(jb->A, i * jb->K, 1, jb->B, j, jb->N, jb->K, jb->dtype, jb->bias, j);
        break;
    case ORACLE_DX:
        u = exact_dot_rounded(jb->A, i * jb->N, 1, jb->B, j * jb->N, 1, jb->N, jb->dtype, NULL, 0);
        break;
    default:
        u = exact_dot_rounded(jb->A, i, jb->K, jb->B, j, jb->N, jb->M, jb->dtype, NULL, 0);
        break;
    }
    if (jb->dtype == ORACLE_F32) {
        memcpy((char *)jb->out + 4 * slot, &u, 4);
    } else {
        uint16_t h = (uint16_t)u;
        memcpy((char *)jb->out + 2 * slot, &h, 2);
    }
}

static void one_output(const job_t *jb, int64_t i, int64_t j, int64_t slot)
{
    double y;
    if (jb->superacc) {
        one_output_rounded(jb, i, j, slot);
        return;
    }
    switch (jb->pass) {
    case ORACLE_FWD:    /* X[i, r] * W[r, j] */
        y = fixed_order_dot(jb->A, i * jb->K, 1, jb->B, j, jb->N, jb->K, jb->dtype);
        if (jb->bias)
            y = y + decode(jb->bias, jb->dtype, j);
        break;
    case ORACLE_DX:     /* dY[i, r] * W[j, r] */
        y = fixed_order_dot(jb->A, i * jb->N, 1, jb->B, j * jb->N, 1, jb->N, jb->dtype);
        break;
    default:            /* X[r, i] * dY[r, j] */
        y = fixed_order_dot(jb->A, i, jb->K, jb->B, j, jb->N, jb->M, jb->dtype);
        break;
    }
    if (jb->y64)
        jb->y64[slot] = y;
    if (jb->out) {
        if (jb->dtype == ORACLE_F32) {
            uint32_t u = round_to_f32_bits(y);
            memcpy((char *)jb->out + 4 * slot, &u, 4);
        } else {
            uint16_t h = jb->dtype == ORACLE_F16 ? round_to_f16_bits(y) : round_to_bf16_bits(y);
            memcpy((char *)jb->out + 2 * slot, &h, 2);
        }
    }
}

static void *run_job(void *arg)
{
    const job_t *jb = (const job_t *)arg;
    int64_t k;
    for (k = jb->first; k < jb->last; ++k) {
        if (jb->rows)
            one_output(jb, jb->rows[k], jb->cols[k], k);
        else
            one_output(jb, k / jb->ncols_out, k % jb->ncols_out, k);
    }
    return NULL;
}

static int launch(job_t proto, int64_t count, int nthreads)
{
    pthread_t *tid;
    job_t *jobs;
    int t, started = 0;
    if (nthreads < 1)
        nthreads = 1;
    if (count < (int64_t)nthreads)
        nthreads = count > 0 ? (int)count : 1;
    tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    if (!tid || !jobs) {
        free(tid);
        free(jobs);
        return -2;
    }
    for (t = 0; t < nthreads; ++t) {
        jobs[t] = proto;
        jobs[t].first = count * t / nthreads;
        jobs[t].last = count * (t + 1) / nthreads;
    }
    if (nthreads == 1) {
        run_job(&jobs[0]);
    } else {
        for (t = 0; t < nthreads; ++t) {
            if (pthread_create(&tid[t], NULL, run_job, &jobs[t]) != 0)
                break;
            ++started;
        }
        for (t = started; t < nthreads; ++t)   /* could not start: run here */
            run_job(&jobs[t]);
        for (t = 0; t < started; ++t)
            pthread_join(tid[t], NULL);
    }
    free(tid);
    free(jobs);
    return 0;
}

static int check(int pass, int dtype, int64_t M, int64_t K, int64_t N)
{
    if (pass < ORACLE_FWD || pass > ORACLE_DW)
        return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F16)
        return -1;
    if (M < 0 || K < 0 || N < 0)
        return -1;
    /* the superaccumulator's digits take 2^28 additions between carry passes;
     * reduction lengths stay far below 2^31 */
    if (M >= ((int64_t)1 << 31) || K >= ((int64_t)1 << 31) || N >= ((int64_t)1 << 31))
        return -1;
    return 0;
}

/* ---- exported API ------------------------------------------------------- */

/* Dense pass.  A/B are (X, W) for fwd, (dY, W) for dX, (X, dY) for dW;
 * bias is used by fwd only (may be NULL).  out (output dtype) and y64
 * (float64) may each be NULL.  Output shape: fwd [M,N], dX [M,K], dW [K,N]. */
int oracle_gemm(int pass, int dtype, const void *A, const void *B, const void *bias,
                int64_t M, int64_t K, int64_t N, void *out, double *y64, int nthreads)
{
    job_t jb;
    int64_t rows, cols;
    if (check(pass, dtype, M, K, N))
        return -1;
    memset(&jb, 0, sizeof jb);
    jb.pass = pass; jb.dtype = dtype; jb.A = A; jb.B = B;
    jb.bias = (pass == ORACLE_FWD) ? bias : NULL;
    jb.M = M; jb.K = K; jb.N = N; jb.out = out; jb.y64 = y64;
    rows = (pass == ORACLE_DW) ? K : M;
    cols = (pass == ORACLE_DX) ? K : N;
    jb.ncols_out = cols;
    return launch(jb, rows * cols, nthreads);
}

/* Selected outputs only: out[k], y64[k] for output (rows[k], cols[k]). */
int oracle_gemm_at(int pass, int dtype, const void *A, const void *B, const void *bias,
                   int64_t M, int64_t K, int64_t N, const int64_t *rows, const int64_t *cols,
                   int64_t count, void *out, double *y64, int nthreads)
{
    job_t jb;
    if (check(pass, dtype, M, K, N) || count < 0 || (count > 0 && (!rows || !cols)))
        return -1;
    memset(&jb, 0, sizeof jb);
    jb.pass = pass; jb.dtype = dtype; jb.A = A; jb.B = B;
    jb.bias = (pass == ORACLE_FWD) ? bias : NULL;
    jb.M = M; jb.K = K; jb.N = N; jb.out = out; jb.y64 = y64;
    jb.rows = rows; jb.cols = cols;
    return launch(jb, count, nthreads);
}

/* The output rounding on its own, for checking it against exact rounding. */
void oracle_round(int dtype, const double *y, void *out, int64_t n)
{
    int64_t k;
    for (k = 0; k < n; ++k) {
        if (dtype == ORACLE_F32) {
            uint32_t u = round_to_f32_bits(y[k]);
            memcpy((char *)out + 4 * k, &u, 4);
        } else {
            uint16_t h = dtype == ORACLE_F16 ? round_to_f16_bits(y[k]) : round_to_bf16_bits(y[k]);
            memcpy((char *)out + 2 * k, &h, 2);
        }
    }
}

int oracle_chunk_width(void) { return ORACLE_CHUNK; }

/* Correctly rounded tier: out = RNE(exact dot product + bias), dense (out
 * non-NULL) or at the listed outputs (rows != NULL, count of them). */
int oracle_gemm_superacc(int pass, int dtype, const void *A, const void *B, const void *bias,
                         int64_t M, int64_t K, int64_t N, const int64_t *rows,
                         const int64_t *cols, int64_t count, void *out, int nthreads)
{
    job_t jb;
    if (check(pass, dtype, M, K, N) || !out || count < 0 || (rows && !cols))
        return -1;
    memset(&jb, 0, sizeof jb);
    jb.pass = pass; jb.dtype = dtype; jb.A = A; jb.B = B; jb.superacc = 1;
    jb.bias = (pass == ORACLE_FWD) ? bias : NULL;
    jb.M = M; jb.K = K; jb.N = N; jb.out = out;
    if (rows) {
        jb.rows = rows; jb.cols = cols;
        return launch(jb, count, nthreads);
    }
    jb.ncols_out = (pass == ORACLE_DX) ? K : N;
    return launch(jb, ((pass == ORACLE_DW) ? K : M) * jb.ncols_out, nthreads);
}
