/*
 * carbon_gemm.h - deterministic, batch-invariant linear-layer GEMM for
 * NVIDIA GB300 (sm_103a).  Public C ABI.
 *
 * The three passes of a linear layer whose weight is stored [in, out]
 * ("GEMM-natural", sgemm-bi page, "Use"):
 *
 *   carbon_gemm_fwd : Y  = X . W + b     X[M,K]  W[K,N]  b[N]  -> Y[M,N]
 *   carbon_gemm_dx  : dX = dY . W^T      dY[M,N] W[K,N]        -> dX[M,K]
 *   carbon_gemm_dw  : dW = X^T . dY      X[M,K]  dY[M,N]       -> dW[K,N]
 *
 * All matrices are dense, row-major and contiguous (row pitch = number of
 * columns).  M is the number of tokens (rows of X, dY); K = in-features,
 * N = out-features.  Every operand and the output have the same dtype.
 *
 * Three tiers (tier argument):
 *
 * CARBON_TIER_EXACT - every product is formed in float64 (exactly: products
 *   of two fp32, two bf16 or two fp16 values fit in binary64), and products
 *   are summed with Kahan-Babushka-Neumaier compensation in a fixed order (Carbon
 *   README, "How It Works": tiles, upcast to float64, KBN compensation in a
 *   fixed order).  The order depends only on the reduction length R (K for
 *   fwd, N for dX, M for dW): R is cut into 256-wide chunks from index 0; each
 *   chunk is summed left to right with KBN and contributes the single double
 *   fl(s + c); the chunk values are combined left to right with KBN again.
 *   The forward pass adds the bias once in float64.  The float64 value is
 *   rounded once, to nearest-even, to fp32, bf16 or fp16 (the RNE downcast of
 *   sgemm-bi's "Determinism contracts").  The result is a pure function of
 *   the inputs' bits: identical on every run, for every M, on every device,
 *   and identical to a plain CPU implementation of the same steps.
 *   Accepts CARBON_F32, CARBON_BF16 and CARBON_F16, any shape, any element
 *   alignment.
 *
 * CARBON_TIER_TC - bf16 x bf16 (or fp16 x fp16) products accumulated in
 *   fp32 on the tensor cores (tcgen05, accumulators in tensor memory), with a
 *   K schedule that depends only on the shape of the reduction and the output
 *   columns, never on the batch size of fwd/dX (sgemm-bi, "Determinism
 *   contracts", tensor core tier: fixed tile families, shape-only dispatch).
 *   fwd adds the bias in fp32; the fp32 value is rounded once, to
 *   nearest-even, to the input type.  Bit-identical run to run; fwd and dX
 *   rows are bit-identical for every M.  Accepts CARBON_BF16 and CARBON_F16
 *   (CARBON_F32 -> CARBON_ERR_UNSUPPORTED).  Base pointers must be 16-byte
 *   aligned and K and N multiples of 8 (16-byte row pitch), else
 *   CARBON_ERR_MISALIGNED.
 *
 * CARBON_TIER_SUPERACC - the correctly rounded tier (Carbon README,
 *   "Roadmap": superaccumulators, exact summation that needs no fixed
 *   order): the exact value of sum_r A(i,r) B(r,j) (+ bias), rounded once, to
 *   nearest-even, to the output type.  No order of the reduction shows in
 *   the result, so it is the same for any split or order of the reduction,
 *   as well as for every run, every M and every device.  An exact sum of
 *   zero gives +0; NaN operands (or inf times 0, or both infinities) give
 *   NaN, otherwise an infinite product or bias gives that infinity.  It
 *   differs from CARBON_TIER_EXACT where KBN's chunk values or its float64
 *   value round (e.g. 2^100 + 1 in one 256-chunk and -2^100 + 1 in the next:
 *   exact tier 0, this tier 2).  Accepts CARBON_F32, CARBON_BF16 and
 *   CARBON_F16, any shape and alignment.  bf16 runs the tensor-core exact
 *   sums of CARBON_TIER_EXACT (same workspace, below) without its rounding of
 *   chunk values; fp32 and fp16 run one warp per output over the reduction
 *   (no workspace; far slower than the bf16 path).
 *
 * Conventions
 *   - Pointers are DEVICE pointers on the current CUDA device; the caller
 *     owns every buffer.
 *   - Workspace: with CARBON_BF16 the exact tier builds a workspace on each
 *     call, taken from the device's stream-ordered memory pool with
 *     cudaMallocAsync on `stream` and released with cudaFreeAsync on
 *     `stream` before the call returns.  With R the reduction length (K, N
 *     or M for fwd, dX, dW), Rp = R rounded up to a multiple of 256, rows and
 *     cols the output's shape, La = rows rounded up to 128, Lb = cols rounded
 *     up to 64, C = Rp / 256 chunks and P in {1, 2, 4, 8} pieces per output
 *     (chosen from the tile and chunk counts), it takes about
 *       8 * Rp * (La + Lb)          digit planes of both operands (four bf16
 *                                   planes per element),
 *     + 12 * rows * cols * P        int64 partial sums and the fix-up list,
 *     + 12 * min(rows*cols*C, 2^22) chunk-repair list,
 *     + 16 * C * (La + Lb)          statistics per operand line and chunk,
 *     + 20 * (La + Lb)              line grains, row flags and row order
 *     bytes; e.g. about 422 MB for fwd with M = 8192, K = 768, N = 3072, and
 *     about 417 MB for dW of the same shapes.  If the pool cannot supply it
 *     the call returns CARBON_ERR_CUDA and enqueues nothing.  The fp32 and
 *     fp16 exact tier and the TC tier use no workspace (carbon_gemm_dw_f32's
 *     exact tier adds an 8-byte float64 staging value per output).
 *   - Calls are asynchronous: they validate, enqueue the kernels on `stream`
 *     and return.  Argument errors are returned synchronously and nothing is
 *     enqueued.  Errors raised while kernels run are reported by
 *     carbon_get_device_status().
 *   - M == 0 or an output dimension of 0: nothing to do, CARBON_OK.
 *     Reduction length 0: every output is +0 (fwd: the bias, rounded).
 *   - Negative sizes, sizes whose element counts overflow int64, and NULL
 *     pointers for operands with a non-zero element count:
 *     CARBON_ERR_INVALID_ARG.  `bias` may be NULL (no bias).
 *   - The output must not overlap any input (undefined result otherwise).
 *   - A current device other than compute capability 10.3 (GB300):
 *     CARBON_ERR_UNSUPPORTED.  There is no fallback path.
 *   - Fault injection, for testing a caller's error handling: with the
 *     environment variable CARBON_FAULT containing "launch" (a
 *     comma-separated list), carbon_gemm_fwd/dx/dw fail after their argument
 *     checks with CARBON_ERR_CUDA, as a failed launch would:
 *     carbon_last_cuda_error() names the injection, nothing is enqueued and
 *     no device is touched.
 *   - Thread-safe.
 */
#ifndef CARBON_GEMM_H
#define CARBON_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream: the same handle as cudaStream_t / CUstream.  NULL is the
 * legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st *carbon_stream_t;

typedef enum { CARBON_PASS_FWD = 0, CARBON_PASS_DX = 1, CARBON_PASS_DW = 2 } carbon_pass_t;

typedef enum {
    CARBON_F32 = 0,     /* IEEE binary32 */
    CARBON_BF16 = 1,    /* bfloat16 (top 16 bits of binary32) */
    CARBON_F16 = 2      /* IEEE binary16 (sgemm-bi lists float16 among its dtypes, "Use") */
} carbon_dtype_t;

typedef enum {
    CARBON_TIER_EXACT = 0,    /* float64 products, fixed-order KBN, one RNE */
    CARBON_TIER_TC = 1,       /* bf16 or fp16 tcgen05 MMA, fp32 accumulate */
    CARBON_TIER_SUPERACC = 2  /* exact sum (+ bias) rounded once: correctly rounded */
} carbon_tier_t;

typedef enum {
    CARBON_OK = 0,
    CARBON_ERR_INVALID_ARG = 1,   /* bad size, pointer, dtype or tier */
    CARBON_ERR_UNSUPPORTED = 2,   /* device or dtype/tier combination */
    CARBON_ERR_MISALIGNED = 3,    /* TC tier: pointer/pitch not 16-byte aligned */
    CARBON_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
    CARBON_ERR_TIMEOUT = 5,       /* a bounded device-side wait gave up */
    CARBON_ERR_SCRATCH_LIMIT = 6, /* needs more than the fixed no-allocation workspace */
    CARBON_ERR_OUT_OF_BOUNDS = 7  /* bounds-checked build only: a kernel skipped an access out of range */
} carbon_status_t;

/* Forward pass Y[M,N] = X[M,K] . W[K,N] + bias[N].
 * Reduction over K.  bias may be NULL. */
carbon_status_t carbon_gemm_fwd(void *Y, const void *X, const void *W, const void *bias,
                                int64_t M, int64_t K, int64_t N,
                                carbon_dtype_t dtype, carbon_tier_t tier,
                                carbon_stream_t stream);

/* Input gradient dX[M,K] = dY[M,N] . W[K,N]^T.  Reduction over N. */
carbon_status_t carbon_gemm_dx(void *dX, const void *dY, const void *W,
                               int64_t M, int64_t K, int64_t N,
                               carbon_dtype_t dtype, carbon_tier_t tier,
                               carbon_stream_t stream);

/* Weight gradient dW[K,N] = X[M,K]^T . dY[M,N].  Reduction over M (tokens). */
carbon_status_t carbon_gemm_dw(void *dW, const void *X, const void *dY,
                               int64_t M, int64_t K, int64_t N,
                               carbon_dtype_t dtype, carbon_tier_t tier,
                               carbon_stream_t stream);

/* Weight gradient of bf16 operands into an fp32 output (sgemm-bi's dW is
 * f32-accumulated, "Determinism contracts"): dW[K,N] fp32 = X[M,K]^T . dY[M,N]
 * with X and dY bf16.  CARBON_TIER_EXACT: the same float64 value as
 * carbon_gemm_dw (fixed-order KBN), rounded once, to nearest-even, to fp32;
 * it takes a float64 staging buffer of 8 bytes per output, on top of
 * carbon_gemm_dw's workspace, from the stream-ordered pool (released before
 * the call returns; CARBON_ERR_CUDA if the pool cannot supply it).
 * CARBON_TIER_TC: the fp32 accumulator of the tensor-core kernels, the value
 * carbon_gemm_dw would round to bf16.  Arguments, alignment and errors as for
 * carbon_gemm_dw with CARBON_BF16.  CARBON_TIER_SUPERACC:
 * CARBON_ERR_UNSUPPORTED. */
carbon_status_t carbon_gemm_dw_f32(float *dW, const void *X, const void *dY,
                                   int64_t M, int64_t K, int64_t N,
                                   carbon_tier_t tier, carbon_stream_t stream);

/* Exact tier, bf16, without any device allocation.  (No counterpart in the
 * source pages: this entry point exists for callers, not for the method.)
 *
 * Same result, bit for bit, as carbon_gemm_fwd / _dx / _dw with CARBON_BF16
 * and CARBON_TIER_EXACT, for callers that cannot allocate device memory while
 * they run -- code inside a framework whose allocator owns all of the GPU's
 * memory, latency-critical loops that must never block on or fail in an
 * allocator, or processes where the stream-ordered pool is unavailable.  The
 * workspace the bf16 exact tier needs comes instead from a fixed 64 MiB array
 * in device memory, part of the library's code module for this entry point.
 * CUDA reserves it on a device when it loads that module there -- with the
 * default lazy module loading, during the first call of this function on
 * that device -- and keeps it until the process exits.  No cudaMalloc,
 * cudaMallocAsync, cudaFree or other allocating call is made by the library;
 * but if the caller's allocator will later hold all free device memory, make
 * one small call (say M = K = N = 64) on each device before it does, so that
 * the module and its array are already in place.
 *
 * pass: CARBON_PASS_FWD (A = X, B = W, bias allowed), CARBON_PASS_DX
 * (A = dY, B = W), CARBON_PASS_DW (A = X, B = dY); out, A, B, bias, M, K, N
 * as in the per-pass entry points; all bf16, device pointers, caller-owned.
 * Limit: 4*Rp*(Lr + Lc) + 16*ceil(R/256)*(Lr + Lc) + 4*(rows*cols + 1) bytes
 * must fit 64 MiB, where R is the reduction length (K, N or M for fwd, dX,
 * dW), Rp = R rounded up to a multiple of 64, Lr, Lc the output's row and
 * column counts rounded up to multiples of 64, and rows*cols the output's size
 * (e.g. fwd with M = 8192, K = 768, N = 768 needs 52.8 MB);
 * larger problems return CARBON_ERR_SCRATCH_LIMIT and enqueue nothing.
 * The first call on each device (and the first after a new context, e.g.
 * after cudaDeviceReset) looks the array's device address up (not a stream
 * operation); make that first call before any stream capture.  Fault
 * injection (CARBON_FAULT=launch) applies as to the other entry points.  All
 * calls share the array and it keeps the last call's contents; the one word
 * that must start at zero is cleared on `stream` by each call.  Calls whose kernels may overlap on the GPU (other
 * streams, other host threads) race on the array: order them on one stream. */
carbon_status_t carbon_gemm_exact_bf16_noalloc(carbon_pass_t pass, void *out, const void *A,
                                               const void *B, const void *bias,
                                               int64_t M, int64_t K, int64_t N,
                                               carbon_stream_t stream);

/* ---- reductions split across ranks (exact tier) ----------------------------
 *
 * The Carbon README ("How It Works") replaces the data-parallel gradient
 * all-reduce with an all-gather followed by a reduction in rank order; its
 * "Roadmap" lists a deterministic multi-GPU all-reduce.  With the exact
 * tier's fixed order, a reduction split across ranks on 256-index chunk
 * boundaries can give the single-device bits exactly: each rank computes the
 * chunk values of its own chunks (they are the same doubles the single-device
 * call forms), the chunk values are gathered in rank order (= chunk order),
 * and the outer KBN, the bias and the rounding run once over all of them.
 * Typical use is dW = X^T . dY with the tokens (M) split across ranks: rank
 * r holds tokens [m_r, m_{r+1}) with every m_r a multiple of 256. */

/* Chunk values of one rank's share of the reduction.  pass, A, B, M, K, N and
 * dtype as in carbon_gemm_fwd / _dx / _dw with CARBON_TIER_EXACT (bias is not
 * taken: it joins in carbon_chunk_values_combine), the reduction being this
 * rank's share only (e.g. dW: A = X rows m_r .. m_{r+1}-1, B = the same rows
 * of dY, M = m_{r+1} - m_r).  P: device float64 [C][rows][cols], C =
 * ceil(R / 256), rows x cols the output shape of the pass; P[q][i][j] is the
 * chunk value fl(s + c) of KBN over the products of reduction indices
 * 256q .. min(256q + 255, R - 1), left to right.  Runs the float64 KBN kernel
 * of the exact tier for every dtype (for bf16 slower than carbon_gemm_dw's
 * tensor-core path); no workspace.  Errors as for the per-pass entry points;
 * R == 0 writes nothing. */
carbon_status_t carbon_gemm_chunk_values(carbon_pass_t pass, double *P, const void *A,
                                         const void *B, int64_t M, int64_t K, int64_t N,
                                         carbon_dtype_t dtype, carbon_stream_t stream);

/* out[i][j] = RNE_dtype( KBN over q = 0 .. nchunks-1 of P[q][i][j], left to
 * right, (+ bias[j]) ): the exact tier's steps after its chunk values.  With P
 * the chunk values of every rank in rank order this is bit-identical to the
 * single-device exact-tier call over the whole reduction.  P: device float64
 * [nchunks][rows][cols]; bias: device, dtype-typed [cols], or NULL; out:
 * device [rows][cols] of dtype.  nchunks == 0 gives +0 (or the bias). */
carbon_status_t carbon_chunk_values_combine(void *out, const double *P, int64_t nchunks,
                                            int64_t rows, int64_t cols, const void *bias,
                                            carbon_dtype_t dtype, carbon_stream_t stream);

/* Synchronises `stream`, then reports (and clears) the device status word
 * that kernels set when a bounded wait gives up (CARBON_ERR_TIMEOUT) or, in
 * the bounds-checked build (libcarbon_gemm_bounds.so, compiled with
 * CARBON_DEBUG_BOUNDS), when a kernel skipped an access outside its buffer
 * (CARBON_ERR_OUT_OF_BOUNDS); or CARBON_ERR_CUDA if the stream reports an
 * error. */
carbon_status_t carbon_get_device_status(carbon_stream_t stream);

/* Static, human-readable name of a status code. */
const char *carbon_status_string(carbon_status_t status);

/* Message of the last CUDA error seen by this thread inside the library
 * ("" if none). */
const char *carbon_last_cuda_error(void);

/* ABI version of this header: (major << 16) | minor.  Minor 1 added
 * carbon_gemm_exact_bf16_noalloc and CARBON_ERR_SCRATCH_LIMIT; minor 2 the
 * CARBON_TIER_SUPERACC tier, carbon_gemm_chunk_values,
 * carbon_chunk_values_combine and CARBON_ERR_OUT_OF_BOUNDS. */
int carbon_abi_version(void);

#define CARBON_ABI_VERSION ((1 << 16) | 2)

#ifdef __cplusplus
}
#endif

#endif /* CARBON_GEMM_H */
