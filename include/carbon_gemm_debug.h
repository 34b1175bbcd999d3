/*
 * carbon_gemm_debug.h - inspection and measurement entry points of the
 * carbon_gemm library.  Not needed to use the GEMMs; used by the parity
 * tests and the benchmark.  Same conventions as carbon_gemm.h (device
 * pointers, asynchronous on `stream` unless stated, status codes).
 */
#ifndef CARBON_GEMM_DEBUG_H
#define CARBON_GEMM_DEBUG_H

#include "carbon_gemm.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Exact tier, float64 value before the output rounding.
 * Runs the same kernel arithmetic as carbon_gemm_{fwd,dx,dw} with
 * CARBON_TIER_EXACT (fixed-order KBN of the float64 products, plus the bias
 * for fwd) and stores the float64 result, so it can be compared bit for bit
 * with a CPU implementation before rounding.
 * pass: CARBON_PASS_*; A, B = (X, W) fwd, (dY, W) dX, (X, dY) dW; bias is
 * used by fwd only (NULL allowed).  y64: float64 [rows x cols] with the
 * output shape of the pass. */
carbon_status_t carbon_debug_exact_y64(carbon_pass_t pass, double *y64,
                                       const void *A, const void *B, const void *bias,
                                       int64_t M, int64_t K, int64_t N,
                                       carbon_dtype_t dtype, carbon_stream_t stream);

/* Tensor-core tier, fp32 value before the bf16 rounding (accumulator plus
 * bias for fwd), same kernel and K schedule as the CARBON_TIER_TC entry
 * points.  acc: fp32 [rows x cols] with the output shape of the pass. */
carbon_status_t carbon_debug_tc_f32(carbon_pass_t pass, float *acc,
                                    const void *A, const void *B, const void *bias,
                                    int64_t M, int64_t K, int64_t N,
                                    carbon_stream_t stream);

/* The exact tier's device-side output rounding applied to n float64 values
 * (out: fp32, bf16 or fp16 elements), to check it against
 * round-to-nearest-even. */
carbon_status_t carbon_debug_round(carbon_dtype_t dtype, void *out, const double *in,
                                   int64_t n, carbon_stream_t stream);

/* Launches one block whose single thread waits on an mbarrier that nothing
 * arrives on, with a budget of `budget_ns` nanoseconds; the wait gives up,
 * sets the device status word and the kernel returns.  A following
 * carbon_get_device_status() must report CARBON_ERR_TIMEOUT.  Exercises the
 * timeout path that every bounded wait in the library shares. */
carbon_status_t carbon_debug_timeout_probe(int64_t budget_ns, carbon_stream_t stream);

/* FP64 issue-rate microbenchmark on the current device (blocking).
 * Runs streams of independent DFMA and of independent DADD instructions
 * on every SM and reports instructions per second (lane operations: one
 * DFMA counts 1).  Used as the FP64 roofline denominator. */
carbon_status_t carbon_measure_fp64_rate(double *dfma_per_s, double *dadd_per_s,
                                         carbon_stream_t stream);

/* Integer multiply-add rate microbenchmark on the current device (blocking):
 * independent 32x32->64-bit mad.wide.s32 chains on every SM, reported as
 * multiply-adds per second.  The roofline denominator of the integer-pipe
 * bf16 kernel (the no-allocation entry point's path). */
carbon_status_t carbon_measure_int_mac_rate(double *macs_per_s, carbon_stream_t stream);

/* Timing of the bf16 exact tier's tensor-core kernel.  enable != 0 starts
 * recording a CUDA event pair on the caller's stream around every launch of
 * that kernel (outside CUDA-graph capture only) and clears the previous
 * record; enable == 0 stops recording.  The kernel also counts the digit
 * plane products it issues: one unit is one A digit plane of 128 rows times
 * one B digit plane of 64 columns over a 256-deep chunk (the share of one
 * plane in 16 tcgen05.mma instructions of M = 128, K = 16 and N = 64 per B
 * plane), 2 * 128 * 64 * 256 flops.  The accumulators' start MMAs are not
 * counted. */
void carbon_debug_kernel_timing(int enable);

/* Sum of the recorded launches' durations in milliseconds (blocking: waits
 * for the recorded events), their number, and the plane products issued
 * since the last carbon_debug_kernel_timing(1).  Any pointer may be NULL. */
carbon_status_t carbon_debug_kernel_time(double *ms, int64_t *launches, int64_t *plane_products);

/* While kernel timing is on, the same calls' time split into three phases,
 * summed over the calls in milliseconds (blocking): pre-pass (from the
 * call's first device operation to the start of the tensor-core kernel:
 * workspace set-up, digit planes, row order), the tensor-core kernel, and
 * post-pass (chunk repair, finalize, fix-up).  Any pointer may be NULL. */
carbon_status_t carbon_debug_exact_phase_time(double *pre_ms, double *main_ms, double *post_ms);

/* While kernel timing is on, the bf16 exact tier also counts, per call, the
 * (output, chunk) pairs it recomputes in the chunk repair (a line of that
 * chunk too wide for the digit planes) and the outputs it recomputes whole
 * in the fix-up (inf/NaN operands, extreme widths, or integer sums that would
 * leave the int64 range).  Returns the totals since timing was enabled
 * (blocking: synchronizes the device).  Any pointer may be NULL. */
carbon_status_t carbon_debug_exact_path_counts(int64_t *chunk_repairs, int64_t *fixups);

/* Number of kernel launches the library has enqueued in this process. */
int64_t carbon_debug_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* CARBON_GEMM_DEBUG_H */
