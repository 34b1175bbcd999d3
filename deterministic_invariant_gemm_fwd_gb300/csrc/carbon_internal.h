// carbon_internal.h - declarations shared by the translation units of the
// carbon_gemm library (never by its tests' CPU reference).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/carbon_gemm.h"
#include "../../include/carbon_gemm_debug.h"

namespace carbon {

// Passes of a linear layer, expressed as one generic product
//   out[i, j] = sum_r A(i, r) * B(r, j),  r = 0 .. R-1
// with A(i, r) = A[i * a_si + r * a_sr] and B(r, j) = B[r * b_sr + j * b_sj].
//   fwd: A = X  [M,K] (a_si = K, a_sr = 1), B = W  [K,N] (b_sr = N, b_sj = 1), R = K
//   dX : A = dY [M,N] (a_si = N, a_sr = 1), B = W  [K,N] (b_sr = 1, b_sj = N), R = N
//   dW : A = X  [M,K] (a_si = 1, a_sr = K), B = dY [M,N] (b_sr = N, b_sj = 1), R = M
struct Problem {
    int pass;                 // CARBON_PASS_*
    int dtype;                // CARBON_F32 / CARBON_BF16
    const void *A, *B, *bias; // bias: fwd only, may be null
    void *out;
    int64_t M, K, N;          // layer sizes
    int64_t rows, cols, R;    // output shape and reduction length
};

inline Problem make_problem(int pass, int dtype, void *out, const void *A, const void *B,
                            const void *bias, int64_t M, int64_t K, int64_t N) {
    Problem p;
    p.pass = pass; p.dtype = dtype; p.A = A; p.B = B;
    p.bias = (pass == CARBON_PASS_FWD) ? bias : nullptr;
    p.out = out; p.M = M; p.K = K; p.N = N;
    p.rows = (pass == CARBON_PASS_DW) ? K : M;
    p.cols = (pass == CARBON_PASS_DX) ? K : N;
    p.R = (pass == CARBON_PASS_FWD) ? K : (pass == CARBON_PASS_DX ? N : M);
    return p;
}

// Launches kernel `kern` on `stream`; with `early`, under programmatic
// stream serialization: it may be scheduled before the previous kernel on
// the stream has finished, and must call wait_prior_grid() (device_sync.cuh)
// before touching global memory.  cluster_x > 1 also sets a cluster of that
// many CTAs along x.
template <typename... Params, typename... Args>
cudaError_t launch_kernel(bool early, void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, unsigned cluster_x, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (early) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = n ? attr : nullptr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// The library's usual launch: scheduled early (see launch_kernel).
template <typename... Params, typename... Args>
cudaError_t launch_k(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t stream, unsigned cluster_x, Args &&...args) {
    return launch_kernel(true, kern, grid, block, smem, stream, cluster_x, static_cast<Args &&>(args)...);
}

// Records a CUDA error message for carbon_last_cuda_error(); returns
// CARBON_ERR_CUDA when err != cudaSuccess, CARBON_OK otherwise.
carbon_status_t note_cuda(cudaError_t err);

// Counts kernel launches enqueued by the library.
void count_launch(int n = 1);

// Checks that the current device is a GB300 (compute capability 10.3) and
// returns its SM count.
carbon_status_t current_device(int *device, int *sm_count);
// Host-side fault injection: CARBON_ERR_CUDA (message names the injection)
// when the environment variable CARBON_FAULT lists "launch", else CARBON_OK.
// Every GEMM entry point calls it after its argument checks.
carbon_status_t injected_launch_failure();

// Exact tier (exact_kbn.cu).  out_f64 selects the float64 pre-rounding output.
carbon_status_t exact_launch(const Problem &p, bool out_f64, cudaStream_t stream);
// bf16 exact tier on the integer pipes (exact_int.cu); same bits.
carbon_status_t exact_int_launch(const Problem &p, bool out_f64, cudaStream_t stream);
// bf16 exact tier on the tensor cores (exact_tc.cu); same bits.  super: the
// correctly rounded tier instead (exact total and bias rounded once).
carbon_status_t exact_tc_launch(const Problem &p, bool out_f64, bool super, cudaStream_t stream);
// Correctly rounded tier, one output per warp, any dtype (superacc.cu).
carbon_status_t superacc_launch(const Problem &p, cudaStream_t stream);
// The same kernel for the bf16 outputs listed in work_list[0 .. *work_count).
cudaError_t superacc_fixup_bf16(const Problem &p, const unsigned int *work_count,
                                const unsigned int *work_list, int blocks, cudaStream_t stream);
carbon_status_t exact_round_launch(int dtype, void *out, const double *in, int64_t n,
                                   cudaStream_t stream);
// Chunk values fl(s + c) of every output into p.out (float64
// [ceil(R/256)][rows][cols]), and the outer KBN + bias + rounding over chunk
// values computed elsewhere (exact_kbn.cu).
carbon_status_t exact_chunk_values_launch(const Problem &p, cudaStream_t stream);
carbon_status_t exact_combine_launch(int dtype, void *out, const double *P, int64_t nchunks,
                                     int64_t rows, int64_t cols, const void *bias,
                                     cudaStream_t stream);

// 2-D tiled TMA tensor map over a row-major [outer, inner] matrix (row pitch
// row_bytes); out-of-range elements read as zero.  cudaErrorInvalidValue if
// the driver rejects the description.
cudaError_t encode_tensor_map_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base,
                                 uint64_t inner, uint64_t outer, uint64_t row_bytes,
                                 uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);

// Read and clear the exact tier's device status words (exact_int.cu,
// exact_tc.cu).
carbon_status_t exact_take_device_status();
carbon_status_t exact_tc_take_device_status();
// Kernel timing of the bf16 exact tier's tensor-core kernel (exact_tc.cu).
void exact_tc_timing(int enable);
carbon_status_t exact_tc_time(double *ms, int64_t *launches, int64_t *kgroups);
carbon_status_t exact_tc_phase_time(double *pre_ms, double *main_ms, double *post_ms);
carbon_status_t exact_tc_path_counts(int64_t *repairs, int64_t *fixups);

// Tensor-core tier (tc_gemm.cu).  out_f32 selects the fp32 pre-rounding output.
carbon_status_t tc_launch(const Problem &p, bool out_f32, cudaStream_t stream);
// Reads and clears the tensor-core tier's device status word.
carbon_status_t tc_take_device_status();

// Measurement helpers (measure.cu).
carbon_status_t measure_take_device_status();
// Status words of the float64 KBN kernels and the superaccumulator
// (bounds-checked build).
carbon_status_t kbn_take_device_status();
carbon_status_t superacc_take_device_status();

}  // namespace carbon
