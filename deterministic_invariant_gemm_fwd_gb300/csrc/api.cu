// api.cu - the C ABI of the carbon_gemm library: argument checks, device
// check, dispatch to the exact and tensor-core tiers, status reporting.
//
// Entry points follow the shape of sgemm-bi's low-level engine call (raw
// device pointers, m/k/n, dtype, explicit stream, tensor-core switch;
// sgemm-bi page, "Use") with weights stored [in, out].
#include "carbon_internal.h"

#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>

namespace carbon {

namespace {
thread_local char g_last_cuda_error[256] = "";
std::atomic<int64_t> g_launches{0};
// Per-device cache: 0 = unknown, -1 = not a GB300, >0 = SM count.
std::atomic<int> g_device_sms[128];
}  // namespace

carbon_status_t note_cuda(cudaError_t err) {
    if (err == cudaSuccess) return CARBON_OK;
    std::snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "%s: %s",
                  cudaGetErrorName(err), cudaGetErrorString(err));
    return CARBON_ERR_CUDA;
}

void count_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

carbon_status_t current_device(int *device, int *sm_count) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return note_cuda(err);
    if (dev < 0 || dev >= 128) return CARBON_ERR_UNSUPPORTED;
    int cached = g_device_sms[dev].load(std::memory_order_acquire);
    if (cached == 0) {
        int major = 0, minor = 0, sms = 0;
        if ((err = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (err = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return note_cuda(err);
        cached = (major == 10 && minor == 3 && sms > 0) ? sms : -1;
        g_device_sms[dev].store(cached, std::memory_order_release);
    }
    if (cached < 0) return CARBON_ERR_UNSUPPORTED;
    if (device) *device = dev;
    if (sm_count) *sm_count = cached;
    return CARBON_OK;
}

namespace {

bool mul_ok(int64_t a, int64_t b, int64_t *out) {
    return !__builtin_mul_overflow(a, b, out);
}

// Checks sizes, dtype, tier and pointers.  Returns CARBON_OK and sets
// *nothing_to_do when the output is empty.
carbon_status_t check_args(const Problem &p, int tier, bool *nothing_to_do) {
    *nothing_to_do = false;
    if (p.M < 0 || p.K < 0 || p.N < 0) return CARBON_ERR_INVALID_ARG;
    if (p.dtype != CARBON_F32 && p.dtype != CARBON_BF16 && p.dtype != CARBON_F16)
        return CARBON_ERR_INVALID_ARG;
    if (tier != CARBON_TIER_EXACT && tier != CARBON_TIER_TC && tier != CARBON_TIER_SUPERACC)
        return CARBON_ERR_INVALID_ARG;
    int64_t mk, kn, mn, t;
    if (!mul_ok(p.M, p.K, &mk) || !mul_ok(p.K, p.N, &kn) || !mul_ok(p.M, p.N, &mn))
        return CARBON_ERR_INVALID_ARG;
    // byte counts must fit as well (8-byte float64 debug outputs included)
    if (!mul_ok(mk, 8, &t) || !mul_ok(kn, 8, &t) || !mul_ok(mn, 8, &t))
        return CARBON_ERR_INVALID_ARG;
    int64_t a_elems, b_elems;
    switch (p.pass) {
    case CARBON_PASS_FWD: a_elems = mk; b_elems = kn; break;
    case CARBON_PASS_DX:  a_elems = mn; b_elems = kn; break;
    case CARBON_PASS_DW:  a_elems = mk; b_elems = mn; break;
    default: return CARBON_ERR_INVALID_ARG;
    }
    const int64_t out_elems = p.rows * p.cols;
    if (out_elems > 0 && p.out == nullptr) return CARBON_ERR_INVALID_ARG;
    if (out_elems > 0 && a_elems > 0 && p.A == nullptr) return CARBON_ERR_INVALID_ARG;
    if (out_elems > 0 && b_elems > 0 && p.B == nullptr) return CARBON_ERR_INVALID_ARG;
    if (tier == CARBON_TIER_TC && p.dtype == CARBON_F32) return CARBON_ERR_UNSUPPORTED;
    if (out_elems == 0) *nothing_to_do = true;
    return CARBON_OK;
}

// Host-side fault injection, for tests of a caller's error handling: the
// environment variable CARBON_FAULT holds a comma-separated list of fault
// names; "launch" makes every GEMM call fail after its argument checks with
// CARBON_ERR_CUDA, as a failed launch would, enqueuing nothing and touching
// no device.  Read at each call; off when unset.
bool fault_injected(const char *name) {
    const char *v = std::getenv("CARBON_FAULT");
    if (v == nullptr) return false;
    const size_t n = std::strlen(name);
    for (const char *q = v; *q;) {
        const char *end = std::strchr(q, ',');
        const size_t len = end ? (size_t)(end - q) : std::strlen(q);
        if (len == n && std::strncmp(q, name, n) == 0) return true;
        if (!end) break;
        q = end + 1;
    }
    return false;
}

}  // namespace

// CARBON_ERR_CUDA with the injection named, when "launch" is injected.
carbon_status_t injected_launch_failure() {
    if (!fault_injected("launch")) return CARBON_OK;
    std::snprintf(g_last_cuda_error, sizeof g_last_cuda_error,
                  "injected launch failure (CARBON_FAULT=launch)");
    return CARBON_ERR_CUDA;
}

namespace {

carbon_status_t run(const Problem &p, int tier, int debug_out, carbon_stream_t stream) {
    bool nothing = false;
    carbon_status_t st = check_args(p, tier, &nothing);
    if (st != CARBON_OK || nothing) return st;
    st = injected_launch_failure();
    if (st != CARBON_OK) return st;
    st = current_device(nullptr, nullptr);
    if (st != CARBON_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (tier == CARBON_TIER_EXACT)
        return p.dtype == CARBON_BF16 ? exact_tc_launch(p, debug_out != 0, false, s)
                                      : exact_launch(p, debug_out != 0, s);
    if (tier == CARBON_TIER_SUPERACC) {
        if (debug_out) return CARBON_ERR_UNSUPPORTED;    // no float64 value: one rounding of the exact sum
        return p.dtype == CARBON_BF16 ? exact_tc_launch(p, false, true, s) : superacc_launch(p, s);
    }
    return tc_launch(p, debug_out != 0, s);
}

}  // namespace
}  // namespace carbon

using carbon::make_problem;

extern "C" {

carbon_status_t carbon_gemm_fwd(void *Y, const void *X, const void *W, const void *bias,
                                int64_t M, int64_t K, int64_t N, carbon_dtype_t dtype,
                                carbon_tier_t tier, carbon_stream_t stream) {
    return carbon::run(make_problem(CARBON_PASS_FWD, dtype, Y, X, W, bias, M, K, N),
                       tier, 0, stream);
}

carbon_status_t carbon_gemm_dx(void *dX, const void *dY, const void *W, int64_t M, int64_t K,
                               int64_t N, carbon_dtype_t dtype, carbon_tier_t tier,
                               carbon_stream_t stream) {
    return carbon::run(make_problem(CARBON_PASS_DX, dtype, dX, dY, W, nullptr, M, K, N),
                       tier, 0, stream);
}

carbon_status_t carbon_gemm_dw(void *dW, const void *X, const void *dY, int64_t M, int64_t K,
                               int64_t N, carbon_dtype_t dtype, carbon_tier_t tier,
                               carbon_stream_t stream) {
    return carbon::run(make_problem(CARBON_PASS_DW, dtype, dW, X, dY, nullptr, M, K, N),
                       tier, 0, stream);
}

carbon_status_t carbon_gemm_dw_f32(float *dW, const void *X, const void *dY, int64_t M, int64_t K,
                                   int64_t N, carbon_tier_t tier, carbon_stream_t stream) {
    const carbon::Problem p = make_problem(CARBON_PASS_DW, CARBON_BF16, dW, X, dY, nullptr, M, K, N);
    if (tier == CARBON_TIER_TC) return carbon::run(p, CARBON_TIER_TC, 1, stream);   // the fp32 accumulator
    if (tier == CARBON_TIER_SUPERACC) return CARBON_ERR_UNSUPPORTED;
    if (tier != CARBON_TIER_EXACT) return CARBON_ERR_INVALID_ARG;
    // exact tier: the float64 value into a staging buffer, then one rounding to fp32
    bool nothing = false;
    carbon_status_t st = carbon::check_args(p, CARBON_TIER_EXACT, &nothing);
    if (st != CARBON_OK || nothing) return st;
    st = carbon::injected_launch_failure();
    if (st != CARBON_OK) return st;
    st = carbon::current_device(nullptr, nullptr);
    if (st != CARBON_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t n = K * N;
    double *y64 = nullptr;
    cudaError_t err = cudaMallocAsync(reinterpret_cast<void **>(&y64), (size_t)n * sizeof(double), s);
    if (err != cudaSuccess) return carbon::note_cuda(err);
    carbon::Problem q = p;
    q.out = y64;
    st = carbon::run(q, CARBON_TIER_EXACT, 1, stream);
    if (st == CARBON_OK) st = carbon::exact_round_launch(CARBON_F32, dW, y64, n, s);
    const cudaError_t ferr = cudaFreeAsync(y64, s);
    if (st == CARBON_OK && ferr != cudaSuccess) st = carbon::note_cuda(ferr);
    return st;
}

carbon_status_t carbon_gemm_chunk_values(carbon_pass_t pass, double *P, const void *A,
                                        const void *B, int64_t M, int64_t K, int64_t N,
                                        carbon_dtype_t dtype, carbon_stream_t stream) {
    if (pass < CARBON_PASS_FWD || pass > CARBON_PASS_DW) return CARBON_ERR_INVALID_ARG;
    const carbon::Problem p = make_problem(pass, dtype, P, A, B, nullptr, M, K, N);
    bool nothing = false;
    carbon_status_t st = carbon::check_args(p, CARBON_TIER_EXACT, &nothing);
    if (st != CARBON_OK || nothing) return st;
    int64_t chunks = (p.R + 255) / 256, total;
    if (__builtin_mul_overflow(chunks, p.rows * p.cols, &total) ||
        __builtin_mul_overflow(total, (int64_t)8, &total))
        return CARBON_ERR_INVALID_ARG;
    st = carbon::injected_launch_failure();
    if (st != CARBON_OK) return st;
    st = carbon::current_device(nullptr, nullptr);
    if (st != CARBON_OK) return st;
    return carbon::exact_chunk_values_launch(p, reinterpret_cast<cudaStream_t>(stream));
}

carbon_status_t carbon_chunk_values_combine(void *out, const double *P, int64_t nchunks,
                                            int64_t rows, int64_t cols, const void *bias,
                                            carbon_dtype_t dtype, carbon_stream_t stream) {
    if (dtype != CARBON_F32 && dtype != CARBON_BF16 && dtype != CARBON_F16) return CARBON_ERR_INVALID_ARG;
    if (nchunks < 0 || rows < 0 || cols < 0) return CARBON_ERR_INVALID_ARG;
    int64_t n, total;
    if (__builtin_mul_overflow(rows, cols, &n) || __builtin_mul_overflow(n, nchunks, &total) ||
        __builtin_mul_overflow(total, (int64_t)8, &total))
        return CARBON_ERR_INVALID_ARG;
    if (n == 0) return CARBON_OK;
    if (out == nullptr || (nchunks > 0 && P == nullptr)) return CARBON_ERR_INVALID_ARG;
    carbon_status_t st = carbon::injected_launch_failure();
    if (st != CARBON_OK) return st;
    st = carbon::current_device(nullptr, nullptr);
    if (st != CARBON_OK) return st;
    return carbon::exact_combine_launch(dtype, out, P, nchunks, rows, cols, bias,
                                        reinterpret_cast<cudaStream_t>(stream));
}

carbon_status_t carbon_debug_exact_y64(carbon_pass_t pass, double *y64, const void *A,
                                       const void *B, const void *bias, int64_t M, int64_t K,
                                       int64_t N, carbon_dtype_t dtype, carbon_stream_t stream) {
    if (pass < CARBON_PASS_FWD || pass > CARBON_PASS_DW) return CARBON_ERR_INVALID_ARG;
    return carbon::run(make_problem(pass, dtype, y64, A, B, bias, M, K, N),
                       CARBON_TIER_EXACT, 1, stream);
}

carbon_status_t carbon_debug_tc_f32(carbon_pass_t pass, float *acc, const void *A,
                                    const void *B, const void *bias, int64_t M, int64_t K,
                                    int64_t N, carbon_stream_t stream) {
    if (pass < CARBON_PASS_FWD || pass > CARBON_PASS_DW) return CARBON_ERR_INVALID_ARG;
    return carbon::run(make_problem(pass, CARBON_BF16, acc, A, B, bias, M, K, N),
                       CARBON_TIER_TC, 1, stream);
}

carbon_status_t carbon_debug_round(carbon_dtype_t dtype, void *out, const double *in,
                                   int64_t n, carbon_stream_t stream) {
    if (dtype != CARBON_F32 && dtype != CARBON_BF16 && dtype != CARBON_F16) return CARBON_ERR_INVALID_ARG;
    if (n < 0 || (n > 0 && (out == nullptr || in == nullptr))) return CARBON_ERR_INVALID_ARG;
    if (n == 0) return CARBON_OK;
    carbon_status_t st = carbon::current_device(nullptr, nullptr);
    if (st != CARBON_OK) return st;
    return carbon::exact_round_launch(dtype, out, in, n, reinterpret_cast<cudaStream_t>(stream));
}

carbon_status_t carbon_get_device_status(carbon_stream_t stream) {
    carbon_status_t st = carbon::note_cuda(
        cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
    const carbon_status_t tc = carbon::tc_take_device_status();
    const carbon_status_t ms = carbon::measure_take_device_status();
    const carbon_status_t ex = carbon::exact_take_device_status();
    const carbon_status_t et = carbon::exact_tc_take_device_status();
    const carbon_status_t kb = carbon::kbn_take_device_status();
    const carbon_status_t sa = carbon::superacc_take_device_status();
    if (st != CARBON_OK) return st;
    if (tc != CARBON_OK) return tc;
    if (ex != CARBON_OK) return ex;
    if (et != CARBON_OK) return et;
    if (kb != CARBON_OK) return kb;
    if (sa != CARBON_OK) return sa;
    return ms;
}

const char *carbon_status_string(carbon_status_t status) {
    switch (status) {
    case CARBON_OK: return "CARBON_OK";
    case CARBON_ERR_INVALID_ARG: return "CARBON_ERR_INVALID_ARG";
    case CARBON_ERR_UNSUPPORTED: return "CARBON_ERR_UNSUPPORTED";
    case CARBON_ERR_MISALIGNED: return "CARBON_ERR_MISALIGNED";
    case CARBON_ERR_CUDA: return "CARBON_ERR_CUDA";
    case CARBON_ERR_TIMEOUT: return "CARBON_ERR_TIMEOUT";
    case CARBON_ERR_SCRATCH_LIMIT: return "CARBON_ERR_SCRATCH_LIMIT";
    case CARBON_ERR_OUT_OF_BOUNDS: return "CARBON_ERR_OUT_OF_BOUNDS";
    }
    return "CARBON_ERR_UNKNOWN";
}

const char *carbon_last_cuda_error(void) { return carbon::g_last_cuda_error; }

int carbon_abi_version(void) { return CARBON_ABI_VERSION; }

int64_t carbon_debug_launch_count(void) { return carbon::g_launches.load(); }

void carbon_debug_kernel_timing(int enable) { carbon::exact_tc_timing(enable); }

carbon_status_t carbon_debug_kernel_time(double *ms, int64_t *launches, int64_t *plane_products) {
    return carbon::exact_tc_time(ms, launches, plane_products);
}

carbon_status_t carbon_debug_exact_phase_time(double *pre_ms, double *main_ms, double *post_ms) {
    return carbon::exact_tc_phase_time(pre_ms, main_ms, post_ms);
}

carbon_status_t carbon_debug_exact_path_counts(int64_t *chunk_repairs, int64_t *fixups) {
    return carbon::exact_tc_path_counts(chunk_repairs, fixups);
}

}  // extern "C"
