// measure.cu - FP64 issue-rate microbenchmark (the exact tier's roofline
// denominator) and the timeout self-test of the bounded device waits.
#include "carbon_internal.h"
#include "device_sync.cuh"

namespace carbon {
namespace {

__device__ unsigned int g_measure_status = 0;

constexpr int kChains = 8;

// Independent DFMA (or DADD) chains per thread: throughput, not latency.
template <bool FMA>
__global__ void fp64_rate_kernel(double *sink, int iters, double a, double b) {
    double x[kChains];
#pragma unroll
    for (int i = 0; i < kChains; ++i) x[i] = threadIdx.x * 1e-3 + i;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < kChains; ++i) x[i] = FMA ? __fma_rn(x[i], a, b) : __dadd_rn(x[i], b);
    }
    double s = 0.0;
#pragma unroll
    for (int i = 0; i < kChains; ++i) s += x[i];
    sink[blockIdx.x * (int64_t)blockDim.x + threadIdx.x] = s;
}

// Independent 32x32->64-bit integer multiply-add chains (one mad.wide.s32
// each), operands refreshed from a 4x4 outer product like a GEMM micro-tile.
__global__ void int_mac_rate_kernel(long long *sink, int iters, int seed) {
    long long acc[4][4];
    int a[4], b[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) { a[i] = seed * 7 + i + (int)threadIdx.x; b[i] = seed * 3 - i; }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = i * 4 + j;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                asm("mad.wide.s32 %0, %1, %2, %0;" : "+l"(acc[i][j]) : "r"(a[i]), "r"(b[j]));
#pragma unroll
        for (int i = 0; i < 4; ++i) { a[i] ^= it; b[i] += 3; }
    }
    long long s = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) s ^= acc[i][j];
    sink[blockIdx.x * (int64_t)blockDim.x + threadIdx.x] = s;
}

__global__ void timeout_probe_kernel(int64_t budget_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = smem_addr(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    if (!mbar_wait(b, 0, (uint64_t)budget_ns))       // nothing ever arrives
        atomicExch(&g_measure_status, (unsigned)CARBON_ERR_TIMEOUT);
}

}  // namespace

carbon_status_t measure_take_device_status() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_measure_status, sizeof v) != cudaSuccess) return CARBON_OK;
    if (v != 0) cudaMemcpyToSymbol(g_measure_status, &zero, sizeof zero);
    return (carbon_status_t)v;
}

}  // namespace carbon

extern "C" carbon_status_t carbon_debug_timeout_probe(int64_t budget_ns, carbon_stream_t stream) {
    if (budget_ns <= 0 || budget_ns > 10000000000ll) return CARBON_ERR_INVALID_ARG;
    carbon_status_t st = carbon::current_device(nullptr, nullptr);
    if (st != CARBON_OK) return st;
    carbon::timeout_probe_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(budget_ns);
    carbon::count_launch();
    return carbon::note_cuda(cudaGetLastError());
}

extern "C" carbon_status_t carbon_measure_fp64_rate(double *dfma_per_s, double *dadd_per_s,
                                                    carbon_stream_t stream) {
    int sms = 0;
    carbon_status_t st = carbon::current_device(nullptr, &sms);
    if (st != CARBON_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int threads = 256, blocks = sms * 8, iters = 2000;
    double *sink = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    cudaError_t err = cudaMalloc(&sink, sizeof(double) * (size_t)threads * blocks);
    if (err == cudaSuccess) err = cudaEventCreate(&e0);
    if (err == cudaSuccess) err = cudaEventCreate(&e1);
    double best[2] = {0.0, 0.0};
    for (int which = 0; which < 2 && err == cudaSuccess; ++which) {
        for (int rep = 0; rep < 4 && err == cudaSuccess; ++rep) {   // rep 0 warms up
            cudaEventRecord(e0, s);
            if (which == 0)
                carbon::fp64_rate_kernel<true><<<blocks, threads, 0, s>>>(sink, iters, 1.0000001, 1e-9);
            else
                carbon::fp64_rate_kernel<false><<<blocks, threads, 0, s>>>(sink, iters, 1.0000001, 1e-9);
            carbon::count_launch();
            cudaEventRecord(e1, s);
            err = cudaEventSynchronize(e1);
            if (err == cudaSuccess) err = cudaGetLastError();
            float ms = 0.f;
            if (err == cudaSuccess) err = cudaEventElapsedTime(&ms, e0, e1);
            const double ops = (double)threads * blocks * iters * carbon::kChains;
            if (rep > 0 && ms > 0.f && ops / (ms * 1e-3) > best[which]) best[which] = ops / (ms * 1e-3);
        }
    }
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    if (sink) cudaFree(sink);
    if (err != cudaSuccess) return carbon::note_cuda(err);
    if (dfma_per_s) *dfma_per_s = best[0];
    if (dadd_per_s) *dadd_per_s = best[1];
    return CARBON_OK;
}

extern "C" carbon_status_t carbon_measure_int_mac_rate(double *macs_per_s, carbon_stream_t stream) {
    int sms = 0;
    carbon_status_t st = carbon::current_device(nullptr, &sms);
    if (st != CARBON_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int threads = 256, blocks = sms * 8, iters = 4000;
    long long *sink = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    cudaError_t err = cudaMalloc(&sink, sizeof(long long) * (size_t)threads * blocks);
    if (err == cudaSuccess) err = cudaEventCreate(&e0);
    if (err == cudaSuccess) err = cudaEventCreate(&e1);
    double best = 0.0;
    for (int rep = 0; rep < 4 && err == cudaSuccess; ++rep) {       // rep 0 warms up
        cudaEventRecord(e0, s);
        carbon::int_mac_rate_kernel<<<blocks, threads, 0, s>>>(sink, iters, rep + 1);
        carbon::count_launch();
        cudaEventRecord(e1, s);
        err = cudaEventSynchronize(e1);
        if (err == cudaSuccess) err = cudaGetLastError();
        float ms = 0.f;
        if (err == cudaSuccess) err = cudaEventElapsedTime(&ms, e0, e1);
        const double macs = (double)threads * blocks * iters * 16;
        if (rep > 0 && ms > 0.f && macs / (ms * 1e-3) > best) best = macs / (ms * 1e-3);
    }
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    if (sink) cudaFree(sink);
    if (err != cudaSuccess) return carbon::note_cuda(err);
    if (macs_per_s) *macs_per_s = best;
    return CARBON_OK;
}
