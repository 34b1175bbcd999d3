// superacc.cu - the correctly rounded tier computed one output per warp:
// every product added exactly into a fixed-point accumulator (superacc.cuh),
// the bias too, and the total rounded once to the output type.  The result is
// the exact dot product plus the bias, rounded once; no order of the
// reduction shows in it (Carbon README, "Roadmap": superaccumulators).
//
// Serves two uses:
//  * the whole tier for fp32 and fp16 operands (and for bf16 outputs too large
//    for the tensor-core path's 32-bit output lists);
//  * the fix-up of the bf16 tensor-core path (exact_tc.cu), for the outputs it
//    lists: inf/NaN operands, lines too wide for its integer grain, sums that
//    leave its 64-bit range.
//
// A warp takes an output, its lanes stride over the reduction index (lane l
// takes r = l, l + 32, ...) adding into their own accumulators in registers,
// then the 32 accumulators are summed digit by digit with shuffles (integer
// additions: exact) and lane 0 rounds.
#include "carbon_internal.h"
#include "bounds.cuh"
#include "device_sync.cuh"
#include "superacc.cuh"

namespace carbon {
namespace {

constexpr int kSaWarps = 8;

// Status word: CARBON_ERR_OUT_OF_BOUNDS in the bounds-checked build.
__device__ unsigned int g_superacc_status = 0;
#define CHK(idx, len, n) in_bounds(&g_superacc_status, (int64_t)(idx), (int64_t)(len), (int64_t)(n))

struct SaArgs {
    const void *A, *B, *bias;
    void *out;
    int64_t rows, cols, R;
    int64_t a_si, a_sr, b_sr, b_sj;
};

template <int DT>
__device__ __forceinline__ uint32_t load_bits(const void *base, int64_t idx) {
    if (DT == CARBON_F32) return __ldg(static_cast<const uint32_t *>(base) + idx);
    return (uint32_t)__ldg(static_cast<const unsigned short *>(base) + idx);
}

template <int DT>
__device__ __forceinline__ void store_bits(void *base, int64_t idx, uint32_t v) {
    if (DT == CARBON_F32) static_cast<uint32_t *>(base)[idx] = v;
    else static_cast<unsigned short *>(base)[idx] = (unsigned short)v;
}

// LIST: outputs work_list[0 .. *work_count) (row-major indices), else all.
template <int DT, bool LIST>
__global__ void __launch_bounds__(kSaWarps * 32)
superacc_kernel(const SaArgs p, const unsigned int *__restrict__ work_count,
                const unsigned int *__restrict__ work_list) {
    wait_prior_grid();
    allow_next_grid();
    const int lane = threadIdx.x % 32;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
    const int64_t nw = (int64_t)gridDim.x * blockDim.x / 32;
    const int64_t count = LIST ? (int64_t)*work_count : p.rows * p.cols;
    const int64_t n_a = (p.rows > 0 && p.R > 0) ? (p.rows - 1) * p.a_si + (p.R - 1) * p.a_sr + 1 : 0;
    const int64_t n_b = (p.cols > 0 && p.R > 0) ? (p.R - 1) * p.b_sr + (p.cols - 1) * p.b_sj + 1 : 0;
    for (int64_t item = gw; item < count; item += nw) {
        const int64_t o = LIST ? (int64_t)work_list[item] : item;
        const int64_t i = o / p.cols, j = o % p.cols;
        if (!CHK(o, 1, p.rows * p.cols)) continue;             // warp-uniform
        long long acc[sacc::kDigits];
#pragma unroll
        for (int d = 0; d < sacc::kDigits; ++d) acc[d] = 0ll;
        int cls = sacc::kFinite;
        uint32_t steps = 0;
        // kUnroll reduction indices per lane and step, their loads issued
        // first (the operand reads are strided: their latency bounds the loop)
        constexpr int kUnroll = 4;
        for (int64_t r0 = lane; r0 < p.R; r0 += 32 * kUnroll) {
            if ((++steps & 0x3ffffu) == 0u) sacc::carry(acc);   // digits stay below 2^53
            uint32_t ha[kUnroll], hb[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t r = r0 + 32 * u;
                const bool in = r < p.R && CHK(i * p.a_si + r * p.a_sr, 1, n_a) &&
                                CHK(r * p.b_sr + j * p.b_sj, 1, n_b);
                ha[u] = in ? load_bits<DT>(p.A, i * p.a_si + r * p.a_sr) : 0u;
                hb[u] = in ? load_bits<DT>(p.B, r * p.b_sr + j * p.b_sj) : 0u;
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                long long ma, mb;
                int ea, eb, ca, cb;
                sacc::decode_value<DT>(ha[u], ma, ea, ca);           // 0 bits: +0, adds nothing
                sacc::decode_value<DT>(hb[u], mb, eb, cb);
                const int pc = sacc::product_class(ca, ma, cb, mb);
                if (pc != sacc::kFinite) { cls |= pc; continue; }
                if (ma != 0 && mb != 0) sacc::add_scaled(acc, ma * mb, ea + eb + sacc::kOff);
            }
        }
        if (p.bias != nullptr && lane == 0) {
            long long mb;
            int eb, cb;
            sacc::decode_value<DT>(load_bits<DT>(p.bias, j), mb, eb, cb);
            if (cb != sacc::kFinite) cls |= cb;
            else if (mb != 0) sacc::add_scaled(acc, mb, eb + sacc::kOff);
        }
        // the lanes' accumulators summed exactly (a lane's digits stay below
        // 2^53: a carry pass every 2^20 additions of values below 2^32)
#pragma unroll
        for (int d = 0; d < sacc::kDigits; ++d)
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc[d] += __shfl_xor_sync(0xffffffffu, acc[d], off);
        cls = (int)__reduce_or_sync(0xffffffffu, (unsigned)cls);
        if (lane == 0) store_bits<DT>(p.out, o, sacc::round_acc<DT>(acc, cls));
    }
}

SaArgs make_args(const Problem &p) {
    SaArgs a;
    a.A = p.A; a.B = p.B; a.bias = p.bias; a.out = p.out;
    a.rows = p.rows; a.cols = p.cols; a.R = p.R;
    switch (p.pass) {
    case CARBON_PASS_FWD: a.a_si = p.K; a.a_sr = 1; a.b_sr = p.N; a.b_sj = 1; break;
    case CARBON_PASS_DX:  a.a_si = p.N; a.a_sr = 1; a.b_sr = 1;   a.b_sj = p.N; break;
    default:              a.a_si = 1;   a.a_sr = p.K; a.b_sr = p.N; a.b_sj = 1; break;
    }
    return a;
}

template <bool LIST>
cudaError_t launch(int dtype, const SaArgs &a, int blocks, const unsigned int *count,
                   const unsigned int *list, cudaStream_t s) {
    const dim3 g((unsigned)blocks), b(kSaWarps * 32);
    cudaError_t err;
    switch (dtype) {
    case CARBON_F32: err = launch_k(superacc_kernel<CARBON_F32, LIST>, g, b, 0, s, 1, a, count, list); break;
    case CARBON_F16: err = launch_k(superacc_kernel<CARBON_F16, LIST>, g, b, 0, s, 1, a, count, list); break;
    default:         err = launch_k(superacc_kernel<CARBON_BF16, LIST>, g, b, 0, s, 1, a, count, list); break;
    }
    count_launch();
    return err;
}

}  // namespace

carbon_status_t superacc_launch(const Problem &p, cudaStream_t stream) {
    if (p.rows == 0 || p.cols == 0) return CARBON_OK;
    int sms = 0;
    carbon_status_t st = current_device(nullptr, &sms);
    if (st != CARBON_OK) return st;
    const int64_t outs = p.rows * p.cols;
    const int64_t want = (outs + kSaWarps - 1) / kSaWarps;
    const int64_t cap = (int64_t)sms * 16;
    const int blocks = (int)(want < cap ? want : cap);
    return note_cuda(launch<false>(p.dtype, make_args(p), blocks, nullptr, nullptr, stream));
}

cudaError_t superacc_fixup_bf16(const Problem &p, const unsigned int *work_count,
                                const unsigned int *work_list, int blocks, cudaStream_t stream) {
    return launch<true>(CARBON_BF16, make_args(p), blocks, work_count, work_list, stream);
}

carbon_status_t superacc_take_device_status() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_superacc_status, sizeof v) != cudaSuccess) return CARBON_OK;
    if (v != 0) cudaMemcpyToSymbol(g_superacc_status, &zero, sizeof zero);
    return (carbon_status_t)v;
}

}  // namespace carbon
