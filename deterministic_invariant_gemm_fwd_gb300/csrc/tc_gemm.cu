// tc_gemm.cu - tensor-core tier: bf16 x bf16 -> fp32 on tcgen05, accumulator
// in tensor memory, operands staged by TMA, fixed K schedule.
//
// What is computed (sgemm-bi page, "Determinism contracts", tensor-core
// tier: fp32-accumulated bf16 products, bit-identical across runs, forward
// batch-invariant across M, shape-only dispatch): out = A.B (+ bias, fwd) in
// fp32, rounded once to bf16 (RNE).
//
// Determinism and batch invariance by construction:
//  * the output tile is always 128 rows x BN columns; BN (128, 192 or 256)
//    depends on the output column count and the pass only; rows past M are
//    zero-filled by TMA and their
//    results dropped, so row i's instruction sequence is the same for every M;
//  * each tile's reduction runs its k-blocks of 64 in ascending order, four
//    K=16 MMAs per block in ascending order, into one TMEM accumulator; the
//    forward and dX reductions are never split; no atomics are used;
//  * tile-to-CTA scheduling depends on M, the arithmetic of a row does not.
//
// Kernels.
//  tc_gemm_kernel (fwd, dX, and dW when its tile count fills the GPU): one CTA
//  per SM, persistent over output tiles.
//   warp 0     TMA producer: fills a ring of shared-memory stages (A 128x64,
//              B BNx64 bf16, 128-byte swizzle), mbarrier transaction counts
//   warp 1     MMA issuer: allocates TMEM (two accumulators of BN columns),
//              issues tcgen05.mma per stage, commits stage release and tile
//              completion to mbarriers
//   warps 2-5  epilogue: tcgen05.ld of their 32-lane quarter of the
//              accumulator, bias from a shared-memory copy, one RNE rounding to
//              bf16, 32x32 sub-tiles written to swizzled shared memory and
//              stored by TMA; while they drain one accumulator the MMA warp
//              fills the other.
//  tc_dw_split_kernel (dW with few output tiles): the token (reduction) range
//  is cut into s contiguous pieces of whole k-blocks, s depending only on the
//  output tile count; the s CTAs of a thread-block cluster each reduce one
//  piece of the same tile, park their fp32 partial in shared memory, and the
//  partials are added in piece order (0, 1, ..., s-1) through distributed
//  shared memory; each CTA rounds and stores 128/s rows.  No atomics, so the
//  result is the same on every run.
// Every mbarrier wait is bounded (device_sync.cuh); a wait that gives up
// records CARBON_ERR_TIMEOUT, raises a CTA-wide abort flag so the other roles
// leave their loops, and the TMEM allocation is still released.
#include "carbon_internal.h"
#include "bounds.cuh"
#include "device_sync.cuh"
#include "tcgen05.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

namespace carbon {
namespace {

__device__ unsigned int g_tc_status = 0;
#define CHK(idx, len, n) in_bounds(&g_tc_status, (int64_t)(idx), (int64_t)(len), (int64_t)(n))

constexpr int kBM = 128;          // tile rows (= MMA M, = TMEM lanes)
constexpr int kBK = 64;           // k-block: 64 bf16 = one 128-byte swizzle row
constexpr int kUMMA_K = 16;       // K of one tcgen05.mma kind::f16
// Ring stages per tile width: as many as the shared memory holds beside the
// staging and bias copies (the kernel waits on operand arrival more than on
// anything else: releasing stages in pairs, which shortens the look-ahead by
// a stage, made the tier 12% slower).
template <int BN>
constexpr int stages_for() { return BN >= 256 ? 4 : (BN >= 192 ? 5 : 6); }
constexpr int kThreads = 192;     // 6 warps
constexpr int kMaxSplits = 8;     // dW token split: pieces per cluster, at most
constexpr int kEpiWarps = 4;
constexpr uint32_t kABytes = kBM * kBK * 2;           // 16 KiB
constexpr uint32_t kMNBlockBytes = 64 * kBK * 2;      // one 64-wide MN block of an MN-major tile

enum Major { K_MAJOR = 0, MN_MAJOR = 1 };

struct TcArgs {
    void *out;
    const void *bias;         // bf16 [cols] or null (fwd only)
    int64_t rows, cols, R;
    int tiles_m, tiles_n, num_kb;
    int splits, kb_per_split; // dW cluster split (tc_dw_split_kernel only)
};

template <int BN>
struct Smem {
    static constexpr int kStages = stages_for<BN>();
    static constexpr uint32_t kBBytes = BN * kBK * 2;
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kPipeBytes = kStages * kStageBytes;
    // epilogue staging: per epilogue warp two 32x32 bf16 sub-tiles (2 KiB each)
    static constexpr uint32_t kStagingOffset = kPipeBytes;
    static constexpr uint32_t kStagingBytes = kEpiWarps * 2 * 2048;
    static constexpr uint32_t kBiasOffset = kStagingOffset + kStagingBytes;
    static constexpr uint32_t kBarOffset = kBiasOffset + kEpiWarps * BN * 4;   // per-warp bias copy
    // full[S], empty[S], tfull[2], tempty[2], then tmem base slot and abort flag
    static constexpr uint32_t kBytes = kBarOffset + (2 * kStages + 4) * 8 + 16;
    static constexpr uint32_t kDynamic = kBytes + 1024;   // room to align the base to 1 KiB
    static_assert(kDynamic <= 232448, "shared memory per block");
    // split kernel: fp32 partial tile [128][BN + 4] placed over the pipeline ring
    static constexpr uint32_t kPartialPitch = BN + 4;
    static_assert(kBM * kPartialPitch * 4 <= kPipeBytes, "partial tile must fit the ring");
};

// The kernels' operand and output types: bf16 operands and output, bf16
// operands with the fp32 accumulator stored (inspection path), fp16
// operands and output.
enum OutType { OT_BF16 = 0, OT_F32 = 1, OT_F16 = 2 };

// Instruction descriptor, kind::f16: fp32 accumulate, A and B both bf16 or
// both fp16 (one format field value for both, so they can never differ),
// majorness of A and B, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t instr_desc(int bn, int a_major, int b_major, bool f16) {
    return (1u << 4) | ((f16 ? 0u : 1u) << 7) | ((f16 ? 0u : 1u) << 10) | ((uint32_t)a_major << 15) |
           ((uint32_t)b_major << 16) | ((uint32_t)(bn >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
}

// Descriptor of the K=16 slice `k` (0..3) of a 64-deep k-block tile whose
// MN extent is `mn` (rows of a K-major tile, or 64-wide blocks of an MN-major one).
template <int MAJOR>
__device__ __forceinline__ uint64_t operand_desc(uint32_t tile_base, int k) {
    if (MAJOR == K_MAJOR)   // rows of 128 B; 8-row atoms 1024 B apart; K slice = +32 B
        return smem_desc(tile_base + (uint32_t)k * (kUMMA_K * 2), 16, 1024);
    // MN-major: rows are k (128 B = 64 MN elements); 8-k groups 1024 B apart (SBO);
    // 64-wide MN blocks kMNBlockBytes apart (LBO); K slice = 16 rows = +2048 B
    return smem_desc(tile_base + (uint32_t)k * (kUMMA_K * 128), kMNBlockBytes, 1024);
}

__device__ __forceinline__ bool aborted(volatile uint32_t *flag) { return *flag != 0; }

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile uint32_t *flag) {
    if (mbar_wait(bar, parity)) return true;
    *flag = 1u;
    atomicExch(&g_tc_status, (unsigned)CARBON_ERR_TIMEOUT);
    return false;
}

// ---- more PTX wrappers: TMA store, bulk groups, proxies, clusters -----------

__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
                 ::"l"(map), "r"(src), "r"(c0), "r"(c1) : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most one committed bulk group still reads shared memory.
__device__ __forceinline__ void bulk_wait_read_1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Make generic-proxy shared-memory writes visible to the async proxy (TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                 ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t local_addr, uint32_t rank) {
    uint32_t remote;
    float4 v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(remote) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);     // RNE, one rounding each
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);                 // RNE, one rounding each
    return *reinterpret_cast<uint32_t *>(&h);
}

// Two fp32 values rounded to the output type and packed (bf16 or fp16).
template <int OT>
__device__ __forceinline__ uint32_t pack_out(float lo, float hi) {
    return OT == OT_F16 ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi);
}

// A 16-bit bias element of the operand type, widened to fp32 (exactly).
template <int OT>
__device__ __forceinline__ float bias_value(const void *bias, int64_t j) {
    const unsigned short h = static_cast<const unsigned short *>(bias)[j];
    return OT == OT_F16 ? __half2float(__ushort_as_half(h)) : __uint_as_float((uint32_t)h << 16);
}

// ---- the roles shared by both kernels -----------------------------------------

struct Bars {
    uint32_t full0, empty0, tfull0, tempty0;
    __device__ uint32_t full(int s) const { return full0 + 8u * s; }
    __device__ uint32_t empty(int s) const { return empty0 + 8u * s; }
    __device__ uint32_t tfull(int b) const { return tfull0 + 8u * b; }
    __device__ uint32_t tempty(int b) const { return tempty0 + 8u * b; }
};

// Producer: k-blocks [kb0, kb1) of the tile at (m0, n0) into the ring.
template <int BN, int A_MAJOR, int B_MAJOR>
__device__ __forceinline__ bool produce_tile(const CUtensorMap *ma, const CUtensorMap *mb,
                                             uint32_t sbase, const Bars &bar, int m0, int n0,
                                             int kb0, int kb1, int &s, uint32_t &ph,
                                             volatile uint32_t *abort_flag) {
    using L = Smem<BN>;
    for (int kb = kb0; kb < kb1; ++kb) {
        if (!wait_or_abort(bar.empty(s), ph ^ 1u, abort_flag)) return false;
        mbar_arrive_expect_tx(bar.full(s), L::kStageBytes);
        const uint32_t sa = sbase + s * L::kStageBytes, sb = sa + kABytes;
        const int k0 = kb * kBK;
        if (A_MAJOR == K_MAJOR) {
            tma_load_2d(sa, ma, bar.full(s), k0, m0);
        } else {
            tma_load_2d(sa, ma, bar.full(s), m0, k0);
            tma_load_2d(sa + kMNBlockBytes, ma, bar.full(s), m0 + 64, k0);
        }
        if (B_MAJOR == K_MAJOR) {
            tma_load_2d(sb, mb, bar.full(s), k0, n0);
        } else {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
                tma_load_2d(sb + j * kMNBlockBytes, mb, bar.full(s), n0 + 64 * j, k0);
        }
        if (++s == L::kStages) { s = 0; ph ^= 1u; }
    }
    return true;
}

// Lets every load the producer issued land before the CTA may exit: a stage
// armed in the last pass completes with parity ph; stages not armed in it
// completed earlier, so their wait returns at once.
template <int BN>
__device__ __forceinline__ void drain_producer(const Bars &bar, int s, uint32_t ph) {
    constexpr int kStages = Smem<BN>::kStages;
    for (int i = 0; i < kStages; ++i) {
        if (--s < 0) { s = kStages - 1; ph ^= 1u; }
        if (!mbar_wait(bar.full(s), ph)) break;
    }
}

// MMA issuer: nkb k-blocks from the ring into the accumulator at TMEM column d.
template <int BN, int A_MAJOR, int B_MAJOR, bool F16>
__device__ __forceinline__ bool mma_tile(uint32_t d, uint32_t sbase, const Bars &bar, int nkb,
                                         int &s, uint32_t &ph, volatile uint32_t *abort_flag) {
    using L = Smem<BN>;
    constexpr uint32_t idesc = instr_desc(BN, A_MAJOR, B_MAJOR, F16);
    for (int kb = 0; kb < nkb; ++kb) {
        if (!wait_or_abort(bar.full(s), ph, abort_flag)) return false;
        tc_fence_after();
        const uint32_t sa = sbase + s * L::kStageBytes, sb = sa + kABytes;
#pragma unroll
        for (int k = 0; k < kBK / kUMMA_K; ++k)
            mma_bf16(d, operand_desc<A_MAJOR>(sa, k), operand_desc<B_MAJOR>(sb, k), idesc,
                     (kb | k) != 0 ? 1u : 0u);
        mma_commit(bar.empty(s));                  // stage free once these MMAs finish
        if (++s == L::kStages) { s = 0; ph ^= 1u; }
    }
    return true;
}

// Sets up barriers and TMEM; returns the TMEM base column address.
template <int BN>
__device__ __forceinline__ uint32_t setup_cta(uint8_t *smem, const Bars &bar,
                                              const CUtensorMap *ma, const CUtensorMap *mb,
                                              uint32_t *tmem_slot, volatile uint32_t *abort_flag,
                                              uint32_t tmem_cols) {
    const int warp = threadIdx.x / 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < Smem<BN>::kStages; ++s) {
            mbar_init(bar.full(s), 1);
            mbar_init(bar.empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar.tfull(b), 1);
            mbar_init(bar.tempty(b), kEpiWarps);
        }
        *abort_flag = 0u;
        fence_mbar_init();
        prefetch_map(ma);
        prefetch_map(mb);
    }
    if (warp == 1) tmem_alloc(smem_addr(tmem_slot), tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // set-up done: wait for the previous kernel on the stream (its outputs
    // may be this GEMM's operands) and let the next one be scheduled
    wait_prior_grid();
    allow_next_grid();
    return *tmem_slot;
}

// ---- persistent kernel (fwd, dX, dW without split) ----------------------------

template <int BN, int A_MAJOR, int B_MAJOR, int OT>
__global__ void __launch_bounds__(kThreads, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
               const __grid_constant__ CUtensorMap map_out, const TcArgs p) {
    using L = Smem<BN>;
    constexpr bool OUT_F32 = OT == OT_F32;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    Bars bar;
    bar.full0 = sbase + L::kBarOffset;
    bar.empty0 = bar.full0 + 8 * L::kStages;
    bar.tfull0 = bar.empty0 + 8 * L::kStages;
    bar.tempty0 = bar.tfull0 + 16;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kBarOffset + (2 * L::kStages + 4) * 8);
    volatile uint32_t *abort_flag = tmem_slot + 1;
    constexpr uint32_t kTmemCols = BN == 128 ? 256u : 512u;   // two accumulators, rounded to a power of two

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t tmem_base = setup_cta<BN>(smem, bar, &map_a, &map_b, tmem_slot, abort_flag, kTmemCols);
    const int num_tiles = p.tiles_m * p.tiles_n;

    if (warp == 0) {
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            for (int t = blockIdx.x; t < num_tiles && !aborted(abort_flag); t += gridDim.x)
                if (!produce_tile<BN, A_MAJOR, B_MAJOR>(&map_a, &map_b, sbase, bar,
                                                        (t / p.tiles_n) * kBM, (t % p.tiles_n) * BN,
                                                        0, p.num_kb, s, ph, abort_flag))
                    break;
            drain_producer<BN>(bar, s, ph);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int s = 0, acc = 0;
            uint32_t ph = 0, aph = 0;
            for (int t = blockIdx.x; t < num_tiles && !aborted(abort_flag); t += gridDim.x) {
                if (!wait_or_abort(bar.tempty(acc), aph ^ 1u, abort_flag)) break;
                tc_fence_after();
                if (!mma_tile<BN, A_MAJOR, B_MAJOR, OT == OT_F16>(tmem_base + (uint32_t)(acc * BN), sbase,
                                                                  bar, p.num_kb, s, ph, abort_flag))
                    break;
                mma_commit(bar.tfull(acc));            // accumulator ready
                if (++acc == 2) { acc = 0; aph ^= 1u; }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - 2;                         // 0..3
        const int quarter = warp % 4;                    // TMEM lanes 32*quarter .. +31
        const uint32_t stg = sbase + L::kStagingOffset + ew * 4096;
        float *bias_s = reinterpret_cast<float *>(smem + L::kBiasOffset) + ew * BN;
        const void *bias = p.bias;
        int acc = 0, nstores = 0;
        uint32_t aph = 0;
        for (int t = blockIdx.x; t < num_tiles && !aborted(abort_flag); t += gridDim.x) {
            const int m0 = (t / p.tiles_n) * kBM;
            const int n0 = (t % p.tiles_n) * BN;
            if (bias) {                                   // this warp's copy of the tile's bias
                __syncwarp();                             // the previous tile's reads are done
                for (int i = lane; i < BN; i += 32)
                    bias_s[i] = (n0 + i < p.cols && CHK(n0 + i, 1, p.cols)) ? bias_value<OT>(bias, n0 + i) : 0.0f;
                __syncwarp();
            }
            if (!wait_or_abort(bar.tfull(acc), aph, abort_flag)) break;
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                if (n0 + c >= p.cols) break;             // whole chunk past the last column
                uint32_t v[32];
                tmem_ld32(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN + c), v);
                float f[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
                if (bias) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        const float4 b4 = *reinterpret_cast<const float4 *>(bias_s + c + i);
                        f[i] = __fadd_rn(f[i], b4.x);
                        f[i + 1] = __fadd_rn(f[i + 1], b4.y);
                        f[i + 2] = __fadd_rn(f[i + 2], b4.z);
                        f[i + 3] = __fadd_rn(f[i + 3], b4.w);
                    }
                }
                if (OUT_F32) {                           // inspection path: direct fp32 stores
                    const int64_t row = (int64_t)m0 + quarter * 32 + lane;
                    if (row < p.rows) {
                        float *o = static_cast<float *>(p.out) + row * p.cols + n0 + c;
#pragma unroll
                        for (int g = 0; g < 8; ++g)
                            if (n0 + c + 4 * g < p.cols &&
                                CHK(row * p.cols + n0 + c + 4 * g, 4, (int64_t)p.rows * p.cols))
                                *reinterpret_cast<float4 *>(o + 4 * g) =
                                    make_float4(f[4 * g], f[4 * g + 1], f[4 * g + 2], f[4 * g + 3]);
                    }
                } else {
                    // 32 rows x 64 bytes, 16-byte pieces swizzled as TMA's 64-byte mode
                    // expects (piece index ^= (row >> 1) & 3): conflict-free v4 stores.
                    const uint32_t buf = stg + (uint32_t)(nstores & 1) * 2048u;
                    if (nstores >= 2 && lane == 0) bulk_wait_read_1();
                    __syncwarp();
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        uint4 w;
                        w.x = pack_out<OT>(f[8 * g + 0], f[8 * g + 1]);
                        w.y = pack_out<OT>(f[8 * g + 2], f[8 * g + 3]);
                        w.z = pack_out<OT>(f[8 * g + 4], f[8 * g + 5]);
                        w.w = pack_out<OT>(f[8 * g + 6], f[8 * g + 7]);
                        st_shared_v4(buf + lane * 64 + 16 * (g ^ ((lane >> 1) & 3)), w);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&map_out, buf, n0 + c, m0 + quarter * 32);   // clipped at rows/cols
                        bulk_commit();
                    }
                    ++nstores;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar.tempty(acc));
            if (++acc == 2) { acc = 0; aph ^= 1u; }
        }
        if (!OUT_F32 && lane == 0) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---- dW with few tiles: token range split over a cluster --------------------

// Rows [piece * 128/S, (piece + 1) * 128/S) of the tile: the S fp32 partials
// parked in the cluster's shared memory, added in piece order 0, 1, ..., S-1,
// rounded once and stored.  A thread takes U = 16/S four-column vectors per
// round and issues all of the round's 16 remote loads before its first
// addition (a remote load's latency is many times a round's arithmetic).
template <int S, int BN, int OT>
__device__ __forceinline__ void combine_pieces(const TcArgs &p, uint32_t part_addr, int piece, int m0,
                                               int n0) {
    using L = Smem<BN>;
    static_assert(S >= 2 && S <= kMaxSplits && kBM % S == 0, "split count");
    constexpr int U = 16 / S, rows_per = kBM / S, vec_per_row = BN / 4, nvec = rows_per * vec_per_row;
    const int r0 = piece * rows_per;
    for (int first = threadIdx.x; first < nvec; first += U * kThreads) {
        float4 b[U][S];
        uint32_t live = 0u;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int idx = first + u * kThreads;
            const int rr = r0 + idx / vec_per_row, cc = (idx % vec_per_row) * 4;
            const int64_t grow = (int64_t)m0 + rr, gcol = (int64_t)n0 + cc;
            if (idx < nvec && grow < p.rows && gcol < p.cols &&
                CHK(grow * p.cols + gcol, 4, (int64_t)p.rows * p.cols)) {
                live |= 1u << u;
                const uint32_t off = part_addr + (uint32_t)(rr * L::kPartialPitch + cc) * 4u;
#pragma unroll
                for (int q = 0; q < S; ++q) b[u][q] = ld_cluster_f4(off, (uint32_t)q);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (!((live >> u) & 1u)) continue;
            const int idx = first + u * kThreads;
            const int64_t grow = (int64_t)m0 + r0 + idx / vec_per_row, gcol = (int64_t)n0 + (idx % vec_per_row) * 4;
            float4 a = b[u][0];
#pragma unroll
            for (int q = 1; q < S; ++q) {
                a.x = __fadd_rn(a.x, b[u][q].x);
                a.y = __fadd_rn(a.y, b[u][q].y);
                a.z = __fadd_rn(a.z, b[u][q].z);
                a.w = __fadd_rn(a.w, b[u][q].w);
            }
            if (OT == OT_F32) {
                *reinterpret_cast<float4 *>(static_cast<float *>(p.out) + grow * p.cols + gcol) = a;
            } else {
                uint2 w;
                w.x = pack_out<OT>(a.x, a.y);
                w.y = pack_out<OT>(a.z, a.w);
                *reinterpret_cast<uint2 *>(static_cast<unsigned short *>(p.out) + grow * p.cols + gcol) = w;
            }
        }
    }
}


template <int BN, int OT>
__global__ void __launch_bounds__(kThreads, 1)
tc_dw_split_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   const TcArgs p) {
    using L = Smem<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    Bars bar;
    bar.full0 = sbase + L::kBarOffset;
    bar.empty0 = bar.full0 + 8 * L::kStages;
    bar.tfull0 = bar.empty0 + 8 * L::kStages;
    bar.tempty0 = bar.tfull0 + 16;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kBarOffset + (2 * L::kStages + 4) * 8);
    volatile uint32_t *abort_flag = tmem_slot + 1;
    // one accumulator of BN columns, the allocation rounded up to a power of two
    constexpr uint32_t kTmemCols = BN <= 128 ? 128u : 256u;
    static_assert(BN <= 256, "one accumulator per CTA");

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t tmem_base = setup_cta<BN>(smem, bar, &map_a, &map_b, tmem_slot, abort_flag, kTmemCols);

    const int piece = (int)cluster_rank();                 // == blockIdx.x
    const int t = blockIdx.y;
    const int m0 = (t / p.tiles_n) * kBM, n0 = (t % p.tiles_n) * BN;
    const int kb0 = piece * p.kb_per_split;
    const int kb1 = min(p.num_kb, kb0 + p.kb_per_split);
    const int nkb = kb1 > kb0 ? kb1 - kb0 : 0;
    float *part = reinterpret_cast<float *>(smem);          // [128][BN + 4] over the ring

    if (warp == 0) {
        if (lane == 0 && nkb > 0) {
            int s = 0;
            uint32_t ph = 0;
            produce_tile<BN, MN_MAJOR, MN_MAJOR>(&map_a, &map_b, sbase, bar, m0, n0, kb0, kb1, s, ph,
                                                 abort_flag);
            drain_producer<BN>(bar, s, ph);
        }
    } else if (warp == 1) {
        if (lane == 0 && nkb > 0) {
            int s = 0;
            uint32_t ph = 0;
            if (mma_tile<BN, MN_MAJOR, MN_MAJOR, OT == OT_F16>(tmem_base, sbase, bar, nkb, s, ph, abort_flag))
                mma_commit(bar.tfull(0));
        }
    } else {
        const int quarter = warp % 4;
        const int row = quarter * 32 + lane;
        bool have = nkb > 0;
        if (have) {
            have = wait_or_abort(bar.tfull(0), 0, abort_flag);
            tc_fence_after();
        }
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
            uint32_t v[32];
            if (have) tmem_ld32(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c, v);
            float *dst = part + row * L::kPartialPitch + c;
#pragma unroll
            for (int i = 0; i < 32; i += 4)
                *reinterpret_cast<float4 *>(dst + i) =
                    have ? make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                       __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();                                    // every partial is parked

    // piece r rounds and stores rows [r*128/s, (r+1)*128/s) of the tile,
    // adding the partials in piece order 0, 1, ..., s-1
    const uint32_t part_addr = smem_addr(part);
    switch (p.splits) {
    case 2: combine_pieces<2, BN, OT>(p, part_addr, piece, m0, n0); break;
    case 4: combine_pieces<4, BN, OT>(p, part_addr, piece, m0, n0); break;
    case 8: combine_pieces<8, BN, OT>(p, part_addr, piece, m0, n0); break;
    default: break;                                        // the host splits in 2, 4 or 8 only
    }
    cluster_sync_all();                                    // peers are done reading this CTA
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// Fills an output whose reduction is empty: bias (fwd) or +0.
template <int OT>
__global__ void tc_fill_kernel(void *out, const void *bias, int64_t rows, int64_t cols) {
    wait_prior_grid();
    allow_next_grid();
    const int64_t n = rows * cols;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float v = (bias && CHK(i % cols, 1, cols)) ? bias_value<OT>(bias, i % cols) : 0.0f;
        if (OT == OT_F32) static_cast<float *>(out)[i] = v;
        else static_cast<unsigned short *>(out)[i] = (unsigned short)(pack_out<OT>(v, 0.0f) & 0xffffu);
    }
}

// ---- host side ----------------------------------------------------------------

// 2-D tensor map of 16-bit elements (bf16, also used for fp16 data: the
// copies move bytes, and the fill of 0x0000 is +0 in both formats) over a
// row-major [outer, inner] matrix with a {box_inner, box_outer} box;
// out-of-range elements read as 0 and are not written by stores.
bool encode_map(CUtensorMap *map, const void *base, int64_t inner, int64_t outer, int box_inner,
                int box_outer, CUtensorMapSwizzle swizzle) {
    return encode_tensor_map_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, (uint64_t)inner,
                                (uint64_t)outer, (uint64_t)inner * 2, (uint32_t)box_inner,
                                (uint32_t)box_outer, swizzle) == cudaSuccess;
}

bool encode_operand(CUtensorMap *map, const void *base, int64_t inner, int64_t outer, int box_outer) {
    return encode_map(map, base, inner, outer, 64, box_outer, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <typename Kern>
cudaError_t prepare(Kern kern, int smem) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

template <int BN, int AM, int BM_, int OT>
cudaError_t launch_persistent(const CUtensorMap &ma, const CUtensorMap &mb, const CUtensorMap &mo,
                              const TcArgs &a, int grid, cudaStream_t stream) {
    auto kern = tc_gemm_kernel<BN, AM, BM_, OT>;
    const int smem = (int)Smem<BN>::kDynamic;
    cudaError_t err = prepare(kern, smem);
    if (err != cudaSuccess) return err;
    return launch_k(kern, dim3(grid), dim3(kThreads), (size_t)smem, stream, 1, ma, mb, mo, a);
}

template <int BN, int OT>
cudaError_t launch_persistent_pass(int pass, const CUtensorMap &ma, const CUtensorMap &mb,
                                   const CUtensorMap &mo, const TcArgs &a, int grid, cudaStream_t s) {
    switch (pass) {
    case CARBON_PASS_FWD: return launch_persistent<BN, K_MAJOR, MN_MAJOR, OT>(ma, mb, mo, a, grid, s);
    case CARBON_PASS_DX:  return launch_persistent<BN, K_MAJOR, K_MAJOR, OT>(ma, mb, mo, a, grid, s);
    default:              return launch_persistent<BN, MN_MAJOR, MN_MAJOR, OT>(ma, mb, mo, a, grid, s);
    }
}

template <int OT>
cudaError_t launch_persistent_bn(int bn, int pass, const CUtensorMap &ma, const CUtensorMap &mb,
                                 const CUtensorMap &mo, const TcArgs &a, int grid, cudaStream_t s) {
    if (bn == 128) return launch_persistent_pass<128, OT>(pass, ma, mb, mo, a, grid, s);
    if (bn == 192) return launch_persistent_pass<192, OT>(pass, ma, mb, mo, a, grid, s);
    return launch_persistent_pass<256, OT>(pass, ma, mb, mo, a, grid, s);
}

template <int BN, int OT>
cudaError_t launch_split(const CUtensorMap &ma, const CUtensorMap &mb, const TcArgs &a,
                         cudaStream_t stream) {
    auto kern = tc_dw_split_kernel<BN, OT>;
    const int smem = (int)Smem<BN>::kDynamic;
    cudaError_t err = prepare(kern, smem);
    if (err != cudaSuccess) return err;
    return launch_k(kern, dim3((unsigned)a.splits, (unsigned)(a.tiles_m * a.tiles_n), 1), dim3(kThreads),
                    (size_t)smem, stream, (unsigned)a.splits, ma, mb, a);
}

// Clusters of s CTAs that run at once on GB300 (152 SMs in 8 GPCs of about
// 19, and a cluster's CTAs share one GPC): 16 of 8, 32 of 4, 72 of 2.  (18
// clusters of 8 ran as two waves: dW of 768 x 768 took 26 us for 12 us of
// work per CTA.)
int clusters_at_once(int s) { return s >= 8 ? 16 : s == 4 ? 32 : s == 2 ? 72 : 152; }

// dW split count from the output tile count only: the largest s in
// {1, 2, 4, 8} whose tiles * s CTAs run in one wave on GB300 (SM count and
// GPC layout fixed here, so the bits do not depend on the device a run
// lands on).
int choose_splits(int64_t tiles) {
    int s = 1;
    while (s < kMaxSplits && tiles * (2 * s) <= 152 && tiles <= clusters_at_once(2 * s)) s *= 2;
    return s;
}

// Output tile width.  Forward and dX: from the column count and the pass only
// (never the row count, so a row's tiles, and its bits, do not depend on the
// batch): 128 for at most 128 columns; otherwise 256, or 192 when that fills
// the SMs better for a reference batch of 8192 rows on 152 SMs (768 columns:
// 256 tiles of 192 run in two fuller waves than 192 tiles of 256).  dW (rows
// and columns both weight dimensions): 256, or 192 when that gives each CTA
// less work for a reference reduction of 8192 tokens (work per CTA = width x
// k-blocks per piece x waves), e.g. 768 x 2304: 72 tiles of 192 in two pieces
// fill 144 SMs where 54 tiles of 256 fill 108.  The width does not change a
// dW output's summation: its pieces and their k-block order depend on the
// split count alone, and 192 is chosen only where that count is the same.
double wave_fill(int64_t tiles) {
    const int64_t waves = (tiles + 151) / 152;
    return (double)tiles / (double)(waves * 152);
}

int choose_bn(int64_t rows, int64_t cols, int pass) {
    if (cols <= 128) return 128;
    if (pass == CARBON_PASS_DW) {
        const int64_t tiles_m = (rows + kBM - 1) / kBM, ref_kb = 8192 / kBK;
        auto work = [&](int64_t bn) {
            const int64_t tiles = tiles_m * ((cols + bn - 1) / bn);
            const int s = choose_splits(tiles);
            const int64_t waves = s > 1 ? 1 : (tiles + 151) / 152;
            return bn * ((ref_kb + s - 1) / s) * waves;
        };
        const int64_t tiles192 = tiles_m * ((cols + 191) / 192), tiles256 = tiles_m * ((cols + 255) / 256);
        const bool same_split = choose_splits(tiles192) == choose_splits(tiles256);
        return (same_split && work(192) < work(256)) ? 192 : 256;
    }
    const int64_t ref_tiles_m = 8192 / kBM;
    const double f256 = wave_fill(ref_tiles_m * ((cols + 255) / 256));
    const double f192 = wave_fill(ref_tiles_m * ((cols + 191) / 192));
    return f192 > f256 ? 192 : 256;
}

}  // namespace

carbon_status_t tc_launch(const Problem &p, bool out_f32, cudaStream_t stream) {
    if (p.rows == 0 || p.cols == 0) return CARBON_OK;
    // 16-byte aligned bases and row pitches (K and N multiples of 8 bf16)
    if ((p.K % 8) != 0 || (p.N % 8) != 0) return CARBON_ERR_MISALIGNED;
    auto mis = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) != 0; };
    if (mis(p.A) || mis(p.B) || mis(p.out) || (p.bias && (reinterpret_cast<uintptr_t>(p.bias) & 1u)))
        return CARBON_ERR_MISALIGNED;
    int dev = 0, sms = 0;
    carbon_status_t st = current_device(&dev, &sms);
    if (st != CARBON_OK) return st;

    if (p.R == 0) {
        const int64_t n = p.rows * p.cols;
        const int blocks = (int)((n + 255) / 256 < 65535 ? (n + 255) / 256 : 65535);
        const dim3 g((unsigned)blocks), b(256);
        cudaError_t ferr;
        if (out_f32) ferr = launch_k(tc_fill_kernel<OT_F32>, g, b, 0, stream, 1, p.out, p.bias, p.rows, p.cols);
        else if (p.dtype == CARBON_F16) ferr = launch_k(tc_fill_kernel<OT_F16>, g, b, 0, stream, 1, p.out, p.bias, p.rows, p.cols);
        else ferr = launch_k(tc_fill_kernel<OT_BF16>, g, b, 0, stream, 1, p.out, p.bias, p.rows, p.cols);
        count_launch();
        return note_cuda(ferr);
    }
    if (p.rows > (int64_t)0x7fffffff || p.cols > (int64_t)0x7fffffff || p.R > (int64_t)0x7fffffff)
        return CARBON_ERR_INVALID_ARG;

    cudaError_t err = cudaSuccess;

    const int bn = choose_bn(p.rows, p.cols, p.pass);
    CUtensorMap ma, mb, mo;
    bool ok;
    switch (p.pass) {
    case CARBON_PASS_FWD:   // A = X [M, K] K-major; B = W [K, N] N-contiguous (MN-major)
        ok = encode_operand(&ma, p.A, p.K, p.M, kBM) && encode_operand(&mb, p.B, p.N, p.K, 64);
        break;
    case CARBON_PASS_DX:    // A = dY [M, N] K-major; B = W [K, N]: rows = out cols, K-major
        ok = encode_operand(&ma, p.A, p.N, p.M, kBM) && encode_operand(&mb, p.B, p.N, p.K, bn);
        break;
    default:                // A = X [M, K] and B = dY [M, N], both MN-major
        ok = encode_operand(&ma, p.A, p.K, p.M, 64) && encode_operand(&mb, p.B, p.N, p.M, 64);
        break;
    }
    // output [rows, cols] bf16, 32x32 boxes, 64-byte swizzle (epilogue staging layout)
    ok = ok && (out_f32 || encode_map(&mo, p.out, p.cols, p.rows, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B));
    if (!ok) return CARBON_ERR_MISALIGNED;
    if (out_f32) mo = ma;                                // unused by the fp32 inspection path

    TcArgs a;
    a.out = p.out; a.bias = p.bias;
    a.rows = p.rows; a.cols = p.cols; a.R = p.R;
    a.tiles_m = (int)((p.rows + kBM - 1) / kBM);
    a.tiles_n = (int)((p.cols + bn - 1) / bn);
    a.num_kb = (int)((p.R + kBK - 1) / kBK);
    a.splits = 1;
    a.kb_per_split = a.num_kb;
    const int64_t tiles = (int64_t)a.tiles_m * a.tiles_n;
    if (tiles > 65535) {
        if (tiles > (int64_t)0x7fffffff) return CARBON_ERR_INVALID_ARG;
    }

    if (p.pass == CARBON_PASS_DW) {
        a.splits = choose_splits(tiles);
        if (a.splits > a.num_kb) a.splits = 1;
        a.kb_per_split = (a.num_kb + a.splits - 1) / a.splits;
    }
    // operand / output type: the fp32 inspection path takes bf16 operands
    const int ot = out_f32 ? OT_F32 : (p.dtype == CARBON_F16 ? OT_F16 : OT_BF16);
    if (a.splits > 1) {
        if (bn == 128)
            err = ot == OT_F32 ? launch_split<128, OT_F32>(ma, mb, a, stream)
                : ot == OT_F16 ? launch_split<128, OT_F16>(ma, mb, a, stream)
                               : launch_split<128, OT_BF16>(ma, mb, a, stream);
        else if (bn == 192)
            err = ot == OT_F32 ? launch_split<192, OT_F32>(ma, mb, a, stream)
                : ot == OT_F16 ? launch_split<192, OT_F16>(ma, mb, a, stream)
                               : launch_split<192, OT_BF16>(ma, mb, a, stream);
        else
            err = ot == OT_F32 ? launch_split<256, OT_F32>(ma, mb, a, stream)
                : ot == OT_F16 ? launch_split<256, OT_F16>(ma, mb, a, stream)
                               : launch_split<256, OT_BF16>(ma, mb, a, stream);
    } else {
        const int grid = (int)(tiles < sms ? tiles : sms);
        err = ot == OT_F32 ? launch_persistent_bn<OT_F32>(bn, p.pass, ma, mb, mo, a, grid, stream)
            : ot == OT_F16 ? launch_persistent_bn<OT_F16>(bn, p.pass, ma, mb, mo, a, grid, stream)
                           : launch_persistent_bn<OT_BF16>(bn, p.pass, ma, mb, mo, a, grid, stream);
    }
    count_launch();
    return note_cuda(err);
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

cudaError_t get_encoder() {
    std::call_once(g_encode_once, [] {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                        cudaEnableDefault, &q);
        if (g_encode_err == cudaSuccess && q != cudaDriverEntryPointSuccess)
            g_encode_err = cudaErrorNotSupported;
        if (g_encode_err == cudaSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode_err;
}

}  // namespace

cudaError_t encode_tensor_map_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base,
                                 uint64_t inner, uint64_t outer, uint64_t row_bytes,
                                 uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
    const cudaError_t err = get_encoder();
    if (err != cudaSuccess) return err;
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = g_encode(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

carbon_status_t tc_take_device_status() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_status, sizeof v) != cudaSuccess) return CARBON_OK;
    if (v != 0) cudaMemcpyToSymbol(g_tc_status, &zero, sizeof zero);
    return (carbon_status_t)v;
}

}  // namespace carbon
