// tc_gemm.cu - tensor-core tier (placeholder until the tcgen05 kernel lands).
#include "carbon_internal.h"

namespace carbon {
namespace {
__device__ unsigned int g_tc_status = 0;
}

carbon_status_t tc_launch(const Problem &, bool, cudaStream_t) { return CARBON_ERR_UNSUPPORTED; }

carbon_status_t tc_take_device_status() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_status, sizeof v) != cudaSuccess) return CARBON_OK;
    if (v != 0) cudaMemcpyToSymbol(g_tc_status, &zero, sizeof zero);
    return (carbon_status_t)v;
}

}  // namespace carbon
