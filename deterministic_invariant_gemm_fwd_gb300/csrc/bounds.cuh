// bounds.cuh - the bounds-checked debug build of the library.
//
// Built with -DCARBON_DEBUG_BOUNDS (build.py builds it as a second library,
// libcarbon_gemm_bounds.so, beside the regular one), every global-memory
// access of the kernels that index memory themselves is first checked
// against the extent of the buffer it falls in: a workspace array, an operand
// or an output.  An access out of range is skipped and the kernel's device
// status word records CARBON_ERR_OUT_OF_BOUNDS, which
// carbon_get_device_status() reports.  This stands in for a memory checker
// on a GPU where none can run.  (TMA copies need no check: the hardware clips
// them to the tensor map's extent.)  In the regular build the checks compile
// to nothing.
#pragma once

#include <stdint.h>

#include "../../include/carbon_gemm.h"

namespace carbon {

#ifdef CARBON_DEBUG_BOUNDS
constexpr bool kBoundsChecked = true;
#else
constexpr bool kBoundsChecked = false;
#endif

// True when elements [idx, idx + len) lie inside [0, n).  In the checked
// build a false result records CARBON_ERR_OUT_OF_BOUNDS in *status.
__device__ __forceinline__ bool in_bounds(unsigned int *status, int64_t idx, int64_t len, int64_t n) {
    if constexpr (!kBoundsChecked) {
        return true;
    } else {
        if (idx >= 0 && len >= 0 && idx <= n - len) return true;
        atomicExch(status, (unsigned int)CARBON_ERR_OUT_OF_BOUNDS);
        return false;
    }
}

}  // namespace carbon
