// Instantiations of the single-launch decode forward (unified.cuh) for one
// weight format and activation format.
#include "unified.cuh"

namespace bqmoe {
BQMOE_UNIFIED_LAUNCHER(launch_unified_nv_nvfp4, W_NVFP4, A_NVFP4)
}  // namespace bqmoe
