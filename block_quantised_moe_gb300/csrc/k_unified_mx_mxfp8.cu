// Instantiations of the single-launch decode forward (unified.cuh) for one
// weight format and activation format.
#include "unified.cuh"

namespace bqmoe {
BQMOE_UNIFIED_LAUNCHER(launch_unified_mx_mxfp8, W_MXFP4, A_MXFP8)
}  // namespace bqmoe
