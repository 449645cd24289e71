// Kernel launch with programmatic dependent launch (PDL).
//
// Every kernel of a forward is launched with programmatic stream
// serialisation: it may start while its predecessor is still running.
// Protocol (all kernels of this library follow it):
//   * a kernel calls pdl_trigger() on entry and pdl_wait() before it reads any
//     output of an earlier kernel; every thread that did not wait waits before
//     it exits, so a kernel's completion implies its predecessor's;
//   * routing triggers early only where its successor waits before reading:
//     the rank launch (followed by the scatter), and, with BF16 x, the launch
//     followed by the register-dequant GEMM1, which then waits before it
//     triggers (so it has passed its wait, and routing has completed, before
//     any later kernel starts);
//   * routing outputs (the expert lists, offsets, sorted pairs, pair_pos) are
//     therefore complete when any kernel after GEMM1 starts, and when any
//     kernel after a routing launch that did not trigger early starts; those
//     kernels may read them before waiting.
#pragma once

#include <cuda_runtime.h>

namespace bqmoe {

// Kernels this host thread has enqueued (read and reset around each forward).
int &launch_counter();

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  ++launch_counter();
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The same with a thread-block cluster of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, int cluster_x,
                                      cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  ++launch_counter();
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace bqmoe
