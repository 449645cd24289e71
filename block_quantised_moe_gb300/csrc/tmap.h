// Tensor-memory-access (TMA) descriptors for the tensor-core kernels.
//
// A kernel that loads a 2-D tile with cp.async.bulk.tensor needs a 128-byte
// CUtensorMap describing the global tensor.  The descriptor is encoded on the
// host with the driver's cuTensorMapEncodeTiled, reached through the runtime's
// driver entry point (the library does not link the driver API), and passed to
// the kernel as a __grid_constant__ parameter.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace bqmoe {

// Rows of 16-bit elements [rows][cols] (row pitch cols * 2 bytes, a multiple
// of 16), loaded as boxes of box_rows x 64 elements (128 bytes) with the
// 128-byte swizzle: the K-major layout the tcgen05 shared-memory descriptors
// expect.  Rows past `rows` read as zeros.  `base` must be 16-byte aligned.
cudaError_t encode_rows16_sw128(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows);

}  // namespace bqmoe
