// Activation rows as 16-bit tensor-core operands.
//
// The tensor-core kernels read activations as FP16 rows in slot order with a
// per-row power-of-two factor (NVFP4 weights: E2M1 x E4M3 is exact in FP16, and
// the factor keeps every BF16 activation exact), or as BF16 rows with factor 1
// (MXFP4 weights: E2M1 x 2^X is exact only in BF16).  This file turns GEMM1's
// output h (FP32 or its re-quantised codes) and the MXFP4 path's x into such
// rows.
#include <algorithm>

#include "common.cuh"
#include "dequant.cuh"
#include "internal.h"
#include "launch.h"

namespace bqmoe {

// ------------------------------------------------ h -> FP16 rows for the tc path
//
// One warp per live slot row: FP32 h with the factor from GEMM1's per-pair max |h|,
// NVFP4 (E2M1*E4M3 exact, factor = row global) or MXFP8 (two passes) -> FP16 + factor.
// With PAIR the rows are written in the CTA-pair kernel's K order (h rows, which
// only that kernel reads); without, in the slot order (the MXFP4 path's x rows,
// which the slot-order gather reorders).
template <int SRC, bool OUT_BF16, bool PAIR>
__global__ void __launch_bounds__(256) k_stage_h16(const void *__restrict__ act, const uint8_t *__restrict__ act_scales,
                                                   const float *__restrict__ act_g, int K, int64_t rows,
                                                   const int32_t *__restrict__ rows_dev, __half *__restrict__ h16,
                                                   float *__restrict__ fac) {
  const int lane = threadIdx.x & 31;
  __shared__ __align__(16) uint32_t sbuf_all[8][8 * kPairStride];  // per warp, for the pair order
  uint32_t *sbuf = sbuf_all[threadIdx.x >> 5];
  pdl_trigger();
  pdl_wait();
  const int64_t live = rows_dev == nullptr || rows < (int64_t)*rows_dev ? rows : (int64_t)*rows_dev;
  for (int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); row < live; row += (int64_t)gridDim.x * 8) {
    if (OUT_BF16) {  // BF16 rows, no factor (the MXFP4 path's BF16 operands)
      if (PAIR) stage_row_pair_order<SRC, true>(act, act_scales, row, K, 1.f, h16 + row * K, sbuf, lane);
      else stage_row_slots<SRC, true>(act, act_scales, row, K, 1.f, h16 + row * K, lane, 32);
      continue;
    }
    float f;
    if (SRC == SRC_H_NVFP4) {
      f = act_g[row];
    } else if (SRC == SRC_H_F32) {
      f = stage_factor(act_g[row]);
    } else {
      float mx = 0.f;
      for (int k = lane * 8; k < K; k += 256) {
        float v[8];
        src_load8<SRC>(act, act_scales, row, k, K, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) mx = fmaxf(mx, fabsf(v[i]));
      }
      f = stage_factor(warp_max(mx));
    }
    const float inv = SRC == SRC_H_NVFP4 ? 1.f : __frcp_rn(f);
    if (PAIR) stage_row_pair_order<SRC>(act, act_scales, row, K, inv, h16 + row * K, sbuf, lane);
    else stage_row_slots<SRC>(act, act_scales, row, K, inv, h16 + row * K, lane, 32);
    if (lane == 0) fac[row] = f;
  }
}

template <bool PAIR>
static cudaError_t launch_stage_h16_t(int src, const void *act, const uint8_t *act_scales, const float *act_g, int K,
                                      int64_t rows, const int32_t *rows_dev, __half *h16, float *fac, bool out_bf16,
                                      cudaStream_t s) {
  const int grid = (int)std::min<int64_t>((rows + 7) / 8, 152 * 16);
#define SH(S, B) \
  return launch_pdl(k_stage_h16<S, B, PAIR>, dim3(grid), dim3(256), 0, s, act, act_scales, act_g, K, rows, rows_dev, h16, fac)
  if (out_bf16) {
    switch (src) {
      case SRC_X_BF16: SH(SRC_X_BF16, true);
      case SRC_H_F32: SH(SRC_H_F32, true);
      case SRC_H_MXFP8: SH(SRC_H_MXFP8, true);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (src) {
    case SRC_H_F32: SH(SRC_H_F32, false);
    case SRC_H_NVFP4: SH(SRC_H_NVFP4, false);
    case SRC_H_MXFP8: SH(SRC_H_MXFP8, false);
    default: return cudaErrorInvalidValue;
  }
#undef SH
}

cudaError_t launch_stage_h16(int src, const void *act, const uint8_t *act_scales, const float *act_g, int K,
                             int64_t rows, const int32_t *rows_dev, __half *h16, float *fac, bool out_bf16,
                             bool pair_order, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (pair_order && K % 64) return cudaErrorInvalidValue;
  return pair_order ? launch_stage_h16_t<true>(src, act, act_scales, act_g, K, rows, rows_dev, h16, fac, out_bf16, s)
                    : launch_stage_h16_t<false>(src, act, act_scales, act_g, K, rows, rows_dev, h16, fac, out_bf16, s);
}

}  // namespace bqmoe
