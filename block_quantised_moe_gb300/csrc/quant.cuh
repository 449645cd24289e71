// Block-quantiser arithmetic shared by the quantiser kernels and the
// single-launch decode forward (see k_quant.cu for the formulas).
#pragma once

#include "common.cuh"

namespace bqmoe {

template <bool BF16>
__device__ __forceinline__ void load8(const void *src, int64_t idx, float (&v)[8]) {
  if (BF16) {
    const uint4 r = *reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(src) + idx);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  } else {
    const float4 a = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(src) + idx);
    const float4 b = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(src) + idx + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

// One NVFP4 block of 16 with global g -> 8 code bytes (uint2) and the scale byte.
__device__ __forceinline__ void nvfp4_block(const float (&x)[16], float g, uint2 &codes, uint32_t &scale) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  scale = 0;
  float d = 0.f;
  if (g > 0.f) {
    scale = f32_to_e4m3(__fdiv_rn(__fdiv_rn(amax, 6.0f), g));
    d = __fmul_rn(e4m3_to_f32(scale), g);
  }
  if (d > 0.f) {
    float a[8], b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      a[i] = __fdiv_rn(x[i], d);
      b[i] = __fdiv_rn(x[8 + i], d);
    }
    codes = make_uint2(f32x8_to_e2m1x8(a), f32x8_to_e2m1x8(b));
  } else {
    codes = make_uint2(0u, 0u);
  }
}

// One MX block of 32 -> codes (16 bytes for E2M1, 32 for E4M3) and the E8M0 byte.
template <int QF>
__device__ __forceinline__ void mx_block(const float (&x)[32], uint32_t (&codes)[8], uint32_t &scale) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
  constexpr int emax = (QF == Q_MXFP8) ? 8 : 2;
  int X = amax > 0.f ? floor_log2_f32(amax) - emax : -127;
  X = max(-127, min(127, X));
  scale = (uint32_t)(X + 127);
  const float p2 = exp2i_f32(X);
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __fdiv_rn(x[i], p2);
  if (QF == Q_MXFP8) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      codes[i] = f32x2_to_e4m3x2(v[4 * i], v[4 * i + 1]) | (f32x2_to_e4m3x2(v[4 * i + 2], v[4 * i + 3]) << 16);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float w[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) w[j] = v[8 * i + j];
      codes[i] = f32x8_to_e2m1x8(w);
    }
  }
}

}  // namespace bqmoe
