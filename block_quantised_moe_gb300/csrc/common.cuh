// Device helpers shared by the kernels of libmoe: format decoders and the
// sm_100-family conversion instructions (cvt to / from E2M1 and E4M3 pairs).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace bqmoe {

// Weight / activation / activation-function codes (mirror include/moe.h).
enum { W_NVFP4 = 1, W_MXFP4 = 2 };
enum { A_BF16 = 1, A_NVFP4 = 2, A_MXFP8 = 3 };
enum { ACT_SILU = 1, ACT_RELU2 = 2 };
enum { Q_NVFP4 = 1, Q_MXFP4 = 2, Q_MXFP8 = 3 };

// Device status word layout (int32 x 4 at the start of scratch).
enum { ST_FLAGS = 0, ST_DROPPED = 1 };
enum { ST_FLAG_DROPPED = 1, ST_FLAG_TIMEOUT = 2 };

// ----------------------------------------------------------------- decode

// E4M3FN byte -> float, exact: sign, 4-bit exponent (bias 7), 3-bit mantissa;
// exponent 0 is subnormal (m * 2^-9); 0x7F / 0xFF are NaN.
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  const uint32_t e = (b >> 3) & 0xFu, m = b & 7u;
  float v = (e == 0) ? (float)m * 0.001953125f : __uint_as_float(((e + 120u) << 23) | (m << 20));
  if ((b & 0x7Fu) == 0x7Fu) v = __uint_as_float(0x7FC00000u);
  return (b & 0x80u) ? -v : v;
}

// E8M0 byte -> float 2^(b-127), exact (b = 0 is the FP32 subnormal 2^-127); 0xFF is NaN.
__device__ __forceinline__ float e8m0_to_f32(uint32_t b) {
  if (b == 0) return __uint_as_float(0x00400000u);
  if (b == 0xFFu) return __uint_as_float(0x7FC00000u);
  return __uint_as_float(b << 23);
}

// Four bytes of packed E2M1 pairs -> four half2, each holding (low nibble, high nibble).
__device__ __forceinline__ void e2m1x8_to_half2x4(uint32_t w, __half2 (&h)[4]) {
  uint32_t r0, r1, r2, r3;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(w));
  h[0] = *reinterpret_cast<__half2 *>(&r0);
  h[1] = *reinterpret_cast<__half2 *>(&r1);
  h[2] = *reinterpret_cast<__half2 *>(&r2);
  h[3] = *reinterpret_cast<__half2 *>(&r3);
}

// Eight E2M1 codes (one 32-bit word, element 2j in the low nibble of byte j) -> floats.
__device__ __forceinline__ void e2m1x8_to_f32(uint32_t w, float (&v)[8]) {
  __half2 h[4];
  e2m1x8_to_half2x4(w, h);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __half22float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

// ----------------------------------------------------------------- encode

// Eight floats -> eight E2M1 codes in one word (element 2j in the low nibble of
// byte j), round-to-nearest-even, saturating at +-6.  cvt packs its first
// source operand into the high nibble of the byte.
__device__ __forceinline__ uint32_t f32x8_to_e2m1x8(const float (&v)[8]) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// Two floats -> two E4M3 bytes (lo in bits 0..7), RNE, saturating to +-448.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t f32_to_e4m3(float v) { return f32x2_to_e4m3x2(v, 0.f) & 0xFFu; }

// Exact floor(log2(a)) for finite a > 0, subnormals included.
__device__ __forceinline__ int floor_log2_f32(float a) {
  const uint32_t u = __float_as_uint(a);
  const int e = (int)((u >> 23) & 0xFFu);
  if (e != 0) return e - 127;
  return (31 - __clz(u & 0x7FFFFFu)) - 149;  // subnormal: mantissa * 2^-149
}

// 2^X as a float for X in [-127, 127] (2^-127 is a subnormal).
__device__ __forceinline__ float exp2i_f32(int X) {
  return X >= -126 ? __uint_as_float((uint32_t)(X + 127) << 23) : __uint_as_float(0x00400000u);
}

// ------------------------------------------------- programmatic dependent launch

// Let the next kernel in the stream start launching (see launch.h for the protocol).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// Wait until the preceding kernel has completed and its writes are visible.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// --------------------------------------------------------------- misc

// SiLU(a) = a * sigmoid(a), with the hardware exponential and approximate
// division (relative error ~1e-6, far inside the output tolerance); large
// negative a gives exp(-a) = inf and a zero sigmoid.
__device__ __forceinline__ float silu_f32(float a) { return a * __fdividef(1.0f, 1.0f + __expf(-a)); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__host__ __device__ __forceinline__ int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ __forceinline__ int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

}  // namespace bqmoe
