// Device helpers for FP4 -> FP16 dequantisation into tensor-core operands and
// for staging activation rows as FP16 with a per-row power-of-two factor.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace bqmoe {

// Four bytes of E2M1 pairs -> four f16x2 (byte j -> r[j], low nibble in the low half).
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&r)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(w));
}

// Four E4M3 bytes -> two f16x2: bytes (0,1) -> lo, bytes (2,3) -> hi, first byte in the low half.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
  asm("{\n\t.reg .b16 h0, h1;\n\t"
      "mov.b32 {h0, h1}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, h0;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h1;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
  return *reinterpret_cast<uint32_t *>(&r);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Power-of-two factor for staging a row with largest magnitude `amax` in FP16:
// amax / f lands in [2^14, 2^15).
__device__ __forceinline__ float stage_factor(float amax) {
  if (!(amax > 0.f)) return 1.f;
  int k = floor_log2_f32(amax) - 14;
  k = max(-126, min(127, k));
  return exp2i_f32(k);
}

// Eight activation values (k % 8 == 0) of a quantised / FP32 row as FP32.
template <int SRC>
__device__ __forceinline__ void src_load8(const void *act, const uint8_t *act_scales, int64_t rid, int k, int K,
                                          float (&v)[8]) {
  if (SRC == SRC_X_BF16) {
    const uint4 r = *reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(act) + rid * K + k);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  } else if (SRC == SRC_H_F32) {
    const float4 p = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(act) + rid * K + k);
    const float4 q = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(act) + rid * K + k + 4);
    v[0] = p.x; v[1] = p.y; v[2] = p.z; v[3] = p.w; v[4] = q.x; v[5] = q.y; v[6] = q.z; v[7] = q.w;
  } else if (SRC == SRC_X_NVFP4 || SRC == SRC_H_NVFP4) {
    // E2M1 * E4M3 only (exact in FP16); the row's FP32 global becomes the factor.
    const uint32_t w = *reinterpret_cast<const uint32_t *>(reinterpret_cast<const uint8_t *>(act) + rid * (K / 2) + k / 2);
    float f[8];
    e2m1x8_to_f32(w, f);
    const float s = e4m3_to_f32(act_scales[rid * (K / 16) + k / 16]);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = f[i] * s;
  } else {  // MXFP8
    const uint2 w = *reinterpret_cast<const uint2 *>(reinterpret_cast<const uint8_t *>(act) + rid * K + k);
    const float s = e8m0_to_f32(act_scales[rid * (K / 32) + k / 32]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[i] = e4m3_to_f32((w.x >> (8 * i)) & 0xFFu) * s;
      v[4 + i] = e4m3_to_f32((w.y >> (8 * i)) & 0xFFu) * s;
    }
  }
}

__device__ __forceinline__ uint4 to_half8(const float (&v)[8], float inv) {
  __align__(16) __half2 h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(v[2 * i] * inv, v[2 * i + 1] * inv);
  return *reinterpret_cast<uint4 *>(h);
}

// FP16 activation rows for the NVFP4 tensor-core kernels are stored in "slot
// order", the K order in which the packer pairs weight codes: inside every
// 64-element K step, the 16 k-slots of mma i (i = 0..3) hold elements
// 8 * (i & 1) + m (m = 0..7) of the step's 16-element scale blocks 2 * (i >> 1)
// (even slots 2m) and 2 * (i >> 1) + 1 (odd slots 2m + 1).  Slot group
// g = 4 * step + i covers row positions [16g, 16g + 16); slot_group_k(g) is the
// natural K offset of its even-slot elements (the odd-slot ones sit 16 further).
__device__ __forceinline__ int slot_group_k(int g) { return 64 * (g >> 2) + 32 * ((g >> 1) & 1) + 8 * (g & 1); }

// Natural elements lo = [k, k + 8) and hi = [k + 16, k + 24) of a slot group,
// times inv, as its 16 FP16 (or BF16) slots (interleaved lo / hi).
template <bool BF16OUT>
__device__ __forceinline__ void to_16bit_slots(const float (&lo)[8], const float (&hi)[8], float inv, uint4 &o0,
                                               uint4 &o1) {
  __align__(16) uint32_t h[8];
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    if (BF16OUT) {
      __nv_bfloat162 b = __floats2bfloat162_rn(lo[m] * inv, hi[m] * inv);
      h[m] = *reinterpret_cast<uint32_t *>(&b);
    } else {
      __half2 f = __floats2half2_rn(lo[m] * inv, hi[m] * inv);
      h[m] = *reinterpret_cast<uint32_t *>(&f);
    }
  }
  o0 = make_uint4(h[0], h[1], h[2], h[3]);
  o1 = make_uint4(h[4], h[5], h[6], h[7]);
}

// Row `rid` of a source as FP16 (or BF16) slot-ordered values times inv,
// written to dst (K 16-bit values); lanes 0..nl-1 of the calling group share
// the work.
template <int SRC, bool BF16OUT = false>
__device__ __forceinline__ void stage_row_slots(const void *act, const uint8_t *act_scales, int64_t rid, int K,
                                                float inv, __half *dst, int lane, int nl) {
  for (int g = lane; g < K / 16; g += nl) {
    const int k = slot_group_k(g);
    float lo[8], hi[8];
    src_load8<SRC>(act, act_scales, rid, k, K, lo);
    src_load8<SRC>(act, act_scales, rid, k + 16, K, hi);
    uint4 o0, o1;
    to_16bit_slots<BF16OUT>(lo, hi, inv, o0, o1);
    reinterpret_cast<uint4 *>(dst + 16 * g)[0] = o0;
    reinterpret_cast<uint4 *>(dst + 16 * g)[1] = o1;
  }
}

// The CTA-pair kernel's K order: within every 64-element step the 32
// slot-ordered pairs (32-bit words) are transposed as a 4 x 8 matrix: pair
// 4 (w & 7) + (w >> 3) of the slot order is pair w of the row.  A warp converts
// eight steps at a time through shared memory: `sbuf` holds them in the slot
// order with a row stride of 36 words (so that both the 16-byte writes and the
// transposing 4-byte reads are free of bank conflicts); each lane then writes one
// 16-byte chunk of the reordered steps per round, the warp's chunks contiguous.
constexpr int kPairStride = 36;  // words per staged step in shared memory
__device__ __forceinline__ void pair_order_flush(const uint32_t *sbuf, uint4 *dst, int nsteps, int lane) {
  for (int c = lane; c < 8 * nsteps; c += 32) {
    const int st = c >> 3, i = c & 7;
    const uint32_t *src = sbuf + st * kPairStride + 16 * (i & 1) + (i >> 1);  // pairs 4t + (i >> 1) (+ 16)
    dst[c] = make_uint4(src[0], src[4], src[8], src[12]);
  }
}

// Row `rid` of a source as 16-bit values times inv in the CTA-pair kernel's K
// order, written to dst by the 32 lanes of a warp; sbuf: 8 x kPairStride words
// of shared memory private to the warp.
template <int SRC, bool BF16OUT = false>
__device__ __forceinline__ void stage_row_pair_order(const void *act, const uint8_t *act_scales, int64_t rid, int K,
                                                     float inv, __half *dst, uint32_t *sbuf, int lane) {
  for (int st0 = 0; st0 < K / 64; st0 += 8) {
    const int ns = min(8, K / 64 - st0);
    // slot-order groups of 16 values, one per lane (4 per step)
    if (lane < 4 * ns) {
      const int g = 4 * st0 + lane;
      const int k = slot_group_k(g);
      float lo[8], hi[8];
      src_load8<SRC>(act, act_scales, rid, k, K, lo);
      src_load8<SRC>(act, act_scales, rid, k + 16, K, hi);
      uint4 o0, o1;
      to_16bit_slots<BF16OUT>(lo, hi, inv, o0, o1);
      uint4 *sb = reinterpret_cast<uint4 *>(sbuf + (lane >> 2) * kPairStride + 8 * (lane & 3));
      sb[0] = o0;
      sb[1] = o1;
    }
    __syncwarp();
    pair_order_flush(sbuf, reinterpret_cast<uint4 *>(dst + 64 * st0), ns, lane);
    __syncwarp();
  }
}

// The same, two slot groups per lane at a time with both groups' loads issued
// before either is stored (a store to shared memory may alias the source, so
// the compiler would otherwise keep each group's loads behind the previous
// group's stores): half the dependent round trips to L2 for a row.
template <int SRC>
__device__ __forceinline__ void stage_row_slots_x2(const void *act, const uint8_t *act_scales, int64_t rid, int K,
                                                   float inv, __half *dst, int lane, int nl) {
  const int ng = K / 16;
  for (int g0 = lane; g0 < ng; g0 += 2 * nl) {
    const int g1 = g0 + nl;
    const bool two = g1 < ng;
    float lo0[8], hi0[8], lo1[8], hi1[8];
    src_load8<SRC>(act, act_scales, rid, slot_group_k(g0), K, lo0);
    src_load8<SRC>(act, act_scales, rid, slot_group_k(g0) + 16, K, hi0);
    if (two) {
      src_load8<SRC>(act, act_scales, rid, slot_group_k(g1), K, lo1);
      src_load8<SRC>(act, act_scales, rid, slot_group_k(g1) + 16, K, hi1);
    }
    uint4 o0, o1;
    to_16bit_slots<false>(lo0, hi0, inv, o0, o1);
    reinterpret_cast<uint4 *>(dst + 16 * g0)[0] = o0;
    reinterpret_cast<uint4 *>(dst + 16 * g0)[1] = o1;
    if (two) {
      to_16bit_slots<false>(lo1, hi1, inv, o0, o1);
      reinterpret_cast<uint4 *>(dst + 16 * g1)[0] = o0;
      reinterpret_cast<uint4 *>(dst + 16 * g1)[1] = o1;
    }
  }
}

}  // namespace bqmoe
