// Grouped expert contractions on the tensor cores with register-resident
// dequantisation, for NVFP4 weights (any activation format).
//
// moe.fused_moe's "W4A16 (BF16 activations, inline FP4 weight dequant)" and its
// decode path (b12x project page, section "What's in here").  At decode sizes an
// expert sees a handful of tokens, so the layer is bound by streaming the
// touched experts' packed bytes from HBM; the tensor cores only have to keep the
// multiply-adds off the FP32 pipe.  Design:
//
// * The packer stores every 16-row x 64-K tile of E2M1 codes as 32 x 16-byte
//   lanes in mma.m16n8k16 A-fragment order, and its 16 x 4 E4M3 block scales
//   as 8-byte groups (rows r and r+8 interleaved).  A warp streams a tile with
//   one coalesced 128-bit load per lane (plus an 8-byte scale load shared by 4
//   lanes), four tiles ahead of use.
// * Codes become FP16 with cvt.rn.f16x2.e2m1x2 and are multiplied by their E4M3
//   scale in FP16 (the product of an E2M1 and an E4M3 value has at most 6
//   significant bits and lies in [2^-10, 2688]: exact), straight into A
//   fragments: no shared-memory round trip for the weights.
// * Activations (the B operand) are staged once per CTA in shared memory as
//   FP16 with a per-row power-of-two factor f (x = f * x16): the factor puts the
//   row's largest magnitude in [2^14, 2^15), so BF16 values convert exactly
//   except those below 2^-31 of the row's maximum; NVFP4 rows are staged as
//   E2M1*E4M3 (exact) with f = the row's FP32 global scale.  f, the weights'
//   FP32 global scale and, for GEMM2, topk_weight are applied to the FP32
//   accumulator in the epilogue.
// * For gated SiLU a 16-row tile holds 8 gate rows and the same 8 up rows, so
//   each thread owns matching gate / up accumulators and computes SiLU(g) * u
//   in registers.
//
// One CTA = 8 warps = 128 weight rows of one expert; it walks the expert's
// sorted pairs in tiles of 8 * NT tokens.
#include "common.cuh"
#include "internal.h"

namespace bqmoe {

constexpr int kMmaWarps = 8;
constexpr int kMmaThreads = kMmaWarps * 32;
constexpr int kPF = 8;  // 64-K super-steps loaded ahead of use

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x2(uint32_t addr, uint32_t &r0, uint32_t &r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0));
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

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

// ---------------------------------------------------------- x -> FP16 rows
//
// One CTA per token row: x (BF16, or the NVFP4 / MXFP8 codes of the activation
// quantiser) -> x16 [T][K] FP16 and f [T] with x^ = f * x16.  Also clears
// `zero` (the per-pair |h| maxima GEMM1 accumulates) for this forward.
constexpr int kStageThreads = 256;

template <int SRC>
__global__ void __launch_bounds__(kStageThreads)
k_stage_x16(const void *__restrict__ act, const uint8_t *__restrict__ act_scales, const float *__restrict__ act_g,
            int K, __half *__restrict__ x16, float *__restrict__ fac, float *__restrict__ zero, int64_t zero_n) {
  __shared__ float red[32];
  const int64_t row = blockIdx.x;
  for (int64_t i = (int64_t)blockIdx.x * kStageThreads + threadIdx.x; i < zero_n; i += (int64_t)gridDim.x * kStageThreads)
    zero[i] = 0.f;
  constexpr bool nv = SRC == SRC_X_NVFP4;
  float f = 1.f;
  if (nv) {
    f = act_g[row];
  } else {
    float m = 0.f;
    for (int k = threadIdx.x * 8; k < K; k += kStageThreads * 8) {
      float v[8];
      src_load8<SRC>(act, act_scales, row, k, K, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
    }
    m = warp_max(m);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) red[warp] = m;
    __syncthreads();
    m = 0.f;
    for (int w = 0; w < kStageThreads / 32; ++w) m = fmaxf(m, red[w]);
    f = stage_factor(m);
  }
  const float inv = nv ? 1.f : __frcp_rn(f);  // exact: f is a power of two
  for (int k = threadIdx.x * 8; k < K; k += kStageThreads * 8) {
    float v[8];
    src_load8<SRC>(act, act_scales, row, k, K, v);
    *reinterpret_cast<uint4 *>(x16 + row * K + k) = to_half8(v, inv);
  }
  if (threadIdx.x == 0) fac[row] = f;
}

// ------------------------------------------------------------ grouped kernel

template <int SRC, int STAGE, int NT>
__global__ void __launch_bounds__(kMmaThreads, 2) k_grouped_mma(const GroupedArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  constexpr int NTOK = 8 * NT;
  const int K = a.K;
  const int pitch = 2 * K + 16;  // bytes per staged row; +16 keeps ldmatrix conflict-free
  __half *xs = reinterpret_cast<__half *>(smem);
  float *fac = reinterpret_cast<float *>(smem + (size_t)NTOK * pitch);
  int64_t *rows = reinterpret_cast<int64_t *>(fac + NTOK);

  const int e = blockIdx.y;
  const int cnt = a.counts[e];
  if (cnt == 0) return;
  const int off = a.offsets[e];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr bool by_token = SRC == SRC_X16;

  const int tile = blockIdx.x * kMmaWarps + warp;  // 16-row tile of this expert
  const int nsteps = K / 64;
  const uint4 *ctile = reinterpret_cast<const uint4 *>(a.codes + (size_t)e * a.codes_expert) + (size_t)tile * nsteps * 32 + lane;
  const uint2 *stile = reinterpret_cast<const uint2 *>(a.scales + (size_t)e * a.scales_expert) + (size_t)tile * nsteps * 8 + (lane >> 2);
  const float *gl = a.globals + 4 * e;
  const uint32_t xs_base = (uint32_t)__cvta_generic_to_shared(xs);
  // ldmatrix row addresses: lanes 0-7 rows 0-7 at k, 8-15 rows 0-7 at k+8,
  // 16-23 rows 8-15 at k, 24-31 rows 8-15 at k+8.
  const int lrow = (lane & 7) + ((lane >> 4) << 3);
  const uint32_t b_addr = xs_base + lrow * pitch + ((lane >> 3) & 1) * 16;

  for (int s0 = off; s0 < off + cnt; s0 += NTOK) {
    const int ntok = min(NTOK, off + cnt - s0);
    // Weight prefetch first: it does not depend on the activations.
    uint4 cbuf[kPF];
    uint2 sbuf[kPF];
#pragma unroll
    for (int p = 0; p < kPF; ++p) {
      if (p < nsteps) {
        cbuf[p] = __ldg(ctile + (size_t)p * 32);
        sbuf[p] = __ldg(stile + (size_t)p * 8);
      }
    }
    __syncthreads();  // the previous tile's staging buffer is free
    if (threadIdx.x < NTOK) {
      int64_t rid = -1;
      if ((int)threadIdx.x < ntok) {
        const int s = s0 + threadIdx.x;
        rid = by_token ? (int64_t)(a.sorted_pair[s] / a.top_k) : (int64_t)s;
      }
      rows[threadIdx.x] = rid;
    }
    __syncthreads();
    // Stage NTOK activation rows as FP16 (warp w: rows w, w+8, ...).
    for (int j = warp; j < NTOK; j += kMmaWarps) {
      const int64_t rid = rows[j];
      uint8_t *dst = reinterpret_cast<uint8_t *>(xs) + (size_t)j * pitch;
      if (SRC == SRC_X16) {
        const __half *src = reinterpret_cast<const __half *>(a.act) + (rid < 0 ? 0 : rid) * K;
        const uint32_t d0 = (uint32_t)__cvta_generic_to_shared(dst);
        for (int k = lane * 8; k < K; k += 256) cp_async16(d0 + 2 * k, src + k, rid >= 0);
        if (lane == 0) fac[j] = rid < 0 ? 0.f : a.act_g[rid];
        continue;
      }
      if (rid < 0) {
        for (int k = lane * 8; k < K; k += 256) *reinterpret_cast<uint4 *>(dst + 2 * k) = make_uint4(0, 0, 0, 0);
        if (lane == 0) fac[j] = 0.f;
        continue;
      }
      float f;
      if (SRC == SRC_H_NVFP4) {
        f = a.act_g[rid];
      } else if (SRC == SRC_H_F32) {
        f = stage_factor(a.act_g[rid]);  // the |h| maximum GEMM1 recorded for this pair
      } else {
        float m = 0.f;
        for (int k = lane * 8; k < K; k += 256) {
          float v[8];
          src_load8<SRC>(a.act, a.act_scales, rid, k, K, v);
#pragma unroll
          for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
        }
        f = stage_factor(warp_max(m));
      }
      const float inv = SRC == SRC_H_NVFP4 ? 1.f : __frcp_rn(f);
      for (int k = lane * 8; k < K; k += 256) {
        float v[8];
        src_load8<SRC>(a.act, a.act_scales, rid, k, K, v);
        *reinterpret_cast<uint4 *>(dst + 2 * k) = to_half8(v, inv);
      }
      if (lane == 0) fac[j] = f;
    }
    if (SRC == SRC_X16) cp_async_wait_all();
    __syncthreads();

    float acc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

    for (int q = 0; q < nsteps; q += kPF) {
#pragma unroll
      for (int p = 0; p < kPF; ++p) {
        const int qq = q + p;
        if (qq < nsteps) {
          const uint4 c = cbuf[p];
          const uint2 sc = sbuf[p];
          if (qq + kPF < nsteps) {
            cbuf[p] = __ldg(ctile + (size_t)(qq + kPF) * 32);
            sbuf[p] = __ldg(stile + (size_t)(qq + kPF) * 8);
          }
          const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
          uint32_t spairs[4];  // (s_r, s_r8) of k16 block i as f16x2
          e4m3x4_to_f16x2x2(sc.x, spairs[0], spairs[1]);
          e4m3x4_to_f16x2x2(sc.y, spairs[2], spairs[3]);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t s_lo = prmt(spairs[i], 0, 0x1010);  // (s_r, s_r)
            const uint32_t s_hi = prmt(spairs[i], 0, 0x3232);  // (s_r8, s_r8)
            uint32_t af[4];
            e2m1x8_to_f16x2x4(cw[i], af);
            af[0] = hmul2(af[0], s_lo);
            af[1] = hmul2(af[1], s_hi);
            af[2] = hmul2(af[2], s_lo);
            af[3] = hmul2(af[3], s_hi);
            const uint32_t kb = (uint32_t)(qq * 64 + i * 16) * 2;
            if (NT == 2) {
              uint32_t b0, b1, b2, b3;
              ldmatrix_x4(b_addr + kb, b0, b1, b2, b3);
              mma_16816(acc[0], af, b0, b1);
              mma_16816(acc[NT - 1], af, b2, b3);
            } else {
              uint32_t b0, b1;
              ldmatrix_x2(b_addr + kb, b0, b1);
              mma_16816(acc[0], af, b0, b1);
            }
          }
        }
      }
    }

    // Epilogue.  Thread owns rows r = lane/4 and r+8, tokens n = 2*(lane%4) + {0,1} of each n8 tile.
    const int r = lane >> 2;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int n = j * 8 + 2 * (lane & 3) + c;
        const bool live = n < ntok;
        const int s = s0 + n;
        const float f = live ? fac[n] : 0.f;
        const float lo = acc[j][c] * f, hi = acc[j][2 + c] * f;
        float hmax = 0.f;
        if (STAGE == STAGE_GATED) {
          const float h = silu_f32(lo * gl[0]) * (hi * gl[1]);
          if (live) a.out[(size_t)s * a.n_rows + tile * 8 + r] = h;
          hmax = fabsf(h);
        } else if (STAGE == STAGE_RELU2) {
          const float v0 = fmaxf(lo * gl[0], 0.f), v1 = fmaxf(hi * gl[0], 0.f);
          if (live) {
            a.out[(size_t)s * a.n_rows + tile * 16 + r] = v0 * v0;
            a.out[(size_t)s * a.n_rows + tile * 16 + r + 8] = v1 * v1;
          }
          hmax = fmaxf(v0 * v0, v1 * v1);
        } else if (live) {
          const float w = a.topk_weights[a.sorted_pair[s]] * gl[2];
          a.out[(size_t)s * a.n_rows + tile * 16 + r] = w * lo;
          a.out[(size_t)s * a.n_rows + tile * 16 + r + 8] = w * hi;
        }
        if (STAGE != STAGE_DOWN && a.out_amax != nullptr) {
          // max over the 8 lanes holding this token (same lane % 4), then one atomic per warp;
          // a max of non-negative floats is exact and order-free, so the result is deterministic.
          hmax = fmaxf(hmax, __shfl_xor_sync(0xffffffffu, hmax, 4));
          hmax = fmaxf(hmax, __shfl_xor_sync(0xffffffffu, hmax, 8));
          hmax = fmaxf(hmax, __shfl_xor_sync(0xffffffffu, hmax, 16));
          if (live && r == 0) atomicMax(reinterpret_cast<unsigned *>(a.out_amax) + s, __float_as_uint(hmax));
        }
      }
    }
  }
}

size_t mma_smem_bytes(int K, int NT) { return (size_t)8 * NT * (2 * K + 16) + 8 * NT * (4 + 8); }

template <int SRC, int STAGE, int NT>
static cudaError_t launch_mma_one(const GroupedArgs &a, int rows_total, int E, cudaStream_t s) {
  const size_t smem = mma_smem_bytes(a.K, NT);
  cudaError_t err = cudaFuncSetAttribute(k_grouped_mma<SRC, STAGE, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
  if (err != cudaSuccess) return err;
  k_grouped_mma<SRC, STAGE, NT><<<dim3(rows_total / (16 * kMmaWarps), E), kMmaThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <int STAGE, int NT>
static cudaError_t launch_mma_src(int src, const GroupedArgs &a, int rows_total, int E, cudaStream_t s) {
  if (STAGE == STAGE_DOWN) {
    switch (src) {
      case SRC_H_F32: return launch_mma_one<SRC_H_F32, STAGE, NT>(a, rows_total, E, s);
      case SRC_H_NVFP4: return launch_mma_one<SRC_H_NVFP4, STAGE, NT>(a, rows_total, E, s);
      case SRC_H_MXFP8: return launch_mma_one<SRC_H_MXFP8, STAGE, NT>(a, rows_total, E, s);
    }
  } else if (src == SRC_X16) {
    return launch_mma_one<SRC_X16, STAGE, NT>(a, rows_total, E, s);
  }
  return cudaErrorInvalidValue;
}

template <int NT>
static cudaError_t launch_mma_nt(int src, int stage, const GroupedArgs &a, int rows_total, int E, cudaStream_t s) {
  switch (stage) {
    case STAGE_GATED: return launch_mma_src<STAGE_GATED, NT>(src, a, rows_total, E, s);
    case STAGE_RELU2: return launch_mma_src<STAGE_RELU2, NT>(src, a, rows_total, E, s);
    case STAGE_DOWN: return launch_mma_src<STAGE_DOWN, NT>(src, a, rows_total, E, s);
  }
  return cudaErrorInvalidValue;
}

// rows_total: rows of the weight matrix of this stage (2I gated, I for ReLU^2, H down).
cudaError_t launch_grouped_mma(int src, int stage, const GroupedArgs &a, int rows_total, int E, cudaStream_t s) {
  if (rows_total % (16 * kMmaWarps) != 0 || a.K % 64 != 0) return cudaErrorInvalidValue;
  // Two n8 token tiles per pass when their staging fits comfortably, else one.
  if (mma_smem_bytes(a.K, 2) <= 100 * 1024) return launch_mma_nt<2>(src, stage, a, rows_total, E, s);
  if (mma_smem_bytes(a.K, 1) <= 200 * 1024) return launch_mma_nt<1>(src, stage, a, rows_total, E, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_stage_x16(int src, const void *act, const uint8_t *act_scales, const float *act_g, int T, int K,
                             __half *x16, float *fac, float *zero, int64_t zero_n, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  switch (src) {
    case SRC_X_BF16:
      k_stage_x16<SRC_X_BF16><<<T, kStageThreads, 0, s>>>(act, act_scales, act_g, K, x16, fac, zero, zero_n);
      break;
    case SRC_X_NVFP4:
      k_stage_x16<SRC_X_NVFP4><<<T, kStageThreads, 0, s>>>(act, act_scales, act_g, K, x16, fac, zero, zero_n);
      break;
    case SRC_X_MXFP8:
      k_stage_x16<SRC_X_MXFP8><<<T, kStageThreads, 0, s>>>(act, act_scales, act_g, K, x16, fac, zero, zero_n);
      break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace bqmoe
