// Grouped expert contractions on CUDA cores (FP32), for every weight and
// activation format: GEMM1 + activation (gated SiLU or ReLU^2) and GEMM2 scaled
// by topk_weights.  The op is moe.fused_moe (b12x project page, section "What's
// in here": "inline FP4 weight dequant"; vLLM docs "b12x Linear and MoE
// Backends", section "ModelOpt block codecs": bias-free SiLU or non-gated ReLU^2).
//
// One CTA = one expert x 32 weight rows; it walks the expert's sorted pairs in
// tiles of 8.  Per 512-wide K chunk the 8 activation rows are staged in shared
// memory as FP32 (dequantised on the way in for NVFP4 / MXFP8 sources), then
// each warp streams 4 weight rows: a lane loads 8 bytes of E2M1 codes (16
// elements) and one block scale, decodes with cvt.rn.f16x2.e2m1x2, scales (exact
// in FP32) and accumulates against the 8 staged rows.  A 31-shuffle
// reduce-scatter leaves lane l holding the dot product of (row l/8, pair l%8).
// Global scales and the activation are applied in the epilogue.  No atomics:
// every output element is written by exactly one thread.
#include "common.cuh"
#include "internal.h"
#include "launch.h"

namespace bqmoe {

constexpr int kThreads = 256;
constexpr int kRows = 32;  // weight rows per CTA
constexpr int kPT = 8;     // pairs per tile
constexpr int kKC = 512;   // K elements per chunk (32 lanes x 16)

// Four consecutive activation values of row `rid` starting at element k (k % 4 == 0).
template <int SRC>
__device__ __forceinline__ void stage_load4(const GroupedArgs &a, int64_t rid, int k, int K, float (&v)[4]) {
  if (SRC == SRC_X_BF16) {
    const uint2 r = *reinterpret_cast<const uint2 *>(reinterpret_cast<const __nv_bfloat16 *>(a.act) + rid * K + k);
    v[0] = __uint_as_float(r.x << 16);
    v[1] = __uint_as_float(r.x & 0xFFFF0000u);
    v[2] = __uint_as_float(r.y << 16);
    v[3] = __uint_as_float(r.y & 0xFFFF0000u);
  } else if (SRC == SRC_H_F32) {
    const float4 r = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(a.act) + rid * K + k);
    v[0] = r.x; v[1] = r.y; v[2] = r.z; v[3] = r.w;
  } else if (SRC == SRC_X_NVFP4 || SRC == SRC_H_NVFP4) {
    const uint8_t *c = reinterpret_cast<const uint8_t *>(a.act) + rid * (K / 2) + k / 2;
    const uint32_t w = (uint32_t)c[0] | ((uint32_t)c[1] << 8);
    float f[8];
    e2m1x8_to_f32(w, f);
    const float s = e4m3_to_f32(a.act_scales[rid * (K / 16) + k / 16]);
    const float g = a.act_g[rid];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = (f[i] * s) * g;
  } else {  // MXFP8
    const uint32_t w = *reinterpret_cast<const uint32_t *>(reinterpret_cast<const uint8_t *>(a.act) + rid * K + k);
    const float s = e8m0_to_f32(a.act_scales[rid * (K / 32) + k / 32]);
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = e4m3_to_f32((w >> (8 * i)) & 0xFFu) * s;
  }
}

template <int STAGE>
__device__ __forceinline__ int weight_row(int r, int I) {
  if (STAGE == STAGE_GATED) {
    const int f0 = blockIdx.x * 16;
    return r < 16 ? f0 + r : I + f0 + r - 16;
  }
  return blockIdx.x * kRows + r;
}

template <int WFMT, int SRC, int STAGE>
__global__ void __launch_bounds__(kThreads) k_grouped_cc(const GroupedArgs a) {
  __shared__ __align__(16) float act[kPT * kKC];
  __shared__ float dots[kRows][kPT + 1];
  __shared__ int64_t row_of_pt[kPT];
  pdl_trigger();
  pdl_wait();

  const int e = blockIdx.y;
  const int cnt = a.counts[e];
  if (cnt == 0 || (a.tc_min_pairs > 0 && cnt >= a.tc_min_pairs)) return;  // nothing, or the tcgen05 kernel's
  const int off = a.offsets[e];
  const int K = a.K;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int bs = WFMT == W_NVFP4 ? 16 : 32;
  const uint8_t *wc = a.codes + (size_t)e * a.codes_expert;
  const uint8_t *ws = a.scales + (size_t)e * a.scales_expert;
  const float *gl = a.globals + 4 * e;
  constexpr bool by_token = SRC == SRC_X_BF16 || SRC == SRC_X_NVFP4 || SRC == SRC_X_MXFP8;

  for (int s0 = off; s0 < off + cnt; s0 += kPT) {
    const int npt = min(kPT, off + cnt - s0);
    if (threadIdx.x < kPT) {
      int64_t rid = -1;
      if ((int)threadIdx.x < npt) {
        const int s = s0 + threadIdx.x;
        rid = by_token ? (int64_t)(a.sorted_pair[s] / a.top_k) : (int64_t)s;
      }
      row_of_pt[threadIdx.x] = rid;
    }
    float acc[4][kPT];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int p = 0; p < kPT; ++p) acc[r][p] = 0.f;

    for (int c0 = 0; c0 < K; c0 += kKC) {
      __syncthreads();
      // Stage 8 rows x 512 as FP32.  Element k of the chunk goes to float4 slot
      // (k%16)/4 * 32 + k/16 so that lane l's four float4 reads are conflict-free.
      for (int u = threadIdx.x; u < kPT * kKC / 4; u += kThreads) {
        const int pt = u / (kKC / 4), k4 = u % (kKC / 4);
        const int k = c0 + 4 * k4;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        const int64_t rid = row_of_pt[pt];
        if (rid >= 0 && k < K) stage_load4<SRC>(a, rid, k, K, v);
        reinterpret_cast<float4 *>(act)[pt * (kKC / 4) + (k4 & 3) * 32 + (k4 >> 2)] = make_float4(v[0], v[1], v[2], v[3]);
      }
      __syncthreads();
      const int kk = c0 + 16 * lane;
      if (kk < K) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const size_t wr = (size_t)weight_row<STAGE>(warp * 4 + r, a.I);
          const uint2 cw = __ldg(reinterpret_cast<const uint2 *>(wc + wr * (K / 2) + kk / 2));
          const uint32_t sb = __ldg(ws + wr * (K / bs) + kk / bs);
          const float sc = WFMT == W_NVFP4 ? e4m3_to_f32(sb) : e8m0_to_f32(sb);
          float w[16];
          e2m1x8_to_f32(cw.x, *reinterpret_cast<float(*)[8]>(w));
          e2m1x8_to_f32(cw.y, *reinterpret_cast<float(*)[8]>(w + 8));
#pragma unroll
          for (int j = 0; j < 16; ++j) w[j] *= sc;
#pragma unroll
          for (int p = 0; p < kPT; ++p) {
            const float4 *ap = reinterpret_cast<const float4 *>(act) + p * (kKC / 4) + lane;
            float sum = acc[r][p];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float4 x4 = ap[q * 32];
              sum = fmaf(w[4 * q + 0], x4.x, sum);
              sum = fmaf(w[4 * q + 1], x4.y, sum);
              sum = fmaf(w[4 * q + 2], x4.z, sum);
              sum = fmaf(w[4 * q + 3], x4.w, sum);
            }
            acc[r][p] = sum;
          }
        }
      }
    }

    // Reduce-scatter 32 partial sums across the warp: lane l ends with index l = r*8 + p.
    float v[32];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int p = 0; p < kPT; ++p) v[r * kPT + p] = acc[r][p];
#pragma unroll
    for (int step = 16; step >= 1; step >>= 1) {
      const bool upper = (lane & step) != 0;
#pragma unroll
      for (int j = 0; j < step; ++j) {
        const float send = upper ? v[j] : v[j + step];
        const float keep = upper ? v[j + step] : v[j];
        v[j] = keep + __shfl_xor_sync(0xffffffffu, send, step);
      }
    }
    dots[warp * 4 + (lane >> 3)][lane & 7] = v[0];
    __syncthreads();

    const int tid = threadIdx.x;
    if (STAGE == STAGE_GATED) {
      if (tid < 16 * kPT) {
        const int p = tid >> 4, f = tid & 15;
        if (p < npt) {
          const float gate = dots[f][p] * gl[0];
          const float up = dots[16 + f][p] * gl[1];
          a.out[(size_t)(s0 + p) * a.n_rows + blockIdx.x * 16 + f] = silu_f32(gate) * up;
        }
      }
    } else if (STAGE == STAGE_RELU2) {
      const int p = tid >> 5, f = tid & 31;
      if (p < npt) {
        const float r = fmaxf(dots[f][p] * gl[0], 0.f);
        a.out[(size_t)(s0 + p) * a.n_rows + blockIdx.x * kRows + f] = r * r;
      }
    } else {
      const int p = tid >> 5, n = tid & 31;
      if (p < npt) {
        const float w = a.topk_weights[a.sorted_pair[s0 + p]];
        a.out[(size_t)(s0 + p) * a.n_rows + blockIdx.x * kRows + n] = w * (dots[n][p] * gl[2]);
      }
    }
    __syncthreads();
  }
}

template <int WFMT, int SRC, int STAGE>
static cudaError_t launch_one(const GroupedArgs &a, int E, cudaStream_t s) {
  const int nb = STAGE == STAGE_GATED ? a.n_rows / 16 : a.n_rows / kRows;
  return launch_pdl(k_grouped_cc<WFMT, SRC, STAGE>, dim3(nb, E), dim3(kThreads), 0, s, a);
}

template <int WFMT, int STAGE>
static cudaError_t launch_src(int src, const GroupedArgs &a, int E, cudaStream_t s) {
  if (STAGE == STAGE_DOWN) {
    switch (src) {
      case SRC_H_F32: return launch_one<WFMT, SRC_H_F32, STAGE>(a, E, s);
      case SRC_H_NVFP4: return launch_one<WFMT, SRC_H_NVFP4, STAGE>(a, E, s);
      case SRC_H_MXFP8: return launch_one<WFMT, SRC_H_MXFP8, STAGE>(a, E, s);
    }
  } else {
    switch (src) {
      case SRC_X_BF16: return launch_one<WFMT, SRC_X_BF16, STAGE>(a, E, s);
      case SRC_X_NVFP4: return launch_one<WFMT, SRC_X_NVFP4, STAGE>(a, E, s);
      case SRC_X_MXFP8: return launch_one<WFMT, SRC_X_MXFP8, STAGE>(a, E, s);
    }
  }
  return cudaErrorInvalidValue;
}

template <int WFMT>
static cudaError_t launch_stage(int src, int stage, const GroupedArgs &a, int E, cudaStream_t s) {
  switch (stage) {
    case STAGE_GATED: return launch_src<WFMT, STAGE_GATED>(src, a, E, s);
    case STAGE_RELU2: return launch_src<WFMT, STAGE_RELU2>(src, a, E, s);
    case STAGE_DOWN: return launch_src<WFMT, STAGE_DOWN>(src, a, E, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_grouped_cc(int wfmt, int src, int stage, const GroupedArgs &a, int E, cudaStream_t s) {
  if (wfmt == W_NVFP4) return launch_stage<W_NVFP4>(src, stage, a, E, s);
  if (wfmt == W_MXFP4) return launch_stage<W_MXFP4>(src, stage, a, E, s);
  return cudaErrorInvalidValue;
}

}  // namespace bqmoe
