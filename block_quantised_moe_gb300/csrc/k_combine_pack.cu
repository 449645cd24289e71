// Per-token combine of the expert outputs, and the one-time weight packer.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace bqmoe {

// ------------------------------------------------------------------ combine
//
// out[t] = sum over the token's valid pairs of partial[pos], in ascending
// sorted position (= ascending expert, then slot), FP32, rounded once to BF16
// (round-to-nearest-even).  The partials already carry w_tk (GEMM2 epilogue,
// where the router's topk_weights are applied: b12x project page, section
// "Using it", bind(..., topk_weights=tw)).  The fixed order makes the output
// bit-identical across runs and under any permutation of the top-k slots; no
// float atomics are used.
constexpr int kCombThreads = 128;
constexpr int kMaxK = 16;

__global__ void __launch_bounds__(kCombThreads)
k_combine(const float *__restrict__ part, int H, const int32_t *__restrict__ pair_pos, int K,
          __nv_bfloat16 *__restrict__ out) {
  const int t = blockIdx.y;
  int pos[kMaxK];
  int n = 0;
  for (int k = 0; k < K; ++k) {
    const int p = pair_pos[(size_t)t * K + k];
    if (p < 0) continue;
    int j = n++;
    while (j > 0 && pos[j - 1] > p) { pos[j] = pos[j - 1]; --j; }
    pos[j] = p;
  }
  for (int c = (blockIdx.x * kCombThreads + threadIdx.x) * 8; c < H; c += gridDim.x * kCombThreads * 8) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int i = 0; i < n; ++i) {
      const float4 *src = reinterpret_cast<const float4 *>(part + (size_t)pos[i] * H + c);
      const float4 a = src[0], b = src[1];
      acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
      acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
    }
    __align__(16) __nv_bfloat162 o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    *reinterpret_cast<uint4 *>(out + (size_t)t * H + c) = *reinterpret_cast<const uint4 *>(o);
  }
}

cudaError_t launch_combine(const float *part, int H, const int32_t *pair_pos, int T, int K, void *out,
                           cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (K > kMaxK) return cudaErrorInvalidValue;
  const int gx = (H + kCombThreads * 8 - 1) / (kCombThreads * 8);
  k_combine<<<dim3(gx, T), kCombThreads, 0, s>>>(part, H, pair_pos, K, reinterpret_cast<__nv_bfloat16 *>(out));
  return cudaGetLastError();
}

// ------------------------------------------------------------------- packer
//
// One-time preparation of the experts (b12x project page, section "Using it":
// "weights prepped once per model", fused_moe.prepare_weights).  The packed
// buffer keeps the checkpoint's row-major, K-contiguous code and scale arrays
// (what the CUDA-core grouped kernels stream with 8-byte coalesced loads) in
// 256-byte aligned segments, and gathers the global scales into an [E][4] FP32
// table (gate|w1, up, down, 1); MXFP4 has no globals and gets 1.0.
__global__ void k_copy16(const uint4 *__restrict__ src, uint4 *__restrict__ dst, int64_t n16) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = __ldg(src + i);
}

__global__ void k_pack_globals(const float *__restrict__ g13, int n13m, const float *__restrict__ g2, int E,
                               float *__restrict__ gout) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  float a = 1.f, b = 1.f, c = 1.f;
  if (g13 != nullptr) {
    a = g13[(size_t)e * n13m];
    b = n13m > 1 ? g13[(size_t)e * n13m + 1] : 1.f;
  }
  if (g2 != nullptr) c = g2[e];
  reinterpret_cast<float4 *>(gout)[e] = make_float4(a, b, c, 1.f);
}

static cudaError_t copy_seg(const void *src, void *dst, size_t bytes, cudaStream_t s) {
  const int64_t n16 = (int64_t)(bytes / 16);
  if (n16 == 0) return cudaSuccess;
  const int grid = (int)std::min<int64_t>((n16 + 255) / 256, 152 * 16);
  k_copy16<<<grid, 256, 0, s>>>(reinterpret_cast<const uint4 *>(src), reinterpret_cast<uint4 *>(dst), n16);
  return cudaGetLastError();
}

cudaError_t launch_pack(const WeightLayout &L, const void *w13_codes, const void *w13_scales, const float *w13_global,
                        const void *w2_codes, const void *w2_scales, const float *w2_global, uint8_t *packed,
                        cudaStream_t s) {
  cudaError_t err;
  if ((err = copy_seg(w13_codes, packed + L.off_c13, L.E * L.c13_expert(), s)) != cudaSuccess) return err;
  if ((err = copy_seg(w13_scales, packed + L.off_s13, L.E * L.s13_expert(), s)) != cudaSuccess) return err;
  if ((err = copy_seg(w2_codes, packed + L.off_c2, L.E * L.c2_expert(), s)) != cudaSuccess) return err;
  if ((err = copy_seg(w2_scales, packed + L.off_s2, L.E * L.s2_expert(), s)) != cudaSuccess) return err;
  k_pack_globals<<<(L.E + 127) / 128, 128, 0, s>>>(w13_global, L.n13 / L.I, w2_global, L.E,
                                                     reinterpret_cast<float *>(packed + L.off_g));
  return cudaGetLastError();
}

}  // namespace bqmoe
