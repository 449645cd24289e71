// Grouped expert contractions on the tensor cores with register-resident
// dequantisation, for NVFP4 weights (any activation format).
//
// moe.fused_moe's W4A16 mode (BF16 activations against FP4 weights dequantised
// in the kernel) and its small-batch decode path (b12x project page, section
// "What's in here").  At decode sizes an
// expert sees a handful of tokens, so the layer is bound by streaming the
// touched experts' packed bytes from HBM; the tensor cores only have to keep the
// multiply-adds off the FP32 pipe.  Design:
//
// * The packer stores every 16-row x 64-K tile of E2M1 codes as 32 x 16-byte
//   lanes in mma.m16n8k16 A-fragment order, and its 16 x 4 E4M3 block scales
//   as 8-byte groups (rows r and r+8 interleaved), codes and scales of a
//   128-row block contiguous per K step.  A producer warp streams them into a
//   shared-memory ring with bulk copies (TMA), and each consumer lane reads its
//   16-byte fragment chunk with one conflict-free shared load.
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
// A unit of work is 128 weight rows of one expert (one per consumer warp) for
// the expert's sorted pairs, in passes of 8 * NT tokens.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "launch.h"
#include "dequant.cuh"
#include "sync.cuh"
#include "grouped_mma.cuh"

namespace bqmoe {


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
  pdl_trigger();
  pdl_wait();
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
  stage_row_slots<SRC>(act, act_scales, row, K, inv, x16 + row * K, threadIdx.x, kStageThreads);
  if (threadIdx.x == 0) fac[row] = f;
}

template <int WF, int SRC, int STAGE, int NT>
__global__ void __maxnreg__(kMmaMaxRegs) k_grouped_mma(const GroupedArgs a, int nst, int ngroups) {
  extern __shared__ __align__(1024) uint8_t smem[];
  grouped_mma_run<WF, SRC, STAGE, NT, true>(a, nst, ngroups, smem, (int)blockIdx.x, (int)gridDim.x);
}

static size_t tma_smem_bytes(int K, int NT, int nst) { return grouped_mma_smem_bytes(K, NT, nst); }

static int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return n;
}

template <int WF, int SRC, int STAGE, int NT>
static cudaError_t launch_mma_one(const GroupedArgs &a, int rows_total, int E, cudaStream_t s) {
  constexpr size_t kSmemMax = 227 * 1024;
  constexpr size_t kSmemHalf = 112 * 1024;  // two CTAs per SM below this
  // Prefer two CTAs per SM (16 consumer warps) with the deepest ring of up to 4
  // stages that still fits twice (at least 2 stages: 37 KB in flight per CTA);
  // else one CTA with the deepest ring that fits.  (Three CTAs with 2-stage
  // rings measured slower at every decode batch size.)
  int ctas_per_sm = 2, nst = 4;
  while (nst > 2 && tma_smem_bytes(a.K, NT, nst) > kSmemHalf) --nst;
  // Tiny batches (at most E/8 pairs: a few items per SM at most) stream each
  // item with as much of it in flight as possible: one CTA per SM, deepest ring
  // (T=1 of the E=128 layer: 26.1 -> 24.4 us; at E/4 pairs it measured slower).
  if (a.tiny || tma_smem_bytes(a.K, NT, nst) > kSmemHalf) {
    ctas_per_sm = 1;
    nst = kMaxStages;
    while (nst > 2 && tma_smem_bytes(a.K, NT, nst) > kSmemMax) --nst;
  }
  const size_t smem = tma_smem_bytes(a.K, NT, nst);
  if (smem > kSmemMax) return cudaErrorInvalidValue;
  cudaError_t err = cudaFuncSetAttribute(k_grouped_mma<WF, SRC, STAGE, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
  if (err != cudaSuccess) return err;
  const int sms = num_sms();
  if (sms <= 0) return cudaErrorInvalidDevice;
  GroupedArgs g = a;
  g.n_blocks = rows_total / (16 * kConsumers);
  const int units_max = E * g.n_blocks;
  const int grid = std::max(1, std::min(sms * ctas_per_sm, units_max));
  // groups of ctas_per_sm CTAs share an item range (blockIdx b, b + ngroups, ...)
  const int ngroups = (grid + ctas_per_sm - 1) / ctas_per_sm;
  if (a.work == nullptr || ngroups > kWorkSlots) return cudaErrorInvalidValue;
  return launch_pdl(k_grouped_mma<WF, SRC, STAGE, NT>, dim3(grid), dim3(kTmaThreads), smem, s, g, nst, ngroups);
}

template <int WF, int STAGE, int NT>
static cudaError_t launch_mma_src(int src, const GroupedArgs &a, int rows_total, int E, cudaStream_t s) {
  if (STAGE == STAGE_DOWN) {
    switch (src) {
      case SRC_H_F32: return launch_mma_one<WF, SRC_H_F32, STAGE, NT>(a, rows_total, E, s);
      case SRC_H_NVFP4:
        if (WF == W_NVFP4) return launch_mma_one<W_NVFP4, SRC_H_NVFP4, STAGE, NT>(a, rows_total, E, s);
        break;
      case SRC_H_MXFP8: return launch_mma_one<WF, SRC_H_MXFP8, STAGE, NT>(a, rows_total, E, s);
    }
  } else if (src == SRC_X16) {
    return launch_mma_one<WF, SRC_X16, STAGE, NT>(a, rows_total, E, s);
  }
  return cudaErrorInvalidValue;
}

template <int WF, int NT>
static cudaError_t launch_mma_nt(int src, int stage, const GroupedArgs &a, int rows_total, int E, cudaStream_t s) {
  switch (stage) {
    case STAGE_GATED: return launch_mma_src<WF, STAGE_GATED, NT>(src, a, rows_total, E, s);
    case STAGE_RELU2: return launch_mma_src<WF, STAGE_RELU2, NT>(src, a, rows_total, E, s);
    case STAGE_DOWN: return launch_mma_src<WF, STAGE_DOWN, NT>(src, a, rows_total, E, s);
  }
  return cudaErrorInvalidValue;
}

template <int WF>
static cudaError_t launch_mma_wf(int src, int stage, const GroupedArgs &a, int rows_total, int E, int ntok,
                                 cudaStream_t s) {
  if (ntok == 16) return launch_mma_nt<WF, 2>(src, stage, a, rows_total, E, s);
  if (ntok == 8) return launch_mma_nt<WF, 1>(src, stage, a, rows_total, E, s);
  return cudaErrorInvalidValue;
}

int mma_tokens_per_pass(int H, int I, bool wide) {
  const int K = H > I ? H : I;
  return wide && tma_smem_bytes(K, 2, 4) <= 227 * 1024 ? 16 : 8;
}

// rows_total: rows of the weight matrix of this stage (2I gated, I for ReLU^2, H down).
// ntok: tokens per pass (8 or 16, from mma_tokens_per_pass; must match routing's).
cudaError_t launch_grouped_mma(int wfmt, int src, int stage, const GroupedArgs &a, int rows_total, int E, int ntok,
                               cudaStream_t s) {
  if (rows_total % (16 * kConsumers) != 0 || a.K % 64 != 0) return cudaErrorInvalidValue;
  if (wfmt == W_NVFP4) return launch_mma_wf<W_NVFP4>(src, stage, a, rows_total, E, ntok, s);
  if (wfmt == W_MXFP4) return launch_mma_wf<W_MXFP4>(src, stage, a, rows_total, E, ntok, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_stage_x16(int src, const void *act, const uint8_t *act_scales, const float *act_g, int T, int K,
                             __half *x16, float *fac, float *zero, int64_t zero_n, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  switch (src) {
    case SRC_X_BF16:
      return launch_pdl(k_stage_x16<SRC_X_BF16>, dim3(T), dim3(kStageThreads), 0, s, act, act_scales, act_g, K, x16, fac,
                        zero, zero_n);
    case SRC_X_NVFP4:
      return launch_pdl(k_stage_x16<SRC_X_NVFP4>, dim3(T), dim3(kStageThreads), 0, s, act, act_scales, act_g, K, x16, fac,
                        zero, zero_n);
    case SRC_X_MXFP8:
      return launch_pdl(k_stage_x16<SRC_X_MXFP8>, dim3(T), dim3(kStageThreads), 0, s, act, act_scales, act_g, K, x16, fac,
                        zero, zero_n);
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace bqmoe
