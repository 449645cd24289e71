// The single-launch decode forward ("a unified dynamic path (persistent
// grid ...)" of moe.fused_moe: b12x project page, section "What's in here").
//
// For decode batches (at most 1024 (token, slot) pairs, no expert on the
// tensor-core kernels) the whole forward runs as one persistent, cooperative
// launch whose CTAs are all resident, in phases separated by grid barriers:
//
//   0  routing (CTA 0: the stable counting sort in shared memory) while the
//      other CTAs stage x as FP16 slot-order rows with a power-of-two factor
//      (BF16 activations) or quantise it (NVFP4 / MXFP8 activations) and stage
//      its codes the same way
//   1  GEMM1 + SiLU(gate)*up or ReLU^2 (the register-dequant grouped kernel's
//      body, items from the routing lists)
//   2  (NVFP4 / MXFP8 activations) re-quantisation of h, one warp per slot row
//   3  GEMM2 x topk_weight into the FP32 partials
//   4  the ordered per-token combine
//
// Every phase performs the same arithmetic, in the same order, as the
// multi-launch forward (the same device code), so the two paths give
// bit-identical outputs.  The grid barriers share one arrival counter in
// scratch, cleared before the launch; a CTA waits, with a two-second bound,
// until every CTA's arrival at the barrier is counted, after which it records
// a timeout in the status word and goes on (the results are then void, the
// context stays usable).
#pragma once

#include "common.cuh"
#include "dequant.cuh"
#include "grouped_mma.cuh"
#include "internal.h"
#include "quant.cuh"
#include "route.cuh"
#include "sync.cuh"
#include "launch.h"

#include <algorithm>

namespace bqmoe {

struct UnifiedArgs {
  const __nv_bfloat16 *x;  // [T][H]
  const int32_t *ids;      // [T][K]
  int T, K, E, H, I;
  int pad, ntok;           // routing: group padding, tokens per pass of the grouped kernel
  RouteOut ro;
  __half *x16;             // [T][H] staged x rows (FP16 slot order)
  float *xfac;             // [T] their factors
  float *hamax;            // [cap] per-pair max |h| (BF16 activations), cleared in phase 0
  int64_t cap_sorted;
  uint8_t *xq_codes, *xq_scales;  // quantised x (NVFP4 / MXFP8 activations)
  float *xq_g;
  uint8_t *hq_codes, *hq_scales;  // quantised h
  float *hq_g;
  GroupedArgs g1, g2;      // the two contractions (act pointers set by the host)
  int nst1, nst2, ngroups;
  const float *part;       // [cap][H] FP32 partials (GEMM2's output)
  __nv_bfloat16 *out;      // [T][H]
  int32_t *gbar;           // grid barrier: arrivals over the launch (0 before it)
  int withhold;            // self-test: CTA 0 does not arrive at the barrier with this tag (-1: never);
                           // tags: 0 after routing, 1 after GEMM1, 2 after the h quantiser, 3 after GEMM2
};

// ------------------------------------------------------------ grid barrier

// All CTAs of the (cooperative, fully resident) grid meet here.  The
// barrier word counts arrivals over the whole launch (cleared before it):
// the launch's barrier number `seq` (0, 1, 2, ...) is complete when seq + 1
// arrivals per CTA have been counted.  Arrivals are fire-and-forget reductions with release semantics
// (no CTA waits for its own atomic's round trip through L2), waiters poll with
// acquire loads.  Bounded: false after kWaitNs without the last arrival.
__device__ __forceinline__ bool grid_sync(const UnifiedArgs &u, int seq, int tag, int *flag_smem) {
  __syncthreads();
  if (threadIdx.x == 0) {
    bool ok = true;
    if (!(u.withhold == tag && blockIdx.x == 0)) {
      asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(u.gbar) : "memory");
      const uint32_t target = (uint32_t)(seq + 1) * gridDim.x;
      uint32_t seen;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(seen) : "l"(u.gbar) : "memory");
      if (seen < target) {
        const unsigned long long t0 = globaltimer_ns();
        for (uint32_t it = 1;; ++it) {
          asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(seen) : "l"(u.gbar) : "memory");
          if (seen >= target) break;
          if ((it & 63u) == 0 && globaltimer_ns() - t0 > kWaitNs) {
            ok = false;
            break;
          }
        }
      }
    }
    *flag_smem = ok ? 1 : 0;
    if (!ok) atomicOr(&u.ro.status[ST_FLAGS], ST_FLAG_TIMEOUT);
  }
  __syncthreads();
  return *flag_smem != 0;
}

// ------------------------------------------------------------ phase 0: routing

// The stable counting sort of k_route_one for at most 1024 pairs, by the
// CTA's warps: 32 virtual warps of 32 pairs each (pair p = 32 vw + lane) give
// the same ranks as the routing kernel's 32 warps.  sm: (2E + 1 + 32E) ints.
static __device__ void route_in_cta(const UnifiedArgs &u, int32_t *sm) {
  constexpr int kVW = 32;
  const int P = u.T * u.K, E = u.E;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  int32_t *hist = sm;                // [E]
  int32_t *base = hist + E;          // [E+1]
  int32_t *vw_hist = base + E + 1;   // [E][kVW]
  __shared__ int32_t dropped;
  for (int i = tid; i < kVW * E; i += blockDim.x) vw_hist[i] = 0;
  if (tid == 0) dropped = 0;
  __syncthreads();
  for (int vw = warp; vw < kVW; vw += nwarps) {
    const int p = vw * 32 + lane;
    const int id = p < P ? u.ids[p] : -1;
    const bool valid = id >= 0 && id < E;
    const unsigned same = __match_any_sync(0xffffffffu, valid ? id : E);
    const int rank = __popc(same & ((1u << lane) - 1u));
    if (valid && rank == 0) vw_hist[id * kVW + vw] = __popc(same);
    const unsigned drops = __ballot_sync(0xffffffffu, p < P && !valid);
    if (lane == 0 && drops) atomicAdd(&dropped, __popc(drops));
  }
  __syncthreads();
  for (int e = warp; e < E; e += nwarps) {  // exclusive prefix over the virtual warps, per expert
    const int v = vw_hist[e * kVW + lane];
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    vw_hist[e * kVW + lane] = incl - v;
    if (lane == 31) hist[e] = incl;
  }
  __syncthreads();
  // no expert goes to the tensor-core kernels on this path
  if (warp == 0)
    scan_experts(hist, E, u.pad, u.ntok, 0x7FFFFFFF, 256, base, true, u.ro.active, u.ro.passes, u.ro.large,
                 u.ro.large_tiles, nullptr, false);
  __syncthreads();
  for (int e = tid; e <= E; e += blockDim.x) u.ro.offsets[e] = base[e];
  for (int e = tid; e < E; e += blockDim.x) u.ro.counts[e] = hist[e];
  for (int e = warp; e < E; e += nwarps)  // padding slots of every group
    for (int j = base[e] + hist[e] + lane; j < base[e + 1]; j += 32) u.ro.sorted_pair[j] = -1;
  for (int vw = warp; vw < kVW; vw += nwarps) {
    const int p = vw * 32 + lane;
    const int id = p < P ? u.ids[p] : -1;
    const bool valid = id >= 0 && id < E;
    const unsigned same = __match_any_sync(0xffffffffu, valid ? id : E);
    const int rank = __popc(same & ((1u << lane) - 1u));
    if (valid) {
      const int pos = base[id] + vw_hist[id * kVW + vw] + rank;
      u.ro.sorted_pair[pos] = p;
      u.ro.pair_pos[p] = pos;
    } else if (p < P) {
      u.ro.pair_pos[p] = -1;
    }
  }
  if (tid == 0) write_status(u.ro.status, dropped);
  for (int i = tid; i < u.ro.work_n; i += blockDim.x) u.ro.work[i] = 0;
}

// ------------------------------------------------------------ phase 0: activations

// Token row `row` of x: quantised (NVFP4 with a per-row global, or MXFP8) when
// the activations are, then staged as FP16 slot-order rows with the factor of
// the multi-launch path (the row's global for NVFP4, a power of two from the
// row's largest magnitude otherwise).  One warp.
template <int AF>
__device__ void stage_token_row(const UnifiedArgs &u, int row, int lane) {
  const int H = u.H;
  __half *dst = u.x16 + (int64_t)row * H;
  if (AF == A_BF16) {
    float m = 0.f;
    for (int k = lane * 8; k < H; k += 256) {
      float v[8];
      src_load8<SRC_X_BF16>(u.x, nullptr, row, k, H, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
    }
    const float f = stage_factor(warp_max(m));
    stage_row_slots<SRC_X_BF16>(u.x, nullptr, row, H, __frcp_rn(f), dst, lane, 32);
    if (lane == 0) u.xfac[row] = f;
    return;
  }
  const int64_t base = (int64_t)row * H;
  if (AF == A_NVFP4) {
    float m = 0.f;
    for (int j = lane * 8; j < H; j += 256) {
      float v[8];
      load8<true>(u.x, base + j, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
    }
    const float g = __fdiv_rn(warp_max(m), 2688.0f);
    for (int b = lane; b < H / 16; b += 32) {
      float xv[16];
      load8<true>(u.x, base + b * 16, *reinterpret_cast<float(*)[8]>(xv));
      load8<true>(u.x, base + b * 16 + 8, *reinterpret_cast<float(*)[8]>(xv + 8));
      uint2 c;
      uint32_t sc;
      nvfp4_block(xv, g, c, sc);
      *reinterpret_cast<uint2 *>(u.xq_codes + (base + b * 16) / 2) = c;
      u.xq_scales[(int64_t)row * (H / 16) + b] = (uint8_t)sc;
    }
    if (lane == 0) u.xq_g[row] = g;
    __syncwarp();  // the row's codes, written by the warp's lanes, are read back below
    stage_row_slots<SRC_X_NVFP4>(u.xq_codes, u.xq_scales, row, H, 1.f, dst, lane, 32);
    if (lane == 0) u.xfac[row] = g;
    return;
  }
  // MXFP8
  for (int b = lane; b < H / 32; b += 32) {
    float xv[32];
#pragma unroll
    for (int q = 0; q < 4; ++q) load8<true>(u.x, base + b * 32 + 8 * q, *reinterpret_cast<float(*)[8]>(xv + 8 * q));
    uint32_t c[8];
    uint32_t sc;
    mx_block<Q_MXFP8>(xv, c, sc);
    uint4 *cd = reinterpret_cast<uint4 *>(u.xq_codes + base + b * 32);
    cd[0] = make_uint4(c[0], c[1], c[2], c[3]);
    cd[1] = make_uint4(c[4], c[5], c[6], c[7]);
    u.xq_scales[(int64_t)row * (H / 32) + b] = (uint8_t)sc;
  }
  __syncwarp();
  float m = 0.f;
  for (int k = lane * 8; k < H; k += 256) {
    float v[8];
    src_load8<SRC_X_MXFP8>(u.xq_codes, u.xq_scales, row, k, H, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
  }
  const float f = stage_factor(warp_max(m));
  stage_row_slots<SRC_X_MXFP8>(u.xq_codes, u.xq_scales, row, H, __frcp_rn(f), dst, lane, 32);
  if (lane == 0) u.xfac[row] = f;
}

// ------------------------------------------------------------ phase 2: h re-quantisation

// Slot row `row` of h (FP32 [cap][I]) re-quantised as the multi-launch
// forward does (NVFP4 with a per-row global, or MXFP8).  One warp.
template <int AF>
__device__ void quant_h_row(const UnifiedArgs &u, int64_t row, int lane) {
  const int I = u.I;
  const float *h = u.g1.out;
  const int64_t base = row * I;
  if (AF == A_NVFP4) {
    float m = 0.f;
    for (int j = lane * 8; j < I; j += 256) {
      float v[8];
      load8<false>(h, base + j, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
    }
    const float g = __fdiv_rn(warp_max(m), 2688.0f);
    if (lane == 0) u.hq_g[row] = g;
    for (int b = lane; b < I / 16; b += 32) {
      float xv[16];
      load8<false>(h, base + b * 16, *reinterpret_cast<float(*)[8]>(xv));
      load8<false>(h, base + b * 16 + 8, *reinterpret_cast<float(*)[8]>(xv + 8));
      uint2 c;
      uint32_t sc;
      nvfp4_block(xv, g, c, sc);
      *reinterpret_cast<uint2 *>(u.hq_codes + (base + b * 16) / 2) = c;
      u.hq_scales[row * (I / 16) + b] = (uint8_t)sc;
    }
  } else {
    for (int b = lane; b < I / 32; b += 32) {
      float xv[32];
#pragma unroll
      for (int q = 0; q < 4; ++q) load8<false>(h, base + b * 32 + 8 * q, *reinterpret_cast<float(*)[8]>(xv + 8 * q));
      uint32_t c[8];
      uint32_t sc;
      mx_block<Q_MXFP8>(xv, c, sc);
      uint4 *cd = reinterpret_cast<uint4 *>(u.hq_codes + base + b * 32);
      cd[0] = make_uint4(c[0], c[1], c[2], c[3]);
      cd[1] = make_uint4(c[4], c[5], c[6], c[7]);
      u.hq_scales[row * (I / 32) + b] = (uint8_t)sc;
    }
  }
}

// ------------------------------------------------------------ phase 4: combine

// out[t] = sum of t's partials in ascending sorted position, FP32, rounded
// once to BF16: the arithmetic of k_combine, with the CTA's threads over the
// columns (8 each).
static __device__ void combine_token(const UnifiedArgs &u, int t) {
  constexpr int kMaxK = 16;
  int pos[kMaxK];
  int n = 0;
  for (int k = 0; k < u.K; ++k) {
    const int p = u.ro.pair_pos[(int64_t)t * u.K + k];
    if (p < 0) continue;
    int j = n++;
    while (j > 0 && pos[j - 1] > p) {
      pos[j] = pos[j - 1];
      --j;
    }
    pos[j] = p;
  }
  for (int c = threadIdx.x * 8; c < u.H; c += blockDim.x * 8) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int i = 0; i < n; ++i) {
      const float4 a = *reinterpret_cast<const float4 *>(u.part + (int64_t)pos[i] * u.H + c);
      const float4 b = *reinterpret_cast<const float4 *>(u.part + (int64_t)pos[i] * u.H + c + 4);
      acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
      acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
    }
    __align__(16) __nv_bfloat162 o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
    *reinterpret_cast<uint4 *>(u.out + (int64_t)t * u.H + c) = *reinterpret_cast<const uint4 *>(o);
  }
}

// ------------------------------------------------------------ the kernel

template <int WF, int AF, int STAGE1, int NT>
__global__ void __maxnreg__(kMmaMaxRegs) k_unified(const UnifiedArgs u) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ int sync_flag;
  const int cta = (int)blockIdx.x, ncta = (int)gridDim.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;

  // phase 0: routing on CTA 0; activation rows and the |h| maxima elsewhere
  if (cta == 0) route_in_cta(u, reinterpret_cast<int32_t *>(smem));
  {
    const int first = ncta > 1 ? 1 : 0;
    const int gw = (cta - first) * nwarps + warp, nw = (ncta - first) * nwarps;
    if (cta >= first) {
      for (int row = gw; row < u.T; row += nw) stage_token_row<AF>(u, row, lane);
      if (AF == A_BF16)
        for (int64_t i = (int64_t)gw * 32 + lane; i < u.cap_sorted; i += (int64_t)nw * 32) u.hamax[i] = 0.f;
    }
  }
  int seq = 0;
  grid_sync(u, seq++, 0, &sync_flag);

  // phase 1: GEMM1
  grouped_mma_run<WF, SRC_X16, STAGE1, NT, false>(u.g1, u.nst1, u.ngroups, smem, cta, ncta);
  grid_sync(u, seq++, 1, &sync_flag);

  // phase 2: h re-quantisation
  constexpr int SRC2 = AF == A_BF16 ? SRC_H_F32 : (AF == A_NVFP4 ? SRC_H_NVFP4 : SRC_H_MXFP8);
  if (AF != A_BF16) {
    const int64_t live = u.ro.offsets[u.E];
    for (int64_t row = (int64_t)cta * nwarps + warp; row < live; row += (int64_t)ncta * nwarps)
      if (u.ro.sorted_pair[row] >= 0) quant_h_row<AF>(u, row, lane);
    grid_sync(u, seq++, 2, &sync_flag);
  }

  // phase 3: GEMM2
  grouped_mma_run<WF, SRC2, STAGE_DOWN, NT, false>(u.g2, u.nst2, u.ngroups, smem, cta, ncta);
  grid_sync(u, seq++, 3, &sync_flag);

  // phase 4: combine
  for (int t = cta; t < u.T; t += ncta) combine_token(u, t);
}

// Cooperative launch (every CTA resident, as the grid barriers need) of a
// unified kernel: kTmaThreads threads per CTA, `smem` bytes of dynamic shared
// memory, `ctas_per_sm` CTAs on each of `sms` SMs, fewer if the kernel's
// occupancy allows fewer.
inline cudaError_t launch_cooperative(void (*k)(const UnifiedArgs), int sms, int ctas_per_sm, size_t smem,
                                      cudaStream_t s, UnifiedArgs u) {
  cudaError_t err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  int occ = 0;
  if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kTmaThreads, smem)) != cudaSuccess) return err;
  if (occ < 1) return cudaErrorInvalidConfiguration;
  const int grid = sms * std::min(ctas_per_sm, occ);
  u.ngroups = sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTmaThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  ++launch_counter();
  return cudaLaunchKernelEx(&cfg, k, u);
}

// Per (weight format, activation format) launchers, one translation unit each
// (k_unified_*.cu) so the instantiations compile in parallel.
#define BQMOE_UNIFIED_LAUNCHER(NAME, WF, AF)                                                                      \
  cudaError_t NAME(int stage1, int nt, const UnifiedArgs &u, int sms, int ctas_per_sm, size_t smem,               \
                   cudaStream_t s) {                                                                             \
    void (*k)(const UnifiedArgs) = nullptr;                                                                       \
    if (stage1 == STAGE_GATED)                                                                                    \
      k = nt == 2 ? k_unified<WF, AF, STAGE_GATED, 2> : k_unified<WF, AF, STAGE_GATED, 1>;                        \
    else if (stage1 == STAGE_RELU2)                                                                               \
      k = nt == 2 ? k_unified<WF, AF, STAGE_RELU2, 2> : k_unified<WF, AF, STAGE_RELU2, 1>;                        \
    else                                                                                                          \
      return cudaErrorInvalidValue;                                                                               \
    return launch_cooperative(k, sms, ctas_per_sm, smem, s, u);                                                   \
  }

}  // namespace bqmoe
