// Measurement helper: back-to-back tcgen05.mma issue rate, the roofline
// denominator of the prefill kernels for their MMA kinds (the block-scaled
// kinds have no cuBLAS counterpart to time against).  One CTA per SM; one warp
// runs the loop and an elected lane issues MMAs from fixed 128-byte-swizzled
// shared-memory operands into TMEM.  The block-scaled kinds read 1.0 scale
// factors from TMEM: UE4M3 for the NVFP4 kind (E2M1 x E2M1, K = 64 per MMA),
// UE8M0 for the MX FP8 kind (E4M3 x E4M3, K = 32 per MMA, one scale per 32).
#include "common.cuh"
#include "internal.h"
#include "moe.h"
#include "sync.cuh"
#include "tcgen05.cuh"

namespace bqmoe {

constexpr int kPeakSmem = 120 * 1024;  // above half an SM's shared memory: one CTA per SM

template <int KIND, int N>
__global__ void __launch_bounds__(128, 1) k_mma_peak(int iters, int32_t *status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = (uint32_t)__cvta_generic_to_shared(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t *base = smem_raw + (base_s - raw_s);
  uint64_t *bar = reinterpret_cast<uint64_t *>(base + 65536);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 1);
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int i = tid; i < 65536 / 4; i += blockDim.x) reinterpret_cast<uint32_t *>(base)[i] = 0x01230123u;
  fence_async_smem();
  const uint32_t mb = (uint32_t)__cvta_generic_to_shared(bar);
  if (tid == 0) {
    mbar_init(mb, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
        (uint32_t)__cvta_generic_to_shared(tmem_slot)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (KIND != 0) {  // scale factors 1.0 (UE4M3 0x38, UE8M0 0x7F) for A and B, every quadrant
    uint32_t r[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) r[j] = KIND == 1 ? 0x38383838u : 0x7F7F7F7Fu;
    tc_st16(tmem + ((uint32_t)(warp * 32) << 16) + 256, r);
    tc_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  bool ok = true;
  if (warp == 0) {
    const uint64_t ad = umma_desc_sw128(base_s), bd = umma_desc_sw128(base_s + 32768);
    for (int it = 0; it < iters; ++it) {
      if (elect_one()) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // 32 bytes of each operand row per MMA
          if (KIND == 0) {
            tc_mma_f16(tmem, ad + 2u * j, bd + 2u * j,
                       (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24), 1u);
          } else if (KIND == 1) {
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], "
                "p;\n\t}" ::"r"(tmem),
                "l"(ad + 2u * j), "l"(bd + 2u * j),
                "r"((1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24)),
                "r"(tmem + 256), "r"(tmem + 260), "r"(1u));
          } else {
            // E4M3 x E4M3 (type 0), UE8M0 scales (bit 23), scale-factor data ID 0
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], "
                "p;\n\t}" ::"r"(tmem),
                "l"(ad + 2u * j), "l"(bd + 2u * j),
                "r"(((uint32_t)(N >> 3) << 17) | (1u << 23) | ((uint32_t)(128 >> 4) << 24)), "r"(tmem + 256),
                "r"(tmem + 260), "r"(1u));
          }
        }
      }
      __syncwarp();
    }
    if (elect_one()) tc_commit(mb);
    __syncwarp();
    ok = mbar_wait(mb, 0);
    if (!ok && tid == 0) atomicOr(&status[0], ST_FLAG_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
}

}  // namespace bqmoe

using namespace bqmoe;

moe_status moe_measure_mma_peak(int32_t kind, int32_t n, int32_t iters, float *tflops) {
  if (!tflops || iters < 1 || (kind != MOE_PEAK_F16 && kind != MOE_PEAK_FP4 && kind != MOE_PEAK_MXFP8) ||
      (n != 128 && n != 256))
    return MOE_ERR_INVALID_ARG;
  void (*k)(int, int32_t *) = nullptr;
  if (kind == MOE_PEAK_F16) k = n == 128 ? k_mma_peak<0, 128> : k_mma_peak<0, 256>;
  else if (kind == MOE_PEAK_FP4) k = n == 128 ? k_mma_peak<1, 128> : k_mma_peak<1, 256>;
  else k = n == 128 ? k_mma_peak<2, 128> : k_mma_peak<2, 256>;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kPeakSmem) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t *status = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  moe_status st = MOE_OK;
  if (cudaMalloc(&status, 16) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemset(status, 0, 16) != cudaSuccess || cudaEventCreate(&e0) != cudaSuccess ||
      cudaEventCreate(&e1) != cudaSuccess) {
    st = MOE_ERR_CUDA;
  } else {
    k<<<sms, 128, kPeakSmem>>>(10, status);  // warm-up
    cudaEventRecord(e0);
    k<<<sms, 128, kPeakSmem>>>(iters, status);
    cudaEventRecord(e1);
    float ms = 0.f;
    int32_t h = 0;
    if (cudaEventSynchronize(e1) != cudaSuccess || cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess ||
        cudaMemcpy(&h, status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) {
      st = MOE_ERR_CUDA;
    } else if (h & ST_FLAG_TIMEOUT) {
      st = MOE_ERR_TIMEOUT;
    } else {
      const double k_per = kind == MOE_PEAK_F16 ? 16.0 : kind == MOE_PEAK_FP4 ? 64.0 : 32.0;
      *tflops = (float)(2.0 * 128 * n * k_per * 4 * (double)iters * sms / (ms * 1e-3) / 1e12);
    }
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  cudaFree(status);
  return st;
}
