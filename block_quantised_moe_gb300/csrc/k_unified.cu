// Host side of the single-launch decode forward (unified.cuh): grid and
// shared-memory sizing, occupancy check and dispatch to the per-format
// instantiations.
#include <algorithm>

#include "unified.cuh"

namespace bqmoe {

cudaError_t launch_unified_nv_bf16(int, int, const UnifiedArgs &, int, int, size_t, cudaStream_t);
cudaError_t launch_unified_nv_nvfp4(int, int, const UnifiedArgs &, int, int, size_t, cudaStream_t);
cudaError_t launch_unified_nv_mxfp8(int, int, const UnifiedArgs &, int, int, size_t, cudaStream_t);
cudaError_t launch_unified_mx_bf16(int, int, const UnifiedArgs &, int, int, size_t, cudaStream_t);
cudaError_t launch_unified_mx_mxfp8(int, int, const UnifiedArgs &, int, int, size_t, cudaStream_t);

bool unified_supported(int wfmt, int afmt, int P, int E, int K) {
  if (P > 1024 || E > kMaxExperts || K > 16) return false;
  if (wfmt == W_NVFP4) return afmt == A_BF16 || afmt == A_NVFP4 || afmt == A_MXFP8;
  if (wfmt == W_MXFP4) return afmt == A_BF16 || afmt == A_MXFP8;
  return false;
}

cudaError_t launch_unified(int wfmt, int afmt, int stage1, int ntok, bool tiny, UnifiedArgs u, cudaStream_t s) {
  const int NT = ntok / 8;
  if (NT != 1 && NT != 2) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t err;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
  // The grouped kernel's sizing: two CTAs per SM with rings of up to 4 stages
  // when they fit (GEMM1's staged rows are the larger), else, and for tiny
  // batches, one CTA per SM with the deepest ring that fits; each GEMM phase
  // takes the deepest ring that fits the CTA's shared memory.
  constexpr size_t kSmemMax = 227 * 1024, kSmemHalf = 112 * 1024;
  const size_t route_bytes = sizeof(int32_t) * ((size_t)2 * u.E + 1 + (size_t)32 * u.E);
  const int Kmax = std::max(u.H, u.I);
  int ctas_per_sm = 2, nst = 4;
  while (nst > 2 && grouped_mma_smem_bytes(Kmax, NT, nst) > kSmemHalf) --nst;
  size_t budget = kSmemHalf;
  if (tiny || grouped_mma_smem_bytes(Kmax, NT, nst) > kSmemHalf || route_bytes > kSmemHalf) {
    ctas_per_sm = 1;
    budget = kSmemMax;
  }
  auto deepest = [&](int K) {
    int n = ctas_per_sm == 1 ? 8 : 4;
    while (n > 2 && grouped_mma_smem_bytes(K, NT, n) > budget) --n;
    return n;
  };
  u.nst1 = deepest(u.H);
  u.nst2 = deepest(u.I);
  const size_t smem = std::max({grouped_mma_smem_bytes(u.H, NT, u.nst1), grouped_mma_smem_bytes(u.I, NT, u.nst2),
                                route_bytes});
  if (smem > budget) return cudaErrorInvalidValue;
  if (sms > kWorkSlots) return cudaErrorInvalidValue;  // one item counter per CTA group (= SM)
  if ((err = cudaMemsetAsync(u.gbar, 0, 2 * sizeof(int32_t), s)) != cudaSuccess) return err;
  if (wfmt == W_NVFP4) {
    if (afmt == A_BF16) return launch_unified_nv_bf16(stage1, NT, u, sms, ctas_per_sm, smem, s);
    if (afmt == A_NVFP4) return launch_unified_nv_nvfp4(stage1, NT, u, sms, ctas_per_sm, smem, s);
    if (afmt == A_MXFP8) return launch_unified_nv_mxfp8(stage1, NT, u, sms, ctas_per_sm, smem, s);
  } else if (wfmt == W_MXFP4) {
    if (afmt == A_BF16) return launch_unified_mx_bf16(stage1, NT, u, sms, ctas_per_sm, smem, s);
    if (afmt == A_MXFP8) return launch_unified_mx_mxfp8(stage1, NT, u, sms, ctas_per_sm, smem, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace bqmoe
