// Routing: stable counting sort of the (token, slot) pairs by expert.
//
// The op receives topk_ids / topk_weights from the router (b12x project page,
// section "Using it": fused_moe.bind(..., topk_weights=tw, topk_ids=ti)) and the
// grouped expert kernels need each expert's pairs contiguous.  One CTA of 1024
// threads: a shared-memory histogram, a warp scan of the padded counts, then
// the pairs are scattered in chunks of 1024 in ascending pair order (one chunk,
// with no atomics at all, for decode batches); inside a chunk a pair's rank
// among equal ids comes from __match_any_sync (within the warp) plus the
// per-warp counts of the earlier warps, so the result is stable in p = t*K + k
// and bit-identical from run to run.  Only integer shared-memory atomics are
// used.
#include "common.cuh"
#include "dequant.cuh"
#include "internal.h"
#include "launch.h"

namespace bqmoe {

constexpr int kRouteThreads = 1024;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kMaxExperts = 512;

__global__ void __launch_bounds__(kRouteThreads)
k_route(const int32_t *__restrict__ ids, int P, int E, int pad, int ntok, int large_min, int large_tile,
        int32_t *__restrict__ counts, int32_t *__restrict__ offsets, int32_t *__restrict__ sorted_pair,
        int32_t *__restrict__ pair_pos, int32_t *__restrict__ active, int32_t *__restrict__ passes,
        int32_t *__restrict__ large, int32_t *__restrict__ large_tiles, int32_t *__restrict__ status,
        const __nv_bfloat16 *__restrict__ x, int H, __half *__restrict__ x16, float *__restrict__ xfac,
        float *__restrict__ zero, int64_t zero_n) {
  extern __shared__ int32_t sm[];
  // Launched with programmatic dependent launch so that its CTAs are resident
  // before the previous kernel ends; it waits for that kernel before touching
  // memory and never triggers early (later kernels read its outputs freely).
  pdl_wait();
  if (blockIdx.x > 0) {
    // CTAs 1..T: BF16 token rows -> FP16 rows with a power-of-two factor (the
    // tensor-core kernels' B operand), and clear the per-pair max |h| array.
    __shared__ float red[kRouteWarps];
    const int64_t row = blockIdx.x - 1;
    for (int64_t i = row * kRouteThreads + threadIdx.x; i < zero_n; i += (int64_t)(gridDim.x - 1) * kRouteThreads)
      zero[i] = 0.f;
    float m = 0.f;
    for (int k = threadIdx.x * 8; k < H; k += kRouteThreads * 8) {
      float v[8];
      src_load8<SRC_X_BF16>(x, nullptr, row, k, H, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
    }
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = 0.f;
    for (int w = 0; w < kRouteWarps; ++w) m = fmaxf(m, red[w]);
    const float f = stage_factor(m);
    const float inv = __frcp_rn(f);
    stage_row_slots<SRC_X_BF16>(x, nullptr, row, H, inv, x16 + row * H, threadIdx.x, kRouteThreads);
    if (threadIdx.x == 0) xfac[row] = f;
    return;
  }
  int32_t *hist = sm;                 // [E]
  int32_t *base = hist + E;           // [E+1]
  int32_t *cursor = base + E + 1;     // [E]
  int32_t *warp_hist = cursor + E;    // [kRouteWarps][E]
  __shared__ int32_t dropped;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < E; e += kRouteThreads) { hist[e] = 0; cursor[e] = 0; }
  for (int i = tid; i < kRouteWarps * E; i += kRouteThreads) warp_hist[i] = 0;
  if (tid == 0) dropped = 0;
  __syncthreads();

  // 1. histogram.  Up to kRouteThreads pairs (decode) one thread per pair:
  // per-warp counts from __match_any_sync, then for every expert an exclusive
  // prefix of those counts over the warps (one warp-wide scan per expert), so
  // the scatter below needs no further pass.  Otherwise shared-memory atomics.
  const bool one_pass = P <= kRouteThreads;
  int my_id = -1, my_rank = 0;
  if (one_pass) {
    const int p = tid;
    my_id = p < P ? ids[p] : -1;
    const bool valid = my_id >= 0 && my_id < E;
    const unsigned same = __match_any_sync(0xffffffffu, valid ? my_id : E);
    my_rank = __popc(same & ((1u << lane) - 1u));
    // expert-major [E][kRouteWarps] here, so the per-expert scans read consecutive words
    if (valid && my_rank == 0) warp_hist[my_id * kRouteWarps + warp] = __popc(same);
    const unsigned drops = __ballot_sync(0xffffffffu, p < P && !valid);
    if (lane == 0 && drops) atomicAdd(&dropped, __popc(drops));
    if (!valid) my_id = -1;
    __syncthreads();
    for (int e = warp; e < E; e += kRouteWarps) {
      const int v = warp_hist[e * kRouteWarps + lane];
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      warp_hist[e * kRouteWarps + lane] = incl - v;
      if (lane == 31) hist[e] = incl;
    }
  } else {
    int my_drop = 0;
    for (int p = tid; p < P; p += kRouteThreads) {
      const int id = ids[p];
      if (id >= 0 && id < E) atomicAdd(&hist[id], 1);
      else ++my_drop;
    }
    if (my_drop) atomicAdd(&dropped, my_drop);
  }
  __syncthreads();

  // 2. exclusive scan of the padded counts (warp 0)
  if (warp == 0) {
    int carry = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int c = e < E ? hist[e] : 0;
      const int v = (c + pad - 1) / pad * pad;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (e < E) base[e] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) base[E] = carry;
    // Two compact, ascending expert lists: "small" experts (1..large_min-1 pairs)
    // with the prefix of their passes of ntok tokens, and "large" experts
    // (>= large_min pairs) with the prefix of their tiles of large_tile tokens.
    // The grouped kernels split (expert, pass | tile, row block) items evenly.
    int ns = 0, nl = 0, cs = 0, cl = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int c = e < E ? hist[e] : 0;
      const bool sm = c > 0 && c < large_min, lg = c >= large_min;
      const unsigned msm = __ballot_sync(0xffffffffu, sm), mlg = __ballot_sync(0xffffffffu, lg);
      const unsigned below = (1u << lane) - 1u;
      const int vs = sm ? (c + ntok - 1) / ntok : 0, vl = lg ? (c + large_tile - 1) / large_tile : 0;
      int is = vs, il = vl;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int ts = __shfl_up_sync(0xffffffffu, is, o), tl = __shfl_up_sync(0xffffffffu, il, o);
        if (lane >= o) {
          is += ts;
          il += tl;
        }
      }
      if (sm) {
        const int i = ns + __popc(msm & below);
        active[1 + i] = e;
        passes[i] = cs + is - vs;
      }
      if (lg) {
        const int i = nl + __popc(mlg & below);
        large[1 + i] = e;
        large_tiles[i] = cl + il - vl;
      }
      ns += __popc(msm);
      nl += __popc(mlg);
      cs += __shfl_sync(0xffffffffu, is, 31);
      cl += __shfl_sync(0xffffffffu, il, 31);
    }
    if (lane == 0) {
      active[0] = ns;
      passes[ns] = cs;
      large[0] = nl;
      large_tiles[nl] = cl;
    }
  }
  __syncthreads();
  for (int e = tid; e <= E; e += kRouteThreads) offsets[e] = base[e];
  for (int e = tid; e < E; e += kRouteThreads) counts[e] = hist[e];
  // padding slots of every group
  for (int e = warp; e < E; e += kRouteWarps)
    for (int j = base[e] + hist[e] + lane; j < base[e + 1]; j += 32) sorted_pair[j] = -1;

  // 3. stable scatter: position = expert base + pairs of the expert in earlier
  // warps + rank in the warp (one pass), else 1024 pairs at a time
  if (one_pass) {
    const int p = tid;
    if (my_id >= 0) {
      const int pos = base[my_id] + warp_hist[my_id * kRouteWarps + warp] + my_rank;
      sorted_pair[pos] = p;
      pair_pos[p] = pos;
    } else if (p < P) {
      pair_pos[p] = -1;
    }
  }
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int c0 = 0; c0 < P && !one_pass; c0 += kRouteThreads) {
    const int p = c0 + tid;
    const int id = p < P ? ids[p] : -1;
    const bool valid = id >= 0 && id < E;
    const int key = valid ? id : E;  // E: sentinel bucket for dropped / past-the-end pairs
    const unsigned same = __match_any_sync(0xffffffffu, key);
    const int rank = __popc(same & lt_mask);
    if (valid && rank == 0) warp_hist[warp * E + id] = __popc(same);
    __syncthreads();
    if (valid) {
      int pre = 0;
      for (int w = 0; w < warp; ++w) pre += warp_hist[w * E + id];
      const int pos = base[id] + cursor[id] + pre + rank;
      sorted_pair[pos] = p;
      pair_pos[p] = pos;
    } else if (p < P) {
      pair_pos[p] = -1;
    }
    __syncthreads();
    for (int e = tid; e < E; e += kRouteThreads) {
      int n = 0;
      for (int w = 0; w < kRouteWarps; ++w) {
        n += warp_hist[w * E + e];
        warp_hist[w * E + e] = 0;
      }
      cursor[e] += n;
    }
    __syncthreads();
  }

  // Routing runs first in every forward, so it (re)initialises the whole status word.
  if (tid == 0) {
    status[ST_FLAGS] = dropped > 0 ? ST_FLAG_DROPPED : 0;
    status[ST_DROPPED] = dropped;
    status[2] = 0;
    status[3] = 0;
  }
}

cudaError_t launch_route(const int32_t *ids, int P, int E, int pad, int ntok, int large_min, int large_tile,
                         int32_t *counts, int32_t *offsets, int32_t *sorted_pair, int32_t *pair_pos, int32_t *active,
                         int32_t *passes, int32_t *large, int32_t *large_tiles, int32_t *status,
                         const RouteStaging *stg, cudaStream_t s) {
  if (E > kMaxExperts) return cudaErrorInvalidValue;
  const size_t smem = sizeof(int32_t) * ((size_t)3 * E + 1 + (size_t)kRouteWarps * E);
  // Per-device function attribute; cheap and idempotent, so set on every launch.
  cudaError_t err = cudaFuncSetAttribute(k_route, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  // Programmatic launch (the kernel waits before touching memory and never
  // triggers): later kernels of the forward may read the routing outputs as
  // soon as they start.
  const int T = stg ? stg->T : 0;
  return launch_pdl(k_route, dim3(1 + T), dim3(kRouteThreads), smem, s, ids, P, E, pad, ntok, large_min, large_tile,
                    counts, offsets, sorted_pair, pair_pos, active, passes, large, large_tiles, status,
                    stg ? stg->x : nullptr, stg ? stg->H : 0, stg ? stg->x16 : nullptr, stg ? stg->xfac : nullptr,
                    stg ? stg->zero : nullptr, stg ? stg->zero_n : (int64_t)0);
}

}  // namespace bqmoe
