// Routing: stable counting sort of the (token, slot) pairs by expert.
//
// The op receives topk_ids / topk_weights from the router (b12x project page,
// section "Using it": fused_moe.bind(..., topk_weights=tw, topk_ids=ti)) and the
// grouped expert kernels need each expert's pairs contiguous.  Pairs are ranked
// in chunks of 1024 (one per thread): a pair's rank among equal ids in its warp
// comes from __match_any_sync, and the counts of the earlier warps of the chunk
// from one warp-wide scan per expert, so the result is stable in p = t*K + k
// and bit-identical from run to run; only integer shared-memory atomics are
// used.
//   P <= 1024 (decode): one CTA ranks, scans the padded counts and scatters.
//   P > 1024: k_route_rank (one CTA per chunk) writes each chunk's expert
//   counts and every pair's rank inside its chunk; k_route_scatter (one CTA
//   per chunk) adds the counts of the earlier chunks and the expert's base.
#include "common.cuh"
#include "dequant.cuh"
#include "internal.h"
#include "launch.h"
#include "route.cuh"

namespace bqmoe {

constexpr int kRouteThreads = 1024;
constexpr int kRouteWarps = kRouteThreads / 32;

// Extra CTAs of the first routing launch: BF16 token row `row` -> FP16 slot-order
// row with a power-of-two factor (the tensor-core kernels' B operand), and a
// share of the clearing of the per-pair max |h| array.
__device__ void stage_x_row(const __nv_bfloat16 *__restrict__ x, int H, __half *__restrict__ x16,
                            float *__restrict__ xfac, float *__restrict__ zero, int64_t zero_n, int64_t row,
                            int64_t nrows) {
  __shared__ float red[kRouteWarps];
  for (int64_t i = row * kRouteThreads + threadIdx.x; i < zero_n; i += nrows * kRouteThreads) zero[i] = 0.f;
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
}

// The same for many rows: warp w of staging CTA c (of n) takes rows
// 32 c + w, + 32 n, ...; one warp per row (a CTA of 1024 threads per row left
// the large launches bound by CTA scheduling).
__device__ void stage_x_rows_by_warp(const RouteStaging &st, int64_t c, int64_t n) {
  const int lane = threadIdx.x & 31;
  for (int64_t i = c * kRouteThreads + threadIdx.x; i < st.zero_n; i += n * kRouteThreads) st.zero[i] = 0.f;
  for (int64_t row = c * kRouteWarps + (threadIdx.x >> 5); row < st.T; row += n * kRouteWarps) {
    float m = 0.f;
    for (int k = lane * 8; k < st.H; k += 256) {
      float v[8];
      src_load8<SRC_X_BF16>(st.x, nullptr, row, k, st.H, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
    }
    const float f = stage_factor(warp_max(m));
    stage_row_slots<SRC_X_BF16>(st.x, nullptr, row, st.H, __frcp_rn(f), st.x16 + row * st.H, lane, 32);
    if (lane == 0) st.xfac[row] = f;
  }
}

// Ranks the pairs [p0, p0 + kRouteThreads) of `ids` (thread i takes p0 + i).
// warp_hist ([E][kRouteWarps], expert-major so the per-expert scans read
// consecutive words) must be zero on entry.  On return (after a barrier):
// hist[e] = pairs of expert e in the chunk, *dropped incremented by the chunk's
// invalid ids, my_id = the thread's expert (-1 if none or invalid) and my_local
// = pairs of the same expert earlier in the chunk.
__device__ void rank_chunk(const int32_t *__restrict__ ids, int p0, int P, int E, int32_t *warp_hist, int32_t *hist,
                           int32_t *dropped, int &my_id, int &my_local) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int p = p0 + tid;
  int id = p < P ? ids[p] : -1;
  const bool valid = id >= 0 && id < E;
  const unsigned same = __match_any_sync(0xffffffffu, valid ? id : E);
  const int rank = __popc(same & ((1u << lane) - 1u));
  if (valid && rank == 0) warp_hist[id * kRouteWarps + warp] = __popc(same);
  const unsigned drops = __ballot_sync(0xffffffffu, p < P && !valid);
  if (lane == 0 && drops) atomicAdd(dropped, __popc(drops));
  __syncthreads();
#pragma unroll 4
  for (int e = warp; e < E; e += kRouteWarps) {  // exclusive prefix over the warps, per expert
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
  __syncthreads();
  my_id = valid ? id : -1;
  my_local = valid ? warp_hist[id * kRouteWarps + warp] + rank : 0;
}

// The routing launches go out with programmatic dependent launch so that their
// CTAs are resident before the previous kernel ends, and each waits for its
// predecessor before touching memory.  The rank launch triggers its dependent
// (the scatter, which waits before reading) on entry.  The launch whose
// successor is GEMM1 (BF16 x, staged here) also triggers on entry, so GEMM1 is
// resident and set up by the time routing ends; GEMM1 then waits before its
// first read of a routing output and triggers only after that wait.  Otherwise
// routing never triggers early: its outputs are complete when the next kernel
// starts, and every later kernel may read them before waiting.

// P <= kRouteThreads: CTA 0 does the whole sort; CTAs 1..nstage stage x rows.
// Up to 64 registers (one CTA per SM): the expert scan spills at 32.  Its x
// staging CTAs number T + 1 <= 1025 here; the chunked launches below keep 32
// registers so that two of their (many) staging CTAs fit on an SM.
__global__ void __launch_bounds__(kRouteThreads, 1)
k_route_one(const int32_t *__restrict__ ids, int P, int E, int pad, int ntok, int large_min, int large_tile,
            RouteOut o, RouteStaging st) {
  extern __shared__ int32_t sm[];
  if (st.x != nullptr) pdl_trigger();  // the successor is GEMM1, which waits first
  pdl_wait();
  if (blockIdx.x > 0) {
    stage_x_row(st.x, st.H, st.x16, st.xfac, st.zero, st.zero_n, blockIdx.x - 1, gridDim.x - 1);
    return;
  }
  int32_t *hist = sm;               // [E]
  int32_t *base = hist + E;         // [E+1]
  int32_t *warp_hist = base + E + 1;  // [E][kRouteWarps]
  __shared__ int32_t dropped;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < kRouteWarps * E; i += kRouteThreads) warp_hist[i] = 0;
  if (tid == 0) dropped = 0;
  __syncthreads();
  int my_id, my_local;
  rank_chunk(ids, 0, P, E, warp_hist, hist, &dropped, my_id, my_local);
  if (warp == 0)
    scan_experts(hist, E, pad, ntok, large_min, large_tile, base, true, o.active, o.passes, o.large, o.large_tiles,
                 o.tiles, o.balanced != 0);
  __syncthreads();
  for (int e = tid; e <= E; e += kRouteThreads) o.offsets[e] = base[e];
  for (int e = tid; e < E; e += kRouteThreads) o.counts[e] = hist[e];
  for (int e = warp; e < E; e += kRouteWarps)  // padding slots of every group
    for (int j = base[e] + hist[e] + lane; j < base[e + 1]; j += 32) o.sorted_pair[j] = -1;
  if (my_id >= 0) {
    const int pos = base[my_id] + my_local;
    o.sorted_pair[pos] = tid;
    o.pair_pos[tid] = pos;
  } else if (tid < P) {
    o.pair_pos[tid] = -1;
  }
  if (tid == 0) write_status(o.status, dropped);
  for (int i = tid; i < o.work_n; i += kRouteThreads) o.work[i] = 0;
}

// P > kRouteThreads, first launch: CTA c < nchunk ranks chunk c, writing
// chunk_hist[c][0..E-1] = its expert counts, chunk_hist[c][E] = its invalid ids
// and pair_pos[p] = the pair's rank among the chunk's pairs of its expert (-1
// for an invalid id); CTAs past nchunk stage x rows, one warp per row.
__global__ void __launch_bounds__(kRouteThreads)
k_route_rank(const int32_t *__restrict__ ids, int P, int E, int nchunk, int32_t *__restrict__ chunk_hist,
             int32_t *__restrict__ pair_pos, RouteStaging st) {
  extern __shared__ int32_t sm[];
  pdl_trigger();
  pdl_wait();
  if ((int)blockIdx.x >= nchunk) {
    stage_x_rows_by_warp(st, blockIdx.x - nchunk, gridDim.x - nchunk);
    return;
  }
  int32_t *hist = sm;           // [E]
  int32_t *warp_hist = hist + E;  // [E][kRouteWarps]
  __shared__ int32_t dropped;
  const int tid = threadIdx.x;
  for (int i = tid; i < kRouteWarps * E; i += kRouteThreads) warp_hist[i] = 0;
  if (tid == 0) dropped = 0;
  __syncthreads();
  const int c = blockIdx.x, p = c * kRouteThreads + tid;
  int my_id, my_local;
  rank_chunk(ids, c * kRouteThreads, P, E, warp_hist, hist, &dropped, my_id, my_local);
  int32_t *row = chunk_hist + (size_t)c * (E + 1);
  for (int e = tid; e < E; e += kRouteThreads) row[e] = hist[e];
  if (tid == 0) row[E] = dropped;
  if (p < P) pair_pos[p] = my_id >= 0 ? my_local : -1;
}

// P > kRouteThreads, second launch: CTA c sums, per expert, the counts of the
// chunks before c (pre) and of all chunks (the expert's total), scans the
// padded totals, and places its chunk's pairs at base + pre + local rank.
// CTA 0 writes the counts, offsets, expert lists and status; the padding
// slots are filled by all CTAs (expert e by CTA e mod nchunk).
__global__ void __launch_bounds__(kRouteThreads)
k_route_scatter(const int32_t *__restrict__ ids, int P, int E, int pad, int ntok, int large_min, int large_tile,
                int nchunk, const int32_t *__restrict__ chunk_hist, RouteOut o, int early) {
  extern __shared__ int32_t sm[];
  if (early) pdl_trigger();  // the successor is GEMM1, which waits first
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = blockIdx.x;
  const int G = kRouteThreads / (E + 1);  // groups of E + 1 threads splitting the chunks
  int32_t *pre_g = sm;              // [G][E]
  int32_t *tot_g = pre_g + G * E;   // [G][E + 1]  (column E: invalid ids)
  int32_t *base = tot_g + G * (E + 1);  // [E+1]
  int32_t *pre = base + E + 1;      // [E]
  int32_t *tot = pre + E;           // [E + 1]
  if (tid < G * (E + 1)) {
    const int g = tid / (E + 1), e = tid % (E + 1);
    int a = 0, b = 0;
#pragma unroll 8
    for (int j = g; j < nchunk; j += G) {
      const int v = chunk_hist[(size_t)j * (E + 1) + e];
      b += v;
      if (j < c) a += v;
    }
    if (e < E) pre_g[g * E + e] = a;
    tot_g[g * (E + 1) + e] = b;
  }
  __syncthreads();
  for (int e = tid; e <= E; e += kRouteThreads) {
    int a = 0, b = 0;
    for (int g = 0; g < G; ++g) {
      if (e < E) a += pre_g[g * E + e];
      b += tot_g[g * (E + 1) + e];
    }
    if (e < E) pre[e] = a;
    tot[e] = b;
  }
  __syncthreads();
  if (warp == 0)
    scan_experts(tot, E, pad, ntok, large_min, large_tile, base, c == 0, o.active, o.passes, o.large, o.large_tiles,
                 o.tiles, o.balanced != 0);
  __syncthreads();
  if (c == 0) {
    for (int e = tid; e <= E; e += kRouteThreads) o.offsets[e] = base[e];
    for (int e = tid; e < E; e += kRouteThreads) o.counts[e] = tot[e];
    if (tid == 0) write_status(o.status, tot[E]);
    for (int i = tid; i < o.work_n; i += kRouteThreads) o.work[i] = 0;
  }
  for (int e = c + nchunk * warp; e < E; e += nchunk * kRouteWarps)
    for (int j = base[e] + tot[e] + lane; j < base[e + 1]; j += 32) o.sorted_pair[j] = -1;
  const int p = c * kRouteThreads + tid;
  if (p < P) {
    const int id = ids[p];
    if (id >= 0 && id < E) {
      const int pos = base[id] + pre[id] + o.pair_pos[p];
      o.sorted_pair[pos] = p;
      o.pair_pos[p] = pos;
    }
  }
}

int route_chunks(int P) { return P <= kRouteThreads ? 0 : (P + kRouteThreads - 1) / kRouteThreads; }

cudaError_t launch_route(const int32_t *ids, int P, int E, int pad, int ntok, int large_min, int large_tile,
                         int32_t *counts, int32_t *offsets, int32_t *sorted_pair, int32_t *pair_pos, int32_t *active,
                         int32_t *passes, int32_t *large, int32_t *large_tiles, int4 *tiles, int balanced,
                         int32_t *status, int32_t *chunk_hist, int32_t *work, int work_n, const RouteStaging *stg,
                         cudaStream_t s) {
  if (E > kMaxExperts || E < 1) return cudaErrorInvalidValue;
  const RouteOut o{counts, offsets, sorted_pair, pair_pos, active,   passes, large,
                   large_tiles, status, tiles, balanced, work, work_n};
  const RouteStaging st = stg ? *stg : RouteStaging{nullptr, 0, 0, nullptr, nullptr, nullptr, 0};
  const int T = stg ? stg->T : 0;
  const int nchunk = route_chunks(P);
  cudaError_t err;
  if (nchunk == 0) {
    const size_t smem = sizeof(int32_t) * ((size_t)2 * E + 1 + (size_t)kRouteWarps * E);
    // Per-device function attribute; cheap and idempotent, so set on every launch.
    if ((err = cudaFuncSetAttribute(k_route_one, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
      return err;
    return launch_pdl(k_route_one, dim3(1 + T), dim3(kRouteThreads), smem, s, ids, P, E, pad, ntok, large_min,
                      large_tile, o, st);
  }
  if (!chunk_hist) return cudaErrorInvalidValue;
  const size_t smem1 = sizeof(int32_t) * ((size_t)E + (size_t)kRouteWarps * E);
  if ((err = cudaFuncSetAttribute(k_route_rank, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1)) !=
      cudaSuccess)
    return err;
  const int nstage = (T + kRouteWarps - 1) / kRouteWarps;  // x staging CTAs, a row per warp
  if ((err = launch_pdl(k_route_rank, dim3(nchunk + nstage), dim3(kRouteThreads), smem1, s, ids, P, E, nchunk,
                        chunk_hist, pair_pos, st)) != cudaSuccess)
    return err;
  const int G = kRouteThreads / (E + 1);
  const size_t smem2 = sizeof(int32_t) * ((size_t)G * E + (size_t)G * (E + 1) + 3 * (size_t)E + 2);
  if ((err = cudaFuncSetAttribute(k_route_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2)) !=
      cudaSuccess)
    return err;
  return launch_pdl(k_route_scatter, dim3(nchunk), dim3(kRouteThreads), smem2, s, ids, P, E, pad, ntok, large_min,
                    large_tile, nchunk, chunk_hist, o, stg != nullptr ? 1 : 0);
}

}  // namespace bqmoe
