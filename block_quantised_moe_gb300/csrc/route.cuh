// Routing pieces shared by the routing kernels and the single-launch decode
// forward: the expert scan that builds the padded offsets and the compact
// expert lists, the status word, and the routing outputs.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace bqmoe {

// Warp 0: base[e] = exclusive prefix of the counts padded to `pad` (base[E] =
// total), and, when `lists`, the two compact ascending expert lists: "small"
// experts (1..large_min-1 pairs) with the prefix of their passes of ntok tokens,
// and "large" experts (>= large_min pairs) with the prefix of their tiles of
// large_tile tokens.  The grouped kernels split (expert, pass | tile, row
// block) items evenly.  Lane l owns the consecutive experts [l*per, l*per+per)
// (per = ceil(E/32)): it sums its experts, one warp scan per quantity turns the
// sums into the lane's starting offsets, and the lane then writes its experts
// in order, so the lists stay ascending.  With `tiles`, the lists pass also
// writes one record per token tile of the large experts, in item order:
// (expert, first slot, live tokens, 0).  An expert with c pairs has
// nt = ceil(c / large_tile) tiles: with `balanced`, of equal size rounded up
// to 16 (the last one possibly shorter), so that no tile is a nearly empty
// remainder; otherwise of large_tile pairs each but the last.
__device__ __forceinline__ int round_up_div(int c, int d) { return (c + d - 1) / d; }

static __device__ void scan_experts(const int32_t *hist, int E, int pad, int ntok, int large_min, int large_tile,
                             int32_t *base, bool lists, int32_t *__restrict__ active, int32_t *__restrict__ passes,
                             int32_t *__restrict__ large, int32_t *__restrict__ large_tiles,
                             int4 *__restrict__ tiles, bool balanced) {
  const int lane = threadIdx.x & 31;
  const int per = (E + 31) / 32;
  const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
  // the lane's padded pairs, small experts and their passes, large experts and their tiles
  int v[5] = {0, 0, 0, 0, 0};
  for (int e = e0; e < e1; ++e) {
    const int c = hist[e];
    v[0] += round_up_div(c, pad) * pad;
    if (c > 0 && c < large_min) {
      v[1] += 1;
      v[2] += round_up_div(c, ntok);
    } else if (c >= large_min) {
      v[3] += 1;
      v[4] += round_up_div(c, large_tile);
    }
  }
  int incl[5];
#pragma unroll
  for (int q = 0; q < 5; ++q) incl[q] = v[q];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int q = 0; q < 5; ++q) {
      const int n = __shfl_up_sync(0xffffffffu, incl[q], o);
      if (lane >= o) incl[q] += n;
    }
  }
  int b = incl[0] - v[0], ns = incl[1] - v[1], cs = incl[2] - v[2], nl = incl[3] - v[3], cl = incl[4] - v[4];
  for (int e = e0; e < e1; ++e) {
    const int c = hist[e];
    base[e] = b;
    b += round_up_div(c, pad) * pad;
    if (!lists) continue;
    if (c > 0 && c < large_min) {
      active[1 + ns] = e;
      passes[ns++] = cs;
      cs += round_up_div(c, ntok);
    } else if (c >= large_min) {
      large[1 + nl] = e;
      large_tiles[nl++] = cl;
      const int nt = round_up_div(c, large_tile);
      if (tiles != nullptr) {
        const int tsz = balanced ? (round_up_div(c, nt) + 15) & ~15 : large_tile;
        for (int t = 0; t < nt; ++t) tiles[cl + t] = make_int4(e, base[e] + t * tsz, max(0, min(tsz, c - t * tsz)), 0);
      }
      cl += nt;
    }
  }
  if (lane == 31) {  // the inclusive sums of the last lane are the totals
    base[E] = incl[0];
    if (lists) {
      active[0] = incl[1];
      passes[incl[1]] = incl[2];
      large[0] = incl[3];
      large_tiles[incl[3]] = incl[4];
    }
  }
}

// Routing runs first in every forward, so it (re)initialises the whole status word.
__device__ __forceinline__ void write_status(int32_t *status, int dropped) {
  status[ST_FLAGS] = dropped > 0 ? ST_FLAG_DROPPED : 0;
  status[ST_DROPPED] = dropped;
  status[2] = 0;
  status[3] = 0;
}

struct RouteOut {
  int32_t *counts, *offsets, *sorted_pair, *pair_pos, *active, *passes, *large, *large_tiles, *status;
  int4 *tiles;    // token tiles of the large experts (may be null)
  int balanced;   // tiles of equal size (else of large_tile pairs but the last)
  int32_t *work;  // work_n counters of the grouped kernels, zeroed here
  int work_n;
};

}  // namespace bqmoe
