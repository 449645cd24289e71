// Block quantisers: NVFP4 (E2M1 + E4M3 per 16 + FP32 global) and MX
// (E2M1 or E4M3 elements + E8M0 per 32), the row quantizers quantization.nvfp4 /
// quantization.mxfp8 of the b12x project page (section "What's in here").
//
// NVFP4:  g = amax/(6*448);  s = E4M3_rne_sat((amax_b/6)/g);  d = s*g;
//         q = E2M1_rne_sat(x/d)  (0 when d == 0)
// MX:     X = floor(log2(amax_b)) - emax (2 for E2M1, 8 for E4M3), clamped to
//         [-127, 127], -127 for an all-zero block;  s = X+127;  q = ELEM_rne_sat(x/2^X)
//
// Every step is a correctly rounded FP32 operation (__fdiv_rn, __fmul_rn) and
// the element conversions are the cvt.rn.satfinite instructions, so the codes
// and scales are a pure function of the input bits.  HBM-bound: one pass over
// the input (two for a per-row or per-tensor global).
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "launch.h"
#include "quant.cuh"

namespace bqmoe {

constexpr int kQThreads = 256;

__device__ __forceinline__ float block_max(float v, float *red) {
  v = warp_max(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.f;
    v = warp_max(v);
    if (lane == 0) red[0] = v;
  }
  __syncthreads();
  const float r = red[0];
  __syncthreads();
  return r;
}

// Position of 16-element block b of a row in a slot-major FP4 tile buffer
// (128 slots x 256 K per 18432-byte tile: codes in the 128-byte-swizzled K-major
// layout, then the slots' scales as four 512-byte blocks, one per 64-K step, in
// the tensor-memory scale layout: lane slot % 32, column slot / 32 % 4, the four
// blocks of the step in the column's four bytes).
__device__ __forceinline__ uint8_t *fp4_tile_codes(uint8_t *tiles, int64_t slot, int64_t b, int nkb) {
  const int64_t kb = b >> 4, r = slot & 127;
  uint8_t *tile = tiles + ((slot >> 7) * nkb + kb) * 18432;
  const int c = (int)((b & 15) >> 1);  // 16-byte chunk of the 128-byte row
  return tile + (r >> 3) * 1024 + (r & 7) * 128 + (((c ^ (int)r) & 7) << 4) + 8 * (b & 1);
}
__device__ __forceinline__ uint8_t *fp4_tile_scale(uint8_t *tiles, int64_t slot, int64_t b, int nkb) {
  // 64-K step (b & 15) >> 2, TMEM lane slot & 31, column (slot & 127) >> 5, byte b & 3
  const int r = (int)(slot & 127), j = (int)(b & 15);
  return tiles + ((slot >> 7) * nkb + (b >> 4)) * 18432 + 16384 + (j >> 2) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (j & 3);
}

// NVFP4 with one global per row, rows up to 2048 wide: one warp per row over a
// persistent grid (a CTA per row made the kernel bound by CTA launches at 65k
// rows of 2048; wide rows keep a CTA each, below).  Pass 1 takes the
// row's amax, pass 2 (re-reading the row, now in L1/L2) quantises 16-element
// blocks, block b on lane b % 32, so loads and stores are coalesced.  With
// `tiles` the row's codes and scales also go to the slot-major FP4 tiles of the
// block-scaled kernel: a token row (tile_slots = pair_pos, top_k > 0) to each of
// its valid slots, a slot row (top_k == 0) to its own slot.
template <bool BF16>
__global__ void __launch_bounds__(kQThreads)
k_quant_rows_nvfp4(const void *__restrict__ src, int64_t rows, int64_t cols, uint8_t *__restrict__ codes,
                   uint8_t *__restrict__ scales, float *__restrict__ g_out, const int32_t *__restrict__ rows_dev,
                   const int32_t *__restrict__ row_live, uint8_t *__restrict__ tiles,
                   const int32_t *__restrict__ tile_slots, int top_k) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t live_rows = rows_dev != nullptr ? min(rows, (int64_t)*rows_dev) : rows;
  const int64_t nwarps = (int64_t)gridDim.x * (kQThreads / 32);
  const int64_t nb = cols / 16;
  const int nkb = (int)(cols / 256);
  for (int64_t row = (int64_t)blockIdx.x * (kQThreads / 32) + (threadIdx.x >> 5); row < live_rows; row += nwarps) {
    if (row_live != nullptr && row_live[row] < 0) continue;  // a padding slot of the expert-sorted list
    const int64_t base = row * cols;
    float m = 0.f;
    for (int64_t j = (int64_t)lane * 8; j < cols; j += 256) {
      float v[8];
      load8<BF16>(src, base + j, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
    }
    const float amax = warp_max(m);
    const float g = __fdiv_rn(amax, 2688.0f);
    if (lane == 0) g_out[row] = g;
    for (int64_t b = lane; b < nb; b += 32) {
      float x[16];
      load8<BF16>(src, base + b * 16, *reinterpret_cast<float(*)[8]>(x));
      load8<BF16>(src, base + b * 16 + 8, *reinterpret_cast<float(*)[8]>(x + 8));
      uint2 c;
      uint32_t sc;
      nvfp4_block(x, g, c, sc);
      *reinterpret_cast<uint2 *>(codes + (base + b * 16) / 2) = c;
      scales[row * nb + b] = (uint8_t)sc;
      if (tiles != nullptr) {
        // Lanes 4i..4i+3 hold the four blocks of one 64-K step (nb is a multiple
        // of 16, so the group is all active): one 32-bit scale store.
        const unsigned grp = 0xFu << (lane & 28);
        const uint32_t s1 = __shfl_down_sync(grp, sc, 1, 4), s2 = __shfl_down_sync(grp, sc, 2, 4),
                       s3 = __shfl_down_sync(grp, sc, 3, 4);
        const uint32_t s4 = (sc & 0xFFu) | (s1 & 0xFFu) << 8 | (s2 & 0xFFu) << 16 | (s3 & 0xFFu) << 24;
        for (int k = 0; k < (top_k > 0 ? top_k : 1); ++k) {
          const int64_t slot = top_k > 0 ? (int64_t)tile_slots[row * top_k + k] : row;
          if (slot < 0) continue;
          *reinterpret_cast<uint2 *>(fp4_tile_codes(tiles, slot, b, nkb)) = c;
          if ((b & 3) == 0) *reinterpret_cast<uint32_t *>(fp4_tile_scale(tiles, slot, b, nkb)) = s4;
        }
      }
    }
  }
}

// NVFP4 with one global per row, one CTA per row (rows wider than 2048).  With `tiles` the row's codes
// and scales also go to the slot-major FP4 tiles of the block-scaled kernel:
// a token row (tile_slots = pair_pos, top_k > 0) to each of its valid slots, a
// slot row (top_k == 0) to its own slot.
template <bool BF16>
__global__ void __launch_bounds__(kQThreads)
k_quant_rows_nvfp4_cta(const void *__restrict__ src, int64_t cols, uint8_t *__restrict__ codes,
                   uint8_t *__restrict__ scales, float *__restrict__ g_out, const int32_t *__restrict__ rows_dev,
                   const int32_t *__restrict__ row_live, uint8_t *__restrict__ tiles,
                   const int32_t *__restrict__ tile_slots, int top_k) {
  __shared__ float red[32];
  pdl_trigger();
  pdl_wait();
  const int64_t row = blockIdx.x;
  if (rows_dev != nullptr && row >= *rows_dev) return;
  if (row_live != nullptr && row_live[row] < 0) return;  // a padding slot of the expert-sorted list
  const int64_t base = row * cols;
  float m = 0.f;
  for (int64_t j = (int64_t)threadIdx.x * 8; j < cols; j += kQThreads * 8) {
    float v[8];
    load8<BF16>(src, base + j, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
  }
  const float amax = block_max(m, red);
  const float g = __fdiv_rn(amax, 2688.0f);
  if (threadIdx.x == 0) g_out[row] = g;
  for (int64_t b = threadIdx.x; b < cols / 16; b += kQThreads) {
    float x[16];
    float *lo = x, *hi = x + 8;
    load8<BF16>(src, base + b * 16, *reinterpret_cast<float(*)[8]>(lo));
    load8<BF16>(src, base + b * 16 + 8, *reinterpret_cast<float(*)[8]>(hi));
    uint2 c;
    uint32_t s;
    nvfp4_block(x, g, c, s);
    *reinterpret_cast<uint2 *>(codes + (base + b * 16) / 2) = c;
    scales[row * (cols / 16) + b] = (uint8_t)s;
    if (tiles != nullptr) {
      const int nkb = (int)(cols / 256);
      // Lanes 4i..4i+3 hold the four blocks of one 64-K step (cols / 16 is a
      // multiple of 16, so the group is all active): one 32-bit scale store.
      const unsigned grp = 0xFu << (threadIdx.x & 28);
      const uint32_t s1 = __shfl_down_sync(grp, s, 1, 4), s2 = __shfl_down_sync(grp, s, 2, 4),
                     s3 = __shfl_down_sync(grp, s, 3, 4);
      const uint32_t s4 = (s & 0xFFu) | (s1 & 0xFFu) << 8 | (s2 & 0xFFu) << 16 | (s3 & 0xFFu) << 24;
      for (int k = 0; k < (top_k > 0 ? top_k : 1); ++k) {
        const int64_t slot = top_k > 0 ? (int64_t)tile_slots[row * top_k + k] : row;
        if (slot < 0) continue;
        *reinterpret_cast<uint2 *>(fp4_tile_codes(tiles, slot, b, nkb)) = c;
        if ((b & 3) == 0) *reinterpret_cast<uint32_t *>(fp4_tile_scale(tiles, slot, b, nkb)) = s4;
      }
    }
  }
}

// Slot-major MX FP8 tiles of the block-scaled FP8 kernel: per 128 slots and
// 128-K block, 16 KB of E4M3 codes in the 128-byte-swizzled K-major layout
// with the K order of each 32-element block transposed as a 8 x 4 matrix
// (logical element 4i + c at physical 8c + i, the order in which that kernel
// writes its widened weights), then 512 bytes of UE8M0 scales in TMEM order
// (lane i, column c = slot i + 32c; byte = the 32-K block within the 128).
// Block b of slot `slot`: codes c (element 4w + i in byte i of c[w]), scale s.
__device__ __forceinline__ void mx8_tile_put(uint8_t *tiles, int64_t slot, int64_t b, int64_t nkb,
                                             const uint32_t (&c)[8], uint32_t s) {
  const int64_t kb = b >> 2;
  const int qb = (int)(b & 3);
  const int r = (int)(slot & 127);
  uint8_t *tile = tiles + ((slot >> 7) * nkb + kb) * kMx8TileBytes;
  // physical word w = byte (w >> 1) of logical words 4 (w & 1) .. 4 (w & 1) + 3:
  // a 4 x 4 byte transpose of c[0..3] (even w) and of c[4..7] (odd w)
  uint32_t o[2][4];
#pragma unroll
  for (int gq = 0; gq < 2; ++gq) {
    const uint32_t t0 = __byte_perm(c[4 * gq], c[4 * gq + 1], 0x5140), t1 = __byte_perm(c[4 * gq], c[4 * gq + 1], 0x7362);
    const uint32_t t2 = __byte_perm(c[4 * gq + 2], c[4 * gq + 3], 0x5140),
                   t3 = __byte_perm(c[4 * gq + 2], c[4 * gq + 3], 0x7362);
    o[gq][0] = __byte_perm(t0, t2, 0x5410);
    o[gq][1] = __byte_perm(t0, t2, 0x7632);
    o[gq][2] = __byte_perm(t1, t3, 0x5410);
    o[gq][3] = __byte_perm(t1, t3, 0x7632);
  }
  uint8_t *row = tile + (r >> 3) * 1024 + (r & 7) * 128;
  const int ch = 2 * qb;  // 16-byte chunk of the row's 128 bytes
  *reinterpret_cast<uint4 *>(row + (((ch ^ r) & 7) << 4)) = make_uint4(o[0][0], o[1][0], o[0][1], o[1][1]);
  *reinterpret_cast<uint4 *>(row + ((((ch + 1) ^ r) & 7) << 4)) = make_uint4(o[0][2], o[1][2], o[0][3], o[1][3]);
  tile[16384 + (r & 31) * 16 + (r >> 5) * 4 + qb] = (uint8_t)s;
}

// One thread per block; NVFP4 reads its global from g[row / rows_per_global].
// With `tiles` (MXFP8, cols a multiple of 128) the block also goes to the
// slot-major MX FP8 tiles: a token row (tile_slots = pair_pos, top_k > 0) to
// each of its valid slots, a slot row (top_k == 0) to its own slot.
template <int QF, bool BF16>
__global__ void __launch_bounds__(kQThreads)
k_quant_blocks(const void *__restrict__ src, int64_t rows, int64_t cols, int64_t rows_per_global,
               const float *__restrict__ g, uint8_t *__restrict__ codes, uint8_t *__restrict__ scales,
               const int32_t *__restrict__ rows_dev, const int32_t *__restrict__ row_live,
               uint8_t *__restrict__ tiles, const int32_t *__restrict__ tile_slots, int top_k) {
  constexpr int bs = QF == Q_NVFP4 ? 16 : 32;
  pdl_trigger();
  pdl_wait();
  const int64_t nb = cols / bs;
  const int64_t live_rows = rows_dev ? (rows < (int64_t)*rows_dev ? rows : (int64_t)*rows_dev) : rows;
  for (int64_t i = (int64_t)blockIdx.x * kQThreads + threadIdx.x; i < live_rows * nb;
       i += (int64_t)gridDim.x * kQThreads) {
    const int64_t row = i / nb, b = i % nb;
    if (row_live != nullptr && row_live[row] < 0) continue;  // a padding slot of the expert-sorted list
    const int64_t e0 = row * cols + b * bs;
    float x[bs];
#pragma unroll
    for (int j = 0; j < bs; j += 8) load8<BF16>(src, e0 + j, *reinterpret_cast<float(*)[8]>(x + j));
    if (QF == Q_NVFP4) {
      uint2 c;
      uint32_t s;
      nvfp4_block(*reinterpret_cast<float(*)[16]>(x), g[row / rows_per_global], c, s);
      *reinterpret_cast<uint2 *>(codes + e0 / 2) = c;
      scales[i] = (uint8_t)s;
    } else {
      uint32_t c[8], s;
      mx_block<QF>(*reinterpret_cast<float(*)[32]>(x), c, s);
      if (QF == Q_MXFP8) {
        uint4 *dst = reinterpret_cast<uint4 *>(codes + e0);
        dst[0] = make_uint4(c[0], c[1], c[2], c[3]);
        dst[1] = make_uint4(c[4], c[5], c[6], c[7]);
        if (tiles != nullptr) {
          for (int k = 0; k < (top_k > 0 ? top_k : 1); ++k) {
            const int64_t slot = top_k > 0 ? (int64_t)tile_slots[row * top_k + k] : row;
            if (slot >= 0) mx8_tile_put(tiles, slot, b, cols / 128, c, s);
          }
        }
      } else {
        *reinterpret_cast<uint4 *>(codes + e0 / 2) = make_uint4(c[0], c[1], c[2], c[3]);
      }
      scales[i] = (uint8_t)s;
    }
  }
}

template <bool BF16>
__global__ void __launch_bounds__(kQThreads)
k_amax_tensor(const void *__restrict__ src, int64_t elems, float *__restrict__ amax) {
  __shared__ float red[32];
  pdl_trigger();
  pdl_wait();
  const int64_t b = blockIdx.y;
  float m = 0.f;
  for (int64_t j = ((int64_t)blockIdx.x * kQThreads + threadIdx.x) * 8; j < elems;
       j += (int64_t)gridDim.x * kQThreads * 8) {
    float v[8];
    load8<BF16>(src, b * elems + j, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
  }
  m = block_max(m, red);
  // Non-negative floats order like their bit patterns: an integer max is exact and order-free.
  if (threadIdx.x == 0) atomicMax(reinterpret_cast<unsigned *>(amax) + b, __float_as_uint(m));
}

__global__ void k_amax_to_global(float *g, int64_t n) {
  pdl_trigger();
  pdl_wait();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) g[i] = __fdiv_rn(g[i], 2688.0f);
}

// ------------------------------------------------------------- launchers

static int grid_for(int64_t work, int per_cta) {
  int64_t g = (work + per_cta - 1) / per_cta;
  return (int)std::max<int64_t>(1, std::min<int64_t>(g, 152 * 64));
}

cudaError_t launch_quant_rows_nvfp4(const void *src, bool src_bf16, int64_t rows, int64_t cols, uint8_t *codes,
                                    uint8_t *scales, float *g, const int32_t *rows_dev, const int32_t *row_live,
                                    cudaStream_t s, uint8_t *tiles, const int32_t *tile_slots, int top_k) {
  if (rows <= 0) return cudaSuccess;
  if (rows > 0x7FFFFFFF) return cudaErrorInvalidValue;
  if (tiles != nullptr && cols % 256 != 0) return cudaErrorInvalidValue;
  if (cols % 16 != 0) return cudaErrorInvalidValue;
  if (cols > 2048) {  // a CTA per row
    if (src_bf16)
      return launch_pdl(k_quant_rows_nvfp4_cta<true>, dim3((unsigned)rows), dim3(kQThreads), 0, s, src, cols, codes,
                        scales, g, rows_dev, row_live, tiles, tile_slots, top_k);
    return launch_pdl(k_quant_rows_nvfp4_cta<false>, dim3((unsigned)rows), dim3(kQThreads), 0, s, src, cols, codes,
                      scales, g, rows_dev, row_live, tiles, tile_slots, top_k);
  }
  // a warp per row; at most 8 CTAs of 8 warps per SM-sized share of the rows
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((rows + 7) / 8, 152 * 8));
  if (src_bf16)
    return launch_pdl(k_quant_rows_nvfp4<true>, dim3(grid), dim3(kQThreads), 0, s, src, rows, cols, codes, scales, g,
                      rows_dev, row_live, tiles, tile_slots, top_k);
  return launch_pdl(k_quant_rows_nvfp4<false>, dim3(grid), dim3(kQThreads), 0, s, src, rows, cols, codes, scales, g,
                    rows_dev, row_live, tiles, tile_slots, top_k);
}

cudaError_t launch_quant_blocks(int qfmt, const void *src, bool src_bf16, int64_t rows, int64_t cols,
                                int64_t rows_per_global, const float *g, uint8_t *codes, uint8_t *scales,
                                const int32_t *rows_dev, const int32_t *row_live, cudaStream_t s, uint8_t *tiles,
                                const int32_t *tile_slots, int top_k) {
  if (rows <= 0) return cudaSuccess;
  if (tiles != nullptr && (qfmt != Q_MXFP8 || cols % 128 != 0)) return cudaErrorInvalidValue;
  const int bs = qfmt == Q_NVFP4 ? 16 : 32;
  const int grid = grid_for(rows * (cols / bs), kQThreads);
#define QB(QF, B) \
  return launch_pdl(k_quant_blocks<QF, B>, dim3(grid), dim3(kQThreads), 0, s, src, rows, cols, rows_per_global, g, \
                    codes, scales, rows_dev, row_live, tiles, tile_slots, top_k)
  if (qfmt == Q_NVFP4) { if (src_bf16) QB(Q_NVFP4, true); else QB(Q_NVFP4, false); }
  else if (qfmt == Q_MXFP4) { if (src_bf16) QB(Q_MXFP4, true); else QB(Q_MXFP4, false); }
  else if (qfmt == Q_MXFP8) { if (src_bf16) QB(Q_MXFP8, true); else QB(Q_MXFP8, false); }
#undef QB
  return cudaErrorInvalidValue;
}

cudaError_t launch_amax_tensor(const void *src, bool src_bf16, int64_t batch, int64_t elems, float *amax,
                               cudaStream_t s) {
  if (batch <= 0) return cudaSuccess;
  cudaError_t err = cudaMemsetAsync(amax, 0, sizeof(float) * batch, s);
  if (err != cudaSuccess) return err;
  const int64_t gx = (elems / 8 + kQThreads * 4 - 1) / (kQThreads * 4);
  dim3 grid((unsigned)std::max<int64_t>(1, std::min<int64_t>(gx, 1024)), (unsigned)batch);
  if (src_bf16) return launch_pdl(k_amax_tensor<true>, grid, dim3(kQThreads), 0, s, src, elems, amax);
  return launch_pdl(k_amax_tensor<false>, grid, dim3(kQThreads), 0, s, src, elems, amax);
}

cudaError_t launch_amax_to_global(float *g, int64_t n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  return launch_pdl(k_amax_to_global, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, g, n);
}

}  // namespace bqmoe
