// Per-token combine of the expert outputs, and the one-time weight packer.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "launch.h"

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

// Eight consecutive partials as FP32 (one 16-byte BF16 load, or two FP32 ones).
template <bool BF16>
__device__ __forceinline__ void load_part8(const void *part, size_t idx, float (&v)[8]) {
  if (BF16) {
    const uint4 r = __ldcs(reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(part) + idx));
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  } else {
    const float4 a = __ldcs(reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(part) + idx));
    const float4 b = __ldcs(reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(part) + idx) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

// Grid (column chunks of 8 * kCombThreads, token groups); each block loops over
// tokens blockIdx.y, blockIdx.y + gridDim.y, ... (one resident wave; a block per
// token made the kernel bound by block launches at large T).  The next token's
// pair_pos row is fetched while the current token's partials load.
template <bool BF16>
__global__ void __launch_bounds__(kCombThreads)
k_combine(const void *__restrict__ part, int H, const int32_t *__restrict__ pair_pos, int T, int K,
          void *__restrict__ out, int out_f32) {
  pdl_trigger();
  const int c = (blockIdx.x * kCombThreads + threadIdx.x) * 8;
  if (c >= H) {
    pdl_wait();
    return;
  }
  // pair_pos row of the block's next token, fetched one token ahead; routing
  // output, complete when this kernel starts, so the first row is in flight
  // while the partials are still being written
  int ids[kMaxK];
#pragma unroll
  for (int k = 0; k < kMaxK; ++k) ids[k] = (k < K && blockIdx.y < T) ? __ldg(pair_pos + (size_t)blockIdx.y * K + k) : -1;
  pdl_wait();  // the partials come from the preceding kernel
  for (int t = blockIdx.y; t < T; t += gridDim.y) {
    int pos[kMaxK];
    int n = 0;
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
      const int p = ids[k];
      if (p < 0) continue;
      int j = n++;
      while (j > 0 && pos[j - 1] > p) { pos[j] = pos[j - 1]; --j; }
      pos[j] = p;
    }
    const int tn = t + gridDim.y;
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) ids[k] = (k < K && tn < T) ? __ldg(pair_pos + (size_t)tn * K + k) : -1;
    // ordered sum in chunks of 8 partials (the chunk's loads all in flight first;
    // BF16 partials stay packed until the sum, which halves their registers)
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int i0 = 0; i0 < n; i0 += 8) {
      if (BF16) {
        uint4 raw[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (i0 + i < n)
            raw[i] = __ldcs(reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(part) +
                                                            (size_t)pos[i0 + i] * H + c));
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (i0 + i < n) {
            const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              acc[2 * e] += __uint_as_float(w[e] << 16);
              acc[2 * e + 1] += __uint_as_float(w[e] & 0xFFFF0000u);
            }
          }
      } else {
        float v[8][8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (i0 + i < n) load_part8<false>(part, (size_t)pos[i0 + i] * H + c, v[i]);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (i0 + i < n) {
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] += v[i][e];
          }
      }
    }
    if (out_f32) {  // a rank's partial of a tensor-parallel layer, summed across ranks before rounding
      float4 *o4 = reinterpret_cast<float4 *>(reinterpret_cast<float *>(out) + (size_t)t * H + c);
      o4[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      o4[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else {
      __align__(16) __nv_bfloat162 o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) o[e] = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
      *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(out) + (size_t)t * H + c) =
          *reinterpret_cast<const uint4 *>(o);
    }
  }
}

cudaError_t launch_combine(const void *part, bool part_bf16, int H, const int32_t *pair_pos, int T, int K, void *out,
                           bool out_f32, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (K > kMaxK || H % 8) return cudaErrorInvalidValue;
  // one resident wave of blocks, each looping over its tokens; the SM count and
  // occupancy are looked up once per device (under a lock: several host threads
  // may launch forwards on different devices)
  constexpr int kMaxDev = 64;
  static std::mutex mu;
  static int dev_sms[kMaxDev], dev_occ[kMaxDev][2];
  int dev = 0, sms = 0, occ[2] = {0, 0};
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= kMaxDev || dev_sms[dev] == 0) {
      if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ[0], k_combine<false>, kCombThreads, 0) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ[1], k_combine<true>, kCombThreads, 0) != cudaSuccess)
        return cudaErrorUnknown;
      if (dev < kMaxDev) {
        dev_sms[dev] = sms;
        dev_occ[dev][0] = occ[0];
        dev_occ[dev][1] = occ[1];
      }
    } else {
      sms = dev_sms[dev];
      occ[0] = dev_occ[dev][0];
      occ[1] = dev_occ[dev][1];
    }
  }
  const int gx = (H + kCombThreads * 8 - 1) / (kCombThreads * 8);
  const int gy = std::max(1, std::min(T, sms * std::max(1, occ[part_bf16 ? 1 : 0]) / gx));
  if (part_bf16)
    return launch_pdl(k_combine<true>, dim3(gx, gy), dim3(kCombThreads), 0, s, part, H, pair_pos, T, K, out,
                      out_f32 ? 1 : 0);
  return launch_pdl(k_combine<false>, dim3(gx, gy), dim3(kCombThreads), 0, s, part, H, pair_pos, T, K, out,
                    out_f32 ? 1 : 0);
}

// ------------------------------------------------------------------- packer
//
// One-time preparation of the experts (b12x project page, section "Using it":
// fused_moe.prepare_weights, run once per model).  The packed
// buffer holds W13 and W2 re-tiled for the tensor-core kernels (below) in
// 256-byte aligned segments, and the global scales gathered into an [E][4]
// FP32 table (gate|w1, up, down, 1); MXFP4 has no globals and gets 1.0.
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

// Experts are re-tiled for the tensor-core kernels.  Rows are grouped in
// 128-row blocks of eight 16-row tiles; for every 64-wide K step a block stores
// 4096 bytes of codes (tile-major, 32 lanes x 16 bytes in mma.m16n8k16
// A-fragment order) then the block scales: NVFP4 512 bytes (tile-major, 8
// groups x 8 bytes; 4608 per step), MXFP4 256 bytes (8 groups x 4 bytes; 4352).  The K order inside a step is the "slot order" (the
// activations are staged in the same order): the two codes of every fragment
// register come from two different 16-element scale blocks, so a register's
// f16x2 scale multiplier is the conversion of two adjacent scale bytes.  Lane t
// (g = t/4, c = t%4), mma i, byte j of a code chunk: tile row g (+8 for j odd),
// m = c + 4 * (j >> 1); low nibble = code at K offset 64q + 32(i >> 1) + 8(i & 1)
// + m (block 2(i >> 1)), high nibble = the code 16 further (the next block).
// NVFP4 scale group g: bytes (s[g][4q], s[g][4q+1], s[g+8][4q], s[g+8][4q+1],
// s[g][4q+2], s[g][4q+3], s[g+8][4q+2], s[g+8][4q+3]).  MXFP4 (32-element
// blocks; mma 0-1 of a step lie in block 2q, mma 2-3 in block 2q+1):
// (s[g][2q], s[g][2q+1], s[g+8][2q], s[g+8][2q+1]).
// For gated W13, tile t's rows 0..7 are gate features 8t..8t+7 and rows 8..15
// the up rows of the same features; otherwise tile rows are consecutive rows.
// A block's K steps are contiguous, so the kernel streams a block with 1-D bulk
// copies.
// Bytes of one 64-K step of a 128-row block: codes, then the block scales.
__host__ __device__ constexpr int64_t mma_step_bytes(int bs) { return 4096 + 128 * 64 / bs; }

__device__ __forceinline__ int64_t tile_src_row(int tile, int rr, int gated, int I) {
  if (gated) return rr < 8 ? (int64_t)tile * 8 + rr : (int64_t)I + tile * 8 + rr - 8;
  return (int64_t)tile * 16 + rr;
}

// byte offset of (expert, 16-row tile, K step) inside a stage's packed segment
__device__ __forceinline__ int64_t mma_step_base(int64_t e, int tile, int q, int ntiles, int nsteps, int bs) {
  const int nblk = ntiles / 8;
  return ((e * nblk + tile / 8) * nsteps + q) * mma_step_bytes(bs);
}

__global__ void k_pack_mma_codes(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst, int E, int rows, int K,
                                 int gated, int I, int bs) {
  const int nsteps = K / 64, ntiles = rows / 16;
  const int64_t n_chunks = (int64_t)E * ntiles * nsteps * 32;
  const int64_t row_bytes = K / 2;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n_chunks;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(idx & 31);
    int64_t r = idx >> 5;
    const int q = (int)(r % nsteps);
    r /= nsteps;
    const int tile = (int)(r % ntiles);
    const int64_t e = r / ntiles;
    const int g = t >> 2, c = t & 3;
    const uint8_t *se = src + e * rows * row_bytes;
    const int64_t row_lo = tile_src_row(tile, g, gated, I), row_hi = tile_src_row(tile, g + 8, gated, I);
    auto code = [&](int64_t row, int k) { return (uint32_t)(se[row * row_bytes + k / 2] >> (4 * (k & 1))) & 0xFu; };
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w[i] = 0u;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t row = (j & 1) ? row_hi : row_lo;
        const int k = 64 * q + 32 * (i >> 1) + 8 * (i & 1) + c + 4 * (j >> 1);
        w[i] |= (code(row, k) | (code(row, k + 16) << 4)) << (8 * j);
      }
    }
    uint8_t *d = dst + mma_step_base(e, tile, q, ntiles, nsteps, bs) + (tile % 8) * 512 + t * 16;
    *reinterpret_cast<uint4 *>(d) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

template <int BS>
__global__ void k_pack_mma_scales(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst, int E, int rows, int K,
                                  int gated, int I) {
  const int nsteps = K / 64, ntiles = rows / 16;
  const int64_t n_groups = (int64_t)E * ntiles * nsteps * 8;
  const int64_t row_bytes = K / BS;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n_groups;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int g = (int)(idx & 7);
    int64_t r = idx >> 3;
    const int q = (int)(r % nsteps);
    r /= nsteps;
    const int tile = (int)(r % ntiles);
    const int64_t e = r / ntiles;
    const uint8_t *se = src + e * rows * row_bytes;
    const int64_t row_lo = tile_src_row(tile, g, gated, I), row_hi = tile_src_row(tile, g + 8, gated, I);
    constexpr int per_step = 64 / BS;  // block scales per row and K step
    auto sc = [&](int64_t row, int b) { return (uint32_t)se[row * row_bytes + per_step * q + b]; };
    uint8_t *d = dst + mma_step_base(e, tile, q, ntiles, nsteps, BS) + 4096 + (tile % 8) * 8 * 2 * per_step +
                 g * 2 * per_step;
    if (BS == 16) {
      const uint32_t w[2] = {sc(row_lo, 0) | sc(row_lo, 1) << 8 | sc(row_hi, 0) << 16 | sc(row_hi, 1) << 24,
                             sc(row_lo, 2) | sc(row_lo, 3) << 8 | sc(row_hi, 2) << 16 | sc(row_hi, 3) << 24};
      *reinterpret_cast<uint2 *>(d) = make_uint2(w[0], w[1]);
    } else {
      *reinterpret_cast<uint32_t *>(d) = sc(row_lo, 0) | sc(row_lo, 1) << 8 | sc(row_hi, 0) << 16 | sc(row_hi, 1) << 24;
    }
  }
}

// FP4 tiles for the block-scaled tensor-core kernel (MOE_WFLAG_FP4_TILES).  For
// every (expert, 128-row block, 256-K block): 16384 bytes of E2M1 codes, rows of
// 128 bytes (K order as in the checkpoint) in the UMMA 128-byte-swizzled K-major
// layout (16-byte chunk c of row r at (r/8)*1024 + (r%8)*128 + ((c ^ r) % 8)*16),
// then 2048 bytes of E4M3 block scales as 32-bit words (four 16-element blocks
// of one row and one 64-K step, first block in the low byte) ordered
// [step t][lane i][column c] for row i + 32c: per 64-K step one 512-byte block
// in the tensor-memory scale layout (32 lanes x 4 columns per 128 rows), which
// the MMA copies into TMEM as it is.  Rows follow
// the same 8 gate + 8 up interleave per 16-row tile as the fragment layout.
constexpr int64_t kFp4Tile = 16384 + 2048;

__global__ void k_pack_fp4_codes(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst, int E, int rows, int K,
                                 int gated, int I) {
  const int nblk = rows / 128, nkb = K / 256;
  const int64_t n = (int64_t)E * nblk * nkb * 128 * 8;  // 16-byte chunks
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(idx & 7), r = (int)((idx >> 3) & 127);
    int64_t t = idx >> 10;
    const int kb = (int)(t % nkb);
    t /= nkb;
    const int blk = (int)(t % nblk);
    const int64_t e = t / nblk;
    const int64_t row = tile_src_row(blk * 8 + r / 16, r % 16, gated, I);
    const uint4 v = *reinterpret_cast<const uint4 *>(src + (e * rows + row) * (K / 2) + (int64_t)kb * 128 + c * 16);
    uint8_t *tile = dst + ((e * nblk + blk) * nkb + kb) * kFp4Tile;
    *reinterpret_cast<uint4 *>(tile + (r >> 3) * 1024 + (r & 7) * 128 + (((c ^ r) & 7) << 4)) = v;
  }
}

__global__ void k_pack_fp4_scales(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst, int E, int rows, int K,
                                  int gated, int I) {
  const int nblk = rows / 128, nkb = K / 256;
  const int64_t n = (int64_t)E * nblk * nkb * 512;  // 32-bit words
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += (int64_t)gridDim.x * blockDim.x) {
    const int w = (int)(idx & 511);
    const int st = w >> 7, i = (w >> 2) & 31, c = w & 3;
    int64_t t = idx >> 9;
    const int kb = (int)(t % nkb);
    t /= nkb;
    const int blk = (int)(t % nblk);
    const int64_t e = t / nblk;
    const int r = i + 32 * c;
    const int64_t row = tile_src_row(blk * 8 + r / 16, r % 16, gated, I);
    const uint32_t v = *reinterpret_cast<const uint32_t *>(src + (e * rows + row) * (K / 16) + (int64_t)kb * 16 + st * 4);
    uint8_t *tile = dst + ((e * nblk + blk) * nkb + kb) * kFp4Tile;
    reinterpret_cast<uint32_t *>(tile + 16384)[w] = v;
  }
}

static int pack_grid(int64_t n) { return (int)std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, 152 * 32)); }

cudaError_t launch_pack(const WeightLayout &L, const void *w13_codes, const void *w13_scales, const float *w13_global,
                        const void *w2_codes, const void *w2_scales, const float *w2_global, uint8_t *packed,
                        cudaStream_t s) {
  const int gated = L.n13 == 2 * L.I;
  const int64_t c13 = (int64_t)L.E * (L.n13 / 16) * (L.H / 64) * 32, g13 = c13 / 4;
  const int64_t c2 = (int64_t)L.E * (L.H / 16) * (L.I / 64) * 32, g2 = c2 / 4;
  const auto *w13c = static_cast<const uint8_t *>(w13_codes), *w2c = static_cast<const uint8_t *>(w2_codes);
  const auto *w13s = static_cast<const uint8_t *>(w13_scales), *w2s = static_cast<const uint8_t *>(w2_scales);
  k_pack_mma_codes<<<pack_grid(c13), 256, 0, s>>>(w13c, packed + L.off_c13, L.E, L.n13, L.H, gated, L.I, L.bs);
  k_pack_mma_codes<<<pack_grid(c2), 256, 0, s>>>(w2c, packed + L.off_c2, L.E, L.H, L.I, 0, L.I, L.bs);
  if (L.bs == 16) {
    k_pack_mma_scales<16><<<pack_grid(g13), 256, 0, s>>>(w13s, packed + L.off_c13, L.E, L.n13, L.H, gated, L.I);
    k_pack_mma_scales<16><<<pack_grid(g2), 256, 0, s>>>(w2s, packed + L.off_c2, L.E, L.H, L.I, 0, L.I);
  } else {
    k_pack_mma_scales<32><<<pack_grid(g13), 256, 0, s>>>(w13s, packed + L.off_c13, L.E, L.n13, L.H, gated, L.I);
    k_pack_mma_scales<32><<<pack_grid(g2), 256, 0, s>>>(w2s, packed + L.off_c2, L.E, L.H, L.I, 0, L.I);
  }
  if (L.fp4_tiles) {
    const int64_t t13 = (int64_t)L.E * (L.n13 / 128) * (L.H / 256), t2 = (int64_t)L.E * (L.H / 128) * (L.I / 256);
    k_pack_fp4_codes<<<pack_grid(t13 * 1024), 256, 0, s>>>(w13c, packed + L.off_t13, L.E, L.n13, L.H, gated, L.I);
    k_pack_fp4_scales<<<pack_grid(t13 * 512), 256, 0, s>>>(w13s, packed + L.off_t13, L.E, L.n13, L.H, gated, L.I);
    k_pack_fp4_codes<<<pack_grid(t2 * 1024), 256, 0, s>>>(w2c, packed + L.off_t2, L.E, L.H, L.I, 0, L.I);
    k_pack_fp4_scales<<<pack_grid(t2 * 512), 256, 0, s>>>(w2s, packed + L.off_t2, L.E, L.H, L.I, 0, L.I);
  }
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  k_pack_globals<<<(L.E + 127) / 128, 128, 0, s>>>(w13_global, L.n13 / L.I, w2_global, L.E,
                                                     reinterpret_cast<float *>(packed + L.off_g));
  return cudaGetLastError();
}

}  // namespace bqmoe
