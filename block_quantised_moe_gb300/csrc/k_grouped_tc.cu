// Grouped expert contractions on the 5th-generation tensor cores (tcgen05 with
// TMEM accumulators), for experts that receive many tokens (prefill).
//
// moe.fused_moe with inline FP4 weight dequant (b12x project page, section
// "What's in here").  Once an expert sees more than a few dozen tokens the
// contraction is a dense GEMM, so it runs as tcgen05.mma kind::f16 with FP32
// accumulation in tensor memory:
//
//   D[256 weight rows x 128 tokens] += A[256 x 64] * B[128 x 64]^T per 64-K block
//
// * A: two 128-row blocks of the packed NVFP4 experts (the same packed bytes the
//   decode kernel streams), dequantised by eight producer warps into FP16
//   (E2M1 * E4M3 is exact in FP16) and written in the UMMA K-major 128-byte
//   swizzled layout.
// * B: 128 activation rows of the expert (FP16 rows with a per-row power-of-two
//   factor, staged once per forward), gathered by two producer warps with
//   cp.async (zero-filled past the expert's last token), same layout.
// * One thread of the MMA warp issues 2 x 4 tcgen05.mma (M=128, N=128, K=16)
//   per k-block into two TMEM accumulators and releases the stage with
//   tcgen05.commit; accumulators are double-buffered (512 TMEM columns) so the
//   four epilogue warps (tcgen05.ld, then SiLU(gate)*up or ReLU^2, or the
//   topk_weight scaling of the down projection) overlap the next tile.
// * Work items are (large expert, 128-token tile, pair of row blocks), split
//   evenly over persistent CTAs (one per SM).
// * Every wait is a bounded mbarrier wait; a timeout sets the status flag, and
//   the MMA warp drains its MMAs before TMEM is released.
#include <algorithm>

#include "common.cuh"
#include "dequant.cuh"
#include "internal.h"
#include "launch.h"
#include "sync.cuh"
#include "tcgen05.cuh"

namespace bqmoe {

constexpr int kTcEpiWarps = 4, kTcAWarps = 8, kTcBWarps = 2;
constexpr int kTcMmaWarp = kTcEpiWarps + kTcAWarps + kTcBWarps;  // warp 14
constexpr int kTcThreads = (kTcMmaWarp + 1) * 32;
constexpr int kTcN = 128;                    // tokens per tile
constexpr int kTcMB = 2;                     // 128-row blocks per tile
constexpr int kTcABytes = 128 * 64 * 2;      // one 128 x 64 FP16 block
constexpr int kTcBBytes = kTcN * 64 * 2;     // 128 x 64 FP16
constexpr int kTcAStageBytes = kTcMB * kTcABytes;
constexpr int kTcAStages = 3;                // dequantised A tiles
constexpr int kTcBStages = 6;                // gathered activation tiles
constexpr int kTcBLag = 4;                   // cp.async stages a B thread keeps in flight
constexpr int kTcAPrefetch = 3;              // k-blocks of packed A bytes an A thread keeps in flight
constexpr int kTcRingBytes = kTcAStages * kTcAStageBytes + kTcBStages * kTcBBytes;
constexpr int kTcAccCols = kTcMB * kTcN;     // TMEM columns per accumulator buffer
constexpr int kTcTmemCols = 2 * kTcAccCols;  // double buffered
constexpr int kTcAChunks = kTcMB * 8 * 32 / (kTcAWarps * 32);  // fragment chunks per A thread per k-block
constexpr int kTcBRows = kTcN * 8 / (kTcBWarps * 32);          // 16-byte chunks per B thread per k-block

// ------------------------------------------------------------------ kernel

// WF: W_NVFP4 (FP16 operands) or W_MXFP4 (BF16 operands: E2M1 * 2^X is exact in
// BF16 for any E8M0 X); both read the packed fragment layout.
template <int STAGE, int WF>
__global__ void __launch_bounds__(kTcThreads, 1) k_grouped_tc(const GroupedArgs a) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base for the swizzled tiles
  const uint32_t raw_s = (uint32_t)__cvta_generic_to_shared(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t *base = smem_raw + (base_s - raw_s);
  const uint32_t ringA = base_s, ringB = base_s + kTcAStages * kTcAStageBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(base + kTcRingBytes);
  constexpr int kBars = 2 * kTcAStages + 2 * kTcBStages + 4 + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kBars);
  const uint32_t afull0 = (uint32_t)__cvta_generic_to_shared(bars);
  const uint32_t aempty0 = afull0 + 8u * kTcAStages;
  const uint32_t bfull0 = aempty0 + 8u * kTcAStages;
  const uint32_t bempty0 = bfull0 + 8u * kTcBStages;
  const uint32_t tfull0 = bempty0 + 8u * kTcBStages;  // 2
  const uint32_t tempty0 = tfull0 + 16u;              // 2
  const uint32_t drain = tempty0 + 16u;               // 1

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int i = 0; i < kTcAStages; ++i) {
      mbar_init(afull0 + 8u * i, kTcAWarps);
      mbar_init(aempty0 + 8u * i, 1);
    }
    for (int i = 0; i < kTcBStages; ++i) {
      mbar_init(bfull0 + 8u * i, kTcBWarps);
      mbar_init(bempty0 + 8u * i, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull0 + 8u * b, 1);
      mbar_init(tempty0 + 8u * b, kTcEpiWarps);
    }
    mbar_init(drain, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kTcMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(tmem_slot)),
                 "n"(kTcTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int K = a.K;
  const int nk = K / 64;
  const int nbp = a.n_blocks / kTcMB;
  const int n_large = a.large[0];
  const int W = n_large > 0 ? a.large_tiles[n_large] * nbp : 0;
  // Items are dealt round-robin: at any moment the CTAs work on neighbouring
  // items, which share token tiles and weight blocks in L2.
  const int w0 = blockIdx.x, wstep = gridDim.x;
  TcCursor cur;
  if (w0 < W) cur.seek(a, w0, nbp);
  bool ok = true;

  if (warp >= kTcEpiWarps && warp < kTcEpiWarps + kTcAWarps) {
    // ------------------------------------------------------ A producers
    // The packed fragment chunks (16 code bytes per lane, the lane group's block
    // scales) of two 128-row blocks, dequantised to 16-bit values and written
    // at their slot positions in the swizzled tile: NVFP4 as FP16 (E2M1 x E4M3
    // is exact), MXFP4 as BF16 (E2M1 x 2^X is exact for every E8M0 X).
    constexpr int SB = WF == W_NVFP4 ? 4608 : 4352;  // bytes of one 64-K step of a block
    const int t = threadIdx.x - kTcEpiWarps * 32;  // 0..kTcAWarps*32-1
    int slot = 0;
    uint32_t phase = 0;
    // Software pipeline: the chunks of the next kTcAPrefetch k-blocks (possibly
    // of the next items) are in flight while the current one is dequantised.
    uint4 cch[kTcAChunks], pch[kTcAPrefetch][kTcAChunks];
    uint2 sch[kTcAChunks], psc[kTcAPrefetch][kTcAChunks];
    auto load = [&](const TcItem &it, int kb, uint4 (&c4)[kTcAChunks], uint2 (&s4)[kTcAChunks]) {
      const uint8_t *ebase = a.codes + (size_t)it.e * a.codes_expert;
#pragma unroll
      for (int i = 0; i < kTcAChunks; ++i) {
        const int c = t + kTcAWarps * 32 * i;
        const int blk = 2 * it.bp + (c >> 8), tile = (c >> 5) & 7, ln = c & 31;
        const uint8_t *step = ebase + ((size_t)blk * nk + kb) * SB;
        c4[i] = __ldg(reinterpret_cast<const uint4 *>(step + tile * 512 + ln * 16));
        if (WF == W_NVFP4) s4[i] = __ldg(reinterpret_cast<const uint2 *>(step + 4096 + tile * 64 + (ln >> 2) * 8));
        else s4[i] = make_uint2(__ldg(reinterpret_cast<const uint32_t *>(step + 4096 + tile * 32 + (ln >> 2) * 4)), 0u);
      }
    };
    TcCursor pcur = cur;  // cursor of the prefetch (kTcAPrefetch k-blocks ahead)
    int pw = w0, pkb = 0;
    bool pv = pw < W;
    TcItem pit;
    if (pv) pit = pcur.at(a, pw, nbp);
    auto advance = [&]() {
      if (++pkb == nk) {
        pkb = 0;
        pw += wstep;
        pv = pw < W;
        if (pv) pit = pcur.at(a, pw, nbp);
      }
    };
#pragma unroll
    for (int d = 0; d < kTcAPrefetch; ++d) {
      if (pv) load(pit, pkb, pch[d], psc[d]);
      advance();
    }
    for (int w = w0; w < W && ok; w += wstep) {
      for (int kb = 0; kb < nk; ++kb) {
#pragma unroll
        for (int i = 0; i < kTcAChunks; ++i) {
          cch[i] = pch[0][i];
          sch[i] = psc[0][i];
        }
#pragma unroll
        for (int d = 0; d + 1 < kTcAPrefetch; ++d)
#pragma unroll
          for (int i = 0; i < kTcAChunks; ++i) {
            pch[d][i] = pch[d + 1][i];
            psc[d][i] = psc[d + 1][i];
          }
        if (pv) load(pit, pkb, pch[kTcAPrefetch - 1], psc[kTcAPrefetch - 1]);
        advance();
        if (!mbar_wait(aempty0 + 8u * slot, phase ^ 1u)) {
          ok = false;
          break;
        }
        uint8_t *stA = base + (size_t)slot * kTcAStageBytes;
#pragma unroll
        for (int i = 0; i < kTcAChunks; ++i) {
          const int c = t + kTcAWarps * 32 * i;
          uint8_t *tileA = stA + (c >> 8) * kTcABytes;
          const int tile = (c >> 5) & 7, ln = c & 31;
          const int g = ln >> 2, c4 = ln & 3;
          const int r0 = 16 * tile + g, r1 = r0 + 8;
          const uint32_t cw[4] = {cch[i].x, cch[i].y, cch[i].z, cch[i].w};
          uint32_t o[4][4];  // 16-bit pairs of mma j: (r0, k), (r1, k), (r0, k + 8), (r1, k + 8)
          if (WF == W_NVFP4) {
            uint32_t sp[4];
            e4m3x4_to_f16x2x2(sch[i].x, sp[0], sp[1]);
            e4m3x4_to_f16x2x2(sch[i].y, sp[2], sp[3]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              // scale pairs (block 2(j>>1), block 2(j>>1)+1) of rows r0 and r1, as f16x2
              const uint32_t s_lo = sp[2 * (j >> 1)], s_hi = sp[2 * (j >> 1) + 1];
              uint32_t af[4];
              e2m1x8_to_f16x2x4(cw[j], af);
              o[j][0] = hmul2(af[0], s_lo);
              o[j][1] = hmul2(af[1], s_hi);
              o[j][2] = hmul2(af[2], s_lo);
              o[j][3] = hmul2(af[3], s_hi);
            }
          } else {
            const uint32_t sw = sch[i].x;  // (r0 block 0, r0 block 1, r1 block 0, r1 block 1)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float s_lo = e8m0_to_f32((sw >> (8 * (j >> 1))) & 0xFFu);
              const float s_hi = e8m0_to_f32((sw >> (16 + 8 * (j >> 1))) & 0xFFu);
              uint32_t af[4];
              e2m1x8_to_f16x2x4(cw[j], af);
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(&af[q]));
                const float sc = (q & 1) ? s_hi : s_lo;
                __nv_bfloat162 b2 = __floats2bfloat162_rn(v.x * sc, v.y * sc);
                o[j][q] = *reinterpret_cast<uint32_t *>(&b2);
              }
            }
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int k = 16 * j + 2 * c4;
            *reinterpret_cast<uint32_t *>(tileA + sw128_elem(r0, k)) = o[j][0];
            *reinterpret_cast<uint32_t *>(tileA + sw128_elem(r1, k)) = o[j][1];
            *reinterpret_cast<uint32_t *>(tileA + sw128_elem(r0, k + 8)) = o[j][2];
            *reinterpret_cast<uint32_t *>(tileA + sw128_elem(r1, k + 8)) = o[j][3];
          }
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(afull0 + 8u * slot);
        if (++slot == kTcAStages) {
          slot = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp >= kTcEpiWarps + kTcAWarps && warp < kTcMmaWarp) {
    // ------------------------------------------------------ B producers
    const int t = threadIdx.x - (kTcEpiWarps + kTcAWarps) * 32;  // 0..kTcBWarps*32-1
    const int cc = t & 7;                                        // 16-byte chunk of the row
    constexpr int kRowStep = kTcBWarps * 32 / 8;                 // rows between a thread's chunks
    const bool by_token = a.act_by_token != 0;
    int slot = 0, issued = 0;
    uint32_t phase = 0;
    const __half *act = reinterpret_cast<const __half *>(a.act);
    pdl_wait();  // activation rows come from the preceding kernels
    for (int w = w0; w < W && ok; w += wstep) {
      const TcItem it = cur.at(a, w, nbp);
      int rid[kTcBRows];
#pragma unroll
      for (int i = 0; i < kTcBRows; ++i) {
        const int r = (t >> 3) + kRowStep * i;
        const int s = it.s0 + r;
        rid[i] = r < it.ntok ? (by_token ? a.sorted_pair[s] / a.top_k : s) : -1;
      }
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait(bempty0 + 8u * slot, phase ^ 1u)) {
          ok = false;
          break;
        }
        const uint32_t stB = ringB + (uint32_t)slot * kTcBBytes;
#pragma unroll
        for (int i = 0; i < kTcBRows; ++i) {
          const int r = (t >> 3) + kRowStep * i;
          const uint32_t dst = stB + (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + (((cc ^ r) & 7) << 4));
          const __half *src = act + (int64_t)(rid[i] < 0 ? 0 : rid[i]) * K + kb * 64 + cc * 8;
          cp_async16(dst, src, rid[i] >= 0);
        }
        cp_async_commit();
        ++issued;
        if (issued > kTcBLag) {  // the stage issued kTcBLag steps ago has landed: hand it to the MMA warp
          cp_async_wait_group<kTcBLag>();
          fence_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bfull0 + 8u * ((slot + kTcBStages - kTcBLag) % kTcBStages));
        }
        if (++slot == kTcBStages) {
          slot = 0;
          phase ^= 1u;
        }
      }
    }
    cp_async_wait_group<0>();
    fence_async_smem();
    __syncwarp();
    if (ok && lane == 0) {  // the last kTcBLag stages
      for (int back = issued < kTcBLag ? issued : kTcBLag; back >= 1; --back)
        mbar_arrive(bfull0 + 8u * ((slot + kTcBStages - back) % kTcBStages));
    }
  } else if (warp == kTcMmaWarp) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t fmt = WF == W_MXFP4 ? 1u : 0u;  // operand type: 0 = F16, 1 = BF16
      const uint32_t idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(kTcN >> 3) << 17) |
                             ((uint32_t)(128 >> 4) << 24);
      int sa = 0, sb = 0, li = 0;
      uint32_t pa = 0, pb = 0;
      bool any = false;
      for (int w = w0; w < W && ok; w += wstep, ++li) {
        const int b = li & 1;
        if (!mbar_wait(tempty0 + 8u * b, ((li >> 1) & 1) ^ 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem + (uint32_t)(b * kTcAccCols);
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(afull0 + 8u * sa, pa) || !mbar_wait(bfull0 + 8u * sb, pb)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sta = ringA + (uint32_t)sa * kTcAStageBytes;
          const uint64_t da0 = umma_desc_sw128(sta), da1 = umma_desc_sw128(sta + kTcABytes);
          const uint64_t db = umma_desc_sw128(ringB + (uint32_t)sb * kTcBBytes);
#pragma unroll
          for (int j = 0; j < 4; ++j) {  // K = 16 per MMA: advance the start address by 32 bytes
            const uint32_t acc = (kb > 0 || j > 0) ? 1u : 0u;
            tc_mma_f16(d0, da0 + 2u * j, db + 2u * j, idesc, acc);
            tc_mma_f16(d0 + kTcN, da1 + 2u * j, db + 2u * j, idesc, acc);
          }
          tc_commit(aempty0 + 8u * sa);  // frees both stages once these MMAs have read them
          tc_commit(bempty0 + 8u * sb);
          any = true;
          if (++sa == kTcAStages) {
            sa = 0;
            pa ^= 1u;
          }
          if (++sb == kTcBStages) {
            sb = 0;
            pb ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(tfull0 + 8u * b);
      }
      if (any) {  // all issued MMAs complete before TMEM can be released
        tc_commit(drain);
        mbar_wait(drain, 0);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------ epilogue
    const int m = warp * 32 + lane;  // accumulator row = TMEM lane
    const float *gl_all = a.globals;
    pdl_wait();  // row factors come from the preceding kernels
    int li = 0;
    for (int w = w0; w < W && ok; w += wstep, ++li) {
      const TcItem it = cur.at(a, w, nbp);
      const int b = li & 1;
      if (!mbar_wait(tfull0 + 8u * b, (li >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float *gl = gl_all + 4 * it.e;
      for (int blk_l = 0; blk_l < kTcMB; ++blk_l) {
        const int blk = 2 * it.bp + blk_l;
        const int tile = 8 * blk + (m >> 4), rr = m & 15;
        for (int c0 = 0; c0 < kTcN; c0 += 32) {
          // Column info (slot, activation factor, topk weight) is fetched once per
          // 32-column chunk, one column per lane, and broadcast with shuffles.
          const int nl = c0 + lane;
          const int sl = it.s0 + nl;
          float f_l = 0.f, w_l = 0.f;
          if (nl < it.ntok) {
            const int p = a.sorted_pair[sl];
            f_l = a.act_g ? a.act_g[a.act_by_token ? (int64_t)(p / a.top_k) : (int64_t)sl] : 1.f;
            if (STAGE == STAGE_DOWN) w_l = a.topk_weights[p] * gl[2];
          }
          uint32_t raw[32];
          tc_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(b * kTcAccCols + blk_l * kTcN + c0), raw);
          float hv[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int n = c0 + j;
            const bool live = n < it.ntok;
            const int s = it.s0 + n;
            const float f = __shfl_sync(0xffffffffu, f_l, j);
            const float v = __uint_as_float(raw[j]) * f;
            hv[j] = 0.f;
            if (STAGE == STAGE_GATED) {
              const float up = __shfl_down_sync(0xffffffffu, v, 8);
              if (rr < 8) {
                const float h = silu_f32(v * gl[0]) * (up * gl[1]);
                if (live) a.out[(size_t)s * a.n_rows + tile * 8 + rr] = h;
                hv[j] = fabsf(h);
              }
            } else if (STAGE == STAGE_RELU2) {
              const float r = fmaxf(v * gl[0], 0.f);
              if (live) a.out[(size_t)s * a.n_rows + tile * 16 + rr] = r * r;
              hv[j] = r * r;
            } else {
              const float wt = __shfl_sync(0xffffffffu, w_l, j);
              if (live) store_partial(a, (size_t)s * a.n_rows + blk * 128 + m, wt * v);
            }
          }
          if (STAGE != STAGE_DOWN && a.out_amax != nullptr) {
            // reduce-scatter max over the 32 lanes: lane l ends with column c0 + l
#pragma unroll
            for (int step = 16; step >= 1; step >>= 1) {
              const bool upper = (lane & step) != 0;
#pragma unroll
              for (int j = 0; j < step; ++j) {
                const float send = upper ? hv[j] : hv[j + step];
                const float keep = upper ? hv[j + step] : hv[j];
                hv[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, step));
              }
            }
            const int n = c0 + lane;
            if (n < it.ntok) atomicMax(reinterpret_cast<unsigned *>(a.out_amax) + it.s0 + n, __float_as_uint(hv[0]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8u * b);
    }
  }

  if (!ok && lane == 0) atomicOr(&a.status[ST_FLAGS], ST_FLAG_TIMEOUT);
  pdl_wait();  // completion implies the predecessor's (a no-op for threads that already waited)
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kTcMmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTcTmemCols));
}

static int tc_num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return n;
}

size_t tc_smem_bytes() { return (size_t)kTcRingBytes + 1024 + 8 * (2 * kTcAStages + 2 * kTcBStages + 5) + 16; }

template <int STAGE, int WF>
static cudaError_t launch_tc_one(const GroupedArgs &a, int rows_total, int E, cudaStream_t s) {
  const size_t smem = tc_smem_bytes();
  cudaError_t err = cudaFuncSetAttribute(k_grouped_tc<STAGE, WF>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int sms = tc_num_sms();
  if (sms <= 0) return cudaErrorInvalidDevice;
  GroupedArgs g = a;
  g.n_blocks = rows_total / 128;
  return launch_pdl(k_grouped_tc<STAGE, WF>, dim3(sms), dim3(kTcThreads), smem, s, g);
}

bool tc_supported(int rows_total, int K) { return rows_total % (128 * kTcMB) == 0 && K % 64 == 0; }

template <int WF>
static cudaError_t launch_tc_wf(int stage, const GroupedArgs &a, int rows_total, int E, cudaStream_t s) {
  switch (stage) {
    case STAGE_GATED: return launch_tc_one<STAGE_GATED, WF>(a, rows_total, E, s);
    case STAGE_RELU2: return launch_tc_one<STAGE_RELU2, WF>(a, rows_total, E, s);
    case STAGE_DOWN: return launch_tc_one<STAGE_DOWN, WF>(a, rows_total, E, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_grouped_tc(int stage, int wfmt, const GroupedArgs &a, int rows_total, int E, cudaStream_t s) {
  if (!tc_supported(rows_total, a.K)) return cudaErrorInvalidValue;
  if (wfmt == W_NVFP4) return launch_tc_wf<W_NVFP4>(stage, a, rows_total, E, s);
  if (wfmt == W_MXFP4) return launch_tc_wf<W_MXFP4>(stage, a, rows_total, E, s);
  return cudaErrorInvalidValue;
}

// ------------------------------------------------ h -> FP16 rows for the tc path
//
// One warp per live slot row: FP32 h with the factor from GEMM1's per-pair max |h|,
// NVFP4 (E2M1*E4M3 exact, factor = row global) or MXFP8 (two passes) -> FP16 + factor.
template <int SRC, bool OUT_BF16>
__global__ void __launch_bounds__(256) k_stage_h16(const void *__restrict__ act, const uint8_t *__restrict__ act_scales,
                                                   const float *__restrict__ act_g, int K, int64_t rows,
                                                   const int32_t *__restrict__ rows_dev, __half *__restrict__ h16,
                                                   float *__restrict__ fac) {
  const int lane = threadIdx.x & 31;
  pdl_trigger();
  pdl_wait();
  const int64_t live = rows_dev == nullptr || rows < (int64_t)*rows_dev ? rows : (int64_t)*rows_dev;
  for (int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); row < live; row += (int64_t)gridDim.x * 8) {
    if (OUT_BF16) {  // BF16 slot-order rows, no factor (the MXFP4 path's BF16 operands)
      stage_row_slots<SRC, true>(act, act_scales, row, K, 1.f, h16 + row * K, lane, 32);
      continue;
    }
    float f;
    if (SRC == SRC_H_NVFP4) {
      f = act_g[row];
    } else if (SRC == SRC_H_F32) {
      f = stage_factor(act_g[row]);
    } else {
      float mx = 0.f;
      for (int k = lane * 8; k < K; k += 256) {
        float v[8];
        src_load8<SRC>(act, act_scales, row, k, K, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) mx = fmaxf(mx, fabsf(v[i]));
      }
      f = stage_factor(warp_max(mx));
    }
    const float inv = SRC == SRC_H_NVFP4 ? 1.f : __frcp_rn(f);
    stage_row_slots<SRC>(act, act_scales, row, K, inv, h16 + row * K, lane, 32);
    if (lane == 0) fac[row] = f;
  }
}

cudaError_t launch_stage_h16(int src, const void *act, const uint8_t *act_scales, const float *act_g, int K,
                             int64_t rows, const int32_t *rows_dev, __half *h16, float *fac, bool out_bf16,
                             cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const int grid = (int)std::min<int64_t>((rows + 7) / 8, 152 * 16);
  if (out_bf16) {
    switch (src) {
      case SRC_X_BF16: return launch_pdl(k_stage_h16<SRC_X_BF16, true>, dim3(grid), dim3(256), 0, s, act, act_scales, act_g, K, rows, rows_dev, h16, fac);
      case SRC_H_F32: return launch_pdl(k_stage_h16<SRC_H_F32, true>, dim3(grid), dim3(256), 0, s, act, act_scales, act_g, K, rows, rows_dev, h16, fac);
      case SRC_H_MXFP8: return launch_pdl(k_stage_h16<SRC_H_MXFP8, true>, dim3(grid), dim3(256), 0, s, act, act_scales, act_g, K, rows, rows_dev, h16, fac);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (src) {
    case SRC_H_F32: return launch_pdl(k_stage_h16<SRC_H_F32, false>, dim3(grid), dim3(256), 0, s, act, act_scales, act_g, K, rows, rows_dev, h16, fac);
    case SRC_H_NVFP4: return launch_pdl(k_stage_h16<SRC_H_NVFP4, false>, dim3(grid), dim3(256), 0, s, act, act_scales, act_g, K, rows, rows_dev, h16, fac);
    case SRC_H_MXFP8: return launch_pdl(k_stage_h16<SRC_H_MXFP8, false>, dim3(grid), dim3(256), 0, s, act, act_scales, act_g, K, rows, rows_dev, h16, fac);
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace bqmoe
