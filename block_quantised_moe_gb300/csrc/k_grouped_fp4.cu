// Grouped expert contractions with NVFP4 weights AND NVFP4 activations (W4A4)
// on the block-scaled FP4 tensor-core MMA, for experts with many pairs
// (prefill).
//
// moe.fused_moe's NVFP4-activation mode (b12x project page, section "What's in
// here"; vLLM docs "b12x Linear and MoE Backends", "Supported Configurations"):
// both operands stay E2M1 codes with E4M3 scales per 16 elements, so the MMA
// takes them as they are -- `tcgen05.mma.cta_group::1.kind::mxf4nvf4
// .block_scale.scale_vec::4X`, M=128 N=128 K=64, FP32 accumulation in TMEM:
//
//   D[128 weight rows x 128 tokens] += sum over 4 MMAs of (A * sA)(B * sB)^T per 256-K block
//
// * A: the weights' FP4 tiles (MOE_WFLAG_FP4_TILES): a 16 KB 128-byte-swizzled
//   tile per 128-row block and 256-K block, one bulk copy; no dequantisation.
// * B: the quantised activations of the item's 128 slots (x^ of each slot's
//   token for GEMM1, h^ for GEMM2), which the row quantiser writes as slot-major
//   tiles in the same swizzled layout (16 KB of codes + 2 KB of scales per
//   256-K block): one bulk copy, like A.  Slots past the expert's last pair hold
//   stale values that only reach accumulator columns that are never read.
// * Scale factors: both tiles end in their rows' E4M3 scales as four 512-byte
//   blocks, one per 64-K step, already in the order the MMA reads them from
//   TMEM (32 lanes x 4 columns, lane i column c = the four scales of row
//   i + 32c); they ride in the same bulk copies as the codes.  Four warps, one
//   per TMEM lane quadrant, move them into TMEM with tcgen05.st (the MMA reads
//   the same words in every quadrant); each lane reads 16 consecutive bytes per
//   block, so the shared-memory loads are free of bank conflicts.  (Issuing
//   the moves as tcgen05.cp from the MMA thread puts them in the MMA's own
//   in-order pipe, between the MMAs, and measured slower.)
// * Epilogue: D x the weights' FP32 global x the row's FP32 activation global,
//   then SiLU(g)*u or ReLU^2 (GEMM1) or the topk_weight (GEMM2).
// * Items (128-token tile, 128-row block) come from the per-tile records the
//   routing writes (expert, first slot, live tokens); each role loads the next
//   item's record while it works on the current one.  The copy and MMA roles
//   run their loops on the whole warp and issue from one elected lane, so the
//   operands of the issued instructions are warp-uniform (issued from a
//   single-thread branch, each MMA cost about 130 cycles of issue).
// Every wait is a bounded mbarrier wait; a timeout sets the status flag, and
// the MMA warp drains its MMAs before TMEM is released.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "launch.h"
#include "sync.cuh"
#include "tcgen05.cuh"

namespace bqmoe {

constexpr int kF4EpiWarps = 8;                       // warps 0-7: epilogue (lane quadrant w % 4, column half w / 4)
constexpr int kF4SfWarp0 = 8;                        // warps 8-11: scale factors into TMEM
constexpr int kF4BWarp = 12;                         // activation tile bulk copies
constexpr int kF4AWarp = 13;                         // weight tile bulk copies
constexpr int kF4MmaWarp = 14;                       // MMA issue
constexpr int kF4Threads = (kF4MmaWarp + 1) * 32;
constexpr int kF4N = 128;                            // tokens per tile
constexpr int kF4TileBytes = 16384;                  // 128 rows x 256 K of E2M1
constexpr int kF4SfBytes = 2048;                     // their scales: 4 K steps x 512 bytes in TMEM order
constexpr int kF4StageBytes = kF4TileBytes + kF4SfBytes;  // one operand's ring stage (a multiple of 1024)
constexpr int kF4Stages = 6;                         // A, B and scale-factor ring depth
constexpr int kF4RingBytes = 2 * kF4Stages * kF4StageBytes;
constexpr int kF4AccCols = kF4N;                     // TMEM columns per accumulator (FP32, N tokens)
constexpr int kF4SfCol0 = 2 * kF4AccCols;            // scale-factor stages after the two accumulators
constexpr int kF4SfCols = 32;                        // per stage: A 16 + B 16 (4 K steps x 4 columns)
constexpr int kF4TmemCols = 512;
static_assert(kF4StageBytes % 1024 == 0, "swizzled tiles need 1024-byte aligned stages");
static_assert(kF4SfCol0 + kF4Stages * kF4SfCols <= kF4TmemCols, "TMEM budget");

// Instruction descriptor of kind::mxf4nvf4: A and B E2M1 (format 1), K-major,
// N >> 3 at bit 17, UE4M3 scales (bit 23 = 0), M >> 4 at bit 24, K = 64.
constexpr uint32_t kF4Idesc = (1u << 7) | (1u << 10) | ((uint32_t)(kF4N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);


struct F4Item {
  int e, bp, s0, ntok;
};
__device__ __forceinline__ int4 fp4_record(const GroupedArgs &a, int w, int nblk) { return a.tiles[w / nblk]; }
__device__ __forceinline__ F4Item fp4_item(const int4 r, int w, int nblk) {
  F4Item it;
  it.e = r.x;
  it.s0 = r.y;
  it.ntok = r.z;
  it.bp = w % nblk;
  return it;
}

__device__ __forceinline__ void tc_mma_fp4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t sfa,
                                           uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(kF4Idesc), "r"(sfa), "r"(sfb), "r"(accumulate));
}

template <int STAGE>
__global__ void __launch_bounds__(kF4Threads, 1) k_grouped_fp4(const GroupedArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = (uint32_t)__cvta_generic_to_shared(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;  // swizzled tiles need 1024-byte alignment
  uint8_t *base = smem_raw + (base_s - raw_s);
  const uint32_t ringA = base_s, ringB = base_s + kF4Stages * kF4StageBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(base + kF4RingBytes);
  constexpr int kBars = 6 * kF4Stages + 4 + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kBars);
  const uint32_t afull0 = (uint32_t)__cvta_generic_to_shared(bars);
  const uint32_t aempty0 = afull0 + 8u * kF4Stages;
  const uint32_t bfull0 = aempty0 + 8u * kF4Stages;
  const uint32_t bempty0 = bfull0 + 8u * kF4Stages;
  const uint32_t sfull0 = bempty0 + 8u * kF4Stages;
  const uint32_t sempty0 = sfull0 + 8u * kF4Stages;
  const uint32_t tfull0 = sempty0 + 8u * kF4Stages;  // 2
  const uint32_t tempty0 = tfull0 + 16u;              // 2
  const uint32_t drain = tempty0 + 16u;               // 1

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int i = 0; i < kF4Stages; ++i) {
      mbar_init(afull0 + 8u * i, 1);
      mbar_init(aempty0 + 8u * i, 1);
      mbar_init(bfull0 + 8u * i, 1);
      mbar_init(bempty0 + 8u * i, 1);
      mbar_init(sfull0 + 8u * i, 4);
      mbar_init(sempty0 + 8u * i, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull0 + 8u * b, 1);
      mbar_init(tempty0 + 8u * b, kF4EpiWarps);
    }
    mbar_init(drain, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kF4MmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(tmem_slot)),
                 "n"(kF4TmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int K = a.K;
  const int nkb = K / 256;
  const int nblk = a.n_blocks;
  const int n_large = a.large[0];
  const int W = n_large > 0 ? a.large_tiles[n_large] * nblk : 0;
  // Items (large expert, 128-token tile, 128-row block) dealt round-robin, so
  // that neighbouring CTAs share token tiles and weight blocks in L2.
  const int w0 = blockIdx.x, wstep = gridDim.x;
  const int4 rec0 = w0 < W ? fp4_record(a, w0, nblk) : make_int4(0, 0, 0, 0);
  bool ok = true;
  const bool by_token = a.act_by_token != 0;

  if (warp == kF4AWarp) {
    // ------------------------------------------------------ weight tiles
    {
      int slot = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;
      int4 rec = rec0;
      for (int w = w0; w < W && ok; w += wstep) {
        const F4Item it = fp4_item(rec, w, nblk);
        if (w + wstep < W) rec = fp4_record(a, w + wstep, nblk);
        const uint8_t *tiles = a.codes + (size_t)it.e * a.codes_expert + (size_t)it.bp * nkb * (kF4TileBytes + kF4SfBytes);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!__all_sync(0xffffffffu, mbar_wait(aempty0 + 8u * slot, phase ^ 1u))) {
            ok = false;
            break;
          }
          // the tile's codes and, right after them, its scale words in TMEM order
          if (elect_one()) {
            mbar_expect_tx(afull0 + 8u * slot, kF4StageBytes);
            bulk_g2s(ringA + (uint32_t)slot * kF4StageBytes, tiles + (size_t)kb * kF4StageBytes, kF4StageBytes,
                     afull0 + 8u * slot);
          }
          __syncwarp();
          issued |= 1u << slot;
          issued_parity = (issued_parity & ~(1u << slot)) | (phase << slot);
          if (++slot == kF4Stages) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
      // Never leave with a copy in flight into this CTA's shared memory.
      for (int i = 0; i < kF4Stages; ++i)
        if (issued & (1u << i)) mbar_wait(afull0 + 8u * i, (issued_parity >> i) & 1u);
    }
    __syncwarp();
  } else if (warp == kF4BWarp) {
    // ------------------------------------------------------ activation tiles
    // The activation rows of an item's 128 slots are one slot-major tile per
    // 256-K block (written by the row quantiser; expert groups are padded to
    // 128 slots, so a tile never straddles two experts): one bulk copy each.
    {
      int slot = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;
      const uint8_t *act = reinterpret_cast<const uint8_t *>(a.act);
      pdl_wait();  // the activation tiles come from the preceding kernel
      int4 rec = rec0;
      for (int w = w0; w < W && ok; w += wstep) {
        const F4Item it = fp4_item(rec, w, nblk);
        if (w + wstep < W) rec = fp4_record(a, w + wstep, nblk);
        const uint8_t *tiles = act + (size_t)(it.s0 / kF4N) * nkb * kF4StageBytes;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!__all_sync(0xffffffffu, mbar_wait(bempty0 + 8u * slot, phase ^ 1u))) {
            ok = false;
            break;
          }
          if (elect_one()) {
            mbar_expect_tx(bfull0 + 8u * slot, kF4StageBytes);
            bulk_g2s(ringB + (uint32_t)slot * kF4StageBytes, tiles + (size_t)kb * kF4StageBytes, kF4StageBytes,
                     bfull0 + 8u * slot);
          }
          __syncwarp();
          issued |= 1u << slot;
          issued_parity = (issued_parity & ~(1u << slot)) | (phase << slot);
          if (++slot == kF4Stages) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
      for (int i = 0; i < kF4Stages; ++i)
        if (issued & (1u << i)) mbar_wait(bfull0 + 8u * i, (issued_parity >> i) & 1u);
    }
    __syncwarp();
  } else if (warp >= kF4SfWarp0 && warp < kF4SfWarp0 + 4) {
    // ------------------------------------------------------ scale factors -> TMEM
    // Warp 8 + q writes lane quadrant q; every quadrant gets the same words:
    // per 64-K step t, this lane's 16 bytes of the weight tile's and of the
    // activation tile's scale blocks.
    const int q = warp - kF4SfWarp0;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    int slot = 0;
    uint32_t phase = 0;
    for (int w = w0; w < W && ok; w += wstep) {
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait(sempty0 + 8u * slot, phase ^ 1u) || !mbar_wait(afull0 + 8u * slot, phase) ||
            !mbar_wait(bfull0 + 8u * slot, phase)) {
          ok = false;
          break;
        }
        const uint8_t *sfa = base + slot * kF4StageBytes + kF4TileBytes + lane * 16;
        const uint8_t *sfb = base + (kF4Stages + slot) * kF4StageBytes + kF4TileBytes + lane * 16;
        uint32_t ra[16], rb[16];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint4 va = *reinterpret_cast<const uint4 *>(sfa + 512 * t);
          const uint4 vb = *reinterpret_cast<const uint4 *>(sfb + 512 * t);
          ra[4 * t + 0] = va.x; ra[4 * t + 1] = va.y; ra[4 * t + 2] = va.z; ra[4 * t + 3] = va.w;
          rb[4 * t + 0] = vb.x; rb[4 * t + 1] = vb.y; rb[4 * t + 2] = vb.z; rb[4 * t + 3] = vb.w;
        }
        tc_fence_after();
        const uint32_t col = tmem + lane_base + (uint32_t)(kF4SfCol0 + slot * kF4SfCols);
        tc_st16(col, ra);
        tc_st16(col + 16, rb);
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sfull0 + 8u * slot);
        if (++slot == kF4Stages) {
          slot = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == kF4MmaWarp) {
    // ------------------------------------------------------ MMA issuer
    {
      int sa = 0, li = 0;
      uint32_t pa = 0;
      bool any = false;
      for (int w = w0; w < W && ok; w += wstep, ++li) {
        const int b = li & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(tempty0 + 8u * b, ((li >> 1) & 1) ^ 1u))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(b * kF4AccCols);
        for (int kb = 0; kb < nkb; ++kb) {
          // A, B and scale-factor rings advance together
          const bool got = mbar_wait(afull0 + 8u * sa, pa) && mbar_wait(bfull0 + 8u * sa, pa) &&
                           mbar_wait(sfull0 + 8u * sa, pa);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
            const uint64_t da = umma_desc_sw128(ringA + (uint32_t)sa * kF4StageBytes);
            const uint64_t db = umma_desc_sw128(ringB + (uint32_t)sa * kF4StageBytes);
            const uint32_t sf = tmem + (uint32_t)(kF4SfCol0 + sa * kF4SfCols);
#pragma unroll
            for (int j = 0; j < 4; ++j)  // K = 64 per MMA: 32 bytes of each operand row
              tc_mma_fp4(d, da + 2u * j, db + 2u * j, sf + 4u * j, sf + 16u + 4u * j, (kb > 0 || j > 0) ? 1u : 0u);
            tc_commit(aempty0 + 8u * sa);
            tc_commit(bempty0 + 8u * sa);
            tc_commit(sempty0 + 8u * sa);
          }
          __syncwarp();
          any = true;
          if (++sa == kF4Stages) {
            sa = 0;
            pa ^= 1u;
          }
        }
        if (!ok) break;
        if (elect_one()) tc_commit(tfull0 + 8u * b);
        __syncwarp();
      }
      if (any) {  // all issued MMAs complete before TMEM can be released
        if (elect_one()) tc_commit(drain);
        __syncwarp();
        mbar_wait(drain, 0);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------ epilogue
    const int m = (warp & 3) * 32 + lane;  // accumulator row = TMEM lane
    const int cbase = (warp >> 2) * (kF4N / 2);  // this warp's half of the 128 token columns
    constexpr int kCh = kF4N / 2 / 32;
    pdl_wait();                      // activation globals come from the preceding kernel
    int li = 0;
    int4 rec = rec0;
    for (int w = w0; w < W && ok; w += wstep, ++li) {
      const F4Item it = fp4_item(rec, w, nblk);
      if (w + wstep < W) rec = fp4_record(a, w + wstep, nblk);
      const int b = li & 1;
      // the expert's global scale of this thread's rows (gate / up / single
      // matrix), applied here; the down projection's goes into the column factor
      const float gsel = a.globals[4 * it.e + ((STAGE == STAGE_GATED && (m & 15) >= 8) ? 1 : 0)];
      const float g2 = STAGE == STAGE_DOWN ? a.globals[4 * it.e + 2] : 1.f;
      // Per column (one per lane and 32-column chunk, broadcast with shuffles):
      // the activation row's FP32 global, times the topk weight and the global
      // scale for the down projection -- loaded before the accumulator is ready.
      float c_l[kCh];
      {
        int p_l[kCh];
#pragma unroll
        for (int ch = 0; ch < kCh; ++ch) {
          const int nl = cbase + 32 * ch + lane;
          p_l[ch] = nl < it.ntok ? a.sorted_pair[it.s0 + nl] : -1;
        }
#pragma unroll
        for (int ch = 0; ch < kCh; ++ch) {
          const int nl = cbase + 32 * ch + lane;
          c_l[ch] = 0.f;
          if (p_l[ch] >= 0) {
            const float f = a.act_g[by_token ? (int64_t)(p_l[ch] / a.top_k) : (int64_t)(it.s0 + nl)];
            c_l[ch] = STAGE == STAGE_DOWN ? f * (a.topk_weights[p_l[ch]] * g2) : f;
          }
        }
      }
      if (!mbar_wait(tfull0 + 8u * b, (li >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int blk = it.bp;
      const int tile = 8 * blk + (m >> 4), rr = m & 15;
      float *__restrict__ outp = a.out;
#pragma unroll
      for (int ch = 0; ch < kCh; ++ch) {
        const int c0 = cbase + 32 * ch;
        uint32_t raw[32];
        tc_ld32(tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(b * kF4AccCols + c0), raw);
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(raw[j]) * __shfl_sync(0xffffffffu, c_l[ch], j);
        if (STAGE == STAGE_GATED) {
          // Rows 0-7 of each 16-row group are gate rows, 8-15 the matching up
          // rows; columns go in pairs, each lane evaluating one SiLU per pair
          // (a gate lane the even column, an up lane the odd one).
          const bool up_lane = rr >= 8;
          const int hrow = tile * 8 + (rr & 7);
#pragma unroll
          for (int p = 0; p < 16; ++p) {
            const float x0 = v[2 * p] * gsel, x1 = v[2 * p + 1] * gsel;
            const float other = __shfl_xor_sync(0xffffffffu, up_lane ? x0 : x1, 8);
            const float gate = up_lane ? other : x0, up = up_lane ? x1 : other;
            const int n = c0 + 2 * p + (up_lane ? 1 : 0);
            if (n < it.ntok) outp[(size_t)(it.s0 + n) * a.n_rows + hrow] = silu_f32(gate) * up;
          }
        } else if (STAGE == STAGE_RELU2) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int n = c0 + j;
            const float r = fmaxf(v[j] * gsel, 0.f);
            if (n < it.ntok) outp[(size_t)(it.s0 + n) * a.n_rows + tile * 16 + rr] = r * r;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int n = c0 + j;
            if (n < it.ntok) store_partial(a, (size_t)(it.s0 + n) * a.n_rows + blk * 128 + m, v[j]);
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
  if (warp == kF4MmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kF4TmemCols));
}

static size_t fp4_smem_bytes() { return (size_t)kF4RingBytes + 1024 + 8 * (6 * kF4Stages + 5) + 16; }
static_assert(kF4RingBytes + 1024 + 8 * (6 * kF4Stages + 5) + 16 <= 227 * 1024, "shared memory budget");

bool fp4_tc_supported(int rows_total, int K) { return rows_total % 128 == 0 && K % 256 == 0; }

template <int STAGE>
static cudaError_t launch_fp4_one(const GroupedArgs &a, int rows_total, cudaStream_t s) {
  const size_t smem = fp4_smem_bytes();
  cudaError_t err = cudaFuncSetAttribute(k_grouped_fp4<STAGE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  int dev = 0, sms = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
  GroupedArgs g = a;
  g.n_blocks = rows_total / 128;
  return launch_pdl(k_grouped_fp4<STAGE>, dim3(sms), dim3(kF4Threads), smem, s, g);
}

cudaError_t launch_grouped_fp4(int stage, const GroupedArgs &a, int rows_total, cudaStream_t s) {
  if (!fp4_tc_supported(rows_total, a.K)) return cudaErrorInvalidValue;
  switch (stage) {
    case STAGE_GATED: return launch_fp4_one<STAGE_GATED>(a, rows_total, s);
    case STAGE_RELU2: return launch_fp4_one<STAGE_RELU2>(a, rows_total, s);
    case STAGE_DOWN: return launch_fp4_one<STAGE_DOWN>(a, rows_total, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace bqmoe
