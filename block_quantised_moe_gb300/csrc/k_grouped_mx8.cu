// Grouped expert contractions with MXFP4 weights and MXFP8 activations (W4A8,
// MX) on the block-scaled FP8 tensor-core MMA, for experts with many pairs
// (prefill).
//
// The MX activation mode of the MXFP4 MoE (vLLM docs "b12x Linear and MoE
// Backends", backend selection: MXFP8 activations for MXFP4 MoE; b12x project
// page, "What's in here": w4a8_mx): activations stay E4M3 codes with one E8M0
// scale per 32 elements, and the weights' E2M1 codes are widened to E4M3 (every
// E2M1 value is an E4M3 value) while their E8M0 scales are used as they are, so
// `tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X` (E4M3 x
// E4M3, UE8M0 scales, M=128 N=128 K=32, FP32 accumulation in TMEM) computes
//
//   D[128 weight rows x 128 tokens] += sum over 4 MMAs of (A * sA)(B * sB)^T per 128-K block
//
// with no dequantisation arithmetic at all.
//
// * A: the packed MXFP4 weights (the fragment-order bytes the decode kernel
//   streams; two 64-K steps per 128-K block, one bulk copy into a raw ring).
//   Three groups of four converter warps take every third 128-K block; each
//   widens its rows' codes to E4M3 (cvt to f16x2, then to e4m3x2) and writes
//   the 128-byte-swizzled K-major A tile.  In the packed fragments, lane c of
//   a quad holds, per 32-element block, the elements 16e + 8j + 4h + c of two
//   rows (word j, byte h per row, nibble e); each lane writes its eight codes
//   of a row contiguously (one 8-byte store) at 8c + 4e + 2j + h, i.e. the K
//   order of every 32-element block is transposed as an 8 x 4 matrix (logical
//   4i + c at physical 8c + i).  The activation tiles carry the same order,
//   and a contraction is indifferent to the order of its K.
// * B: the quantised activations of the item's 128 slots (x^ of each slot's
//   token for GEMM1, h^ for GEMM2), which the MXFP8 quantiser writes as
//   slot-major tiles (16 KB of codes, permuted as above, + 512 bytes of scales
//   in TMEM order per 128-K block): one bulk copy per block.
// * Scale factors: scale_vec::1X reads one UE8M0 byte per row per MMA from a
//   32-bit TMEM word (lane i, column c = row i + 32c), the byte chosen by the
//   instruction's scale-factor data ID: MMA j of a 128-K block takes byte j, so
//   one word holds a row's four scales of the block.  The converter warps put
//   the weight words (from the raw ring) and the activation words (from the B
//   stage) into TMEM with tcgen05.st, the same words in every lane quadrant.
// * Epilogue: as the other tcgen05 kernels (ReLU^2 or SiLU(g)*u into h for
//   GEMM1, the topk weight into the BF16 partials for GEMM2).
// * Items (128-token tile, 128-row block) come from the per-tile records the
//   routing writes; the copy and MMA roles run their loops on the whole warp
//   and issue from one elected lane.
// Every wait is a bounded mbarrier wait; a timeout sets the status flag, and
// the MMA warp drains its MMAs before TMEM is released.
#include <algorithm>

#include "common.cuh"
#include "dequant.cuh"
#include "internal.h"
#include "launch.h"
#include "sync.cuh"
#include "tcgen05.cuh"

namespace bqmoe {

constexpr int k8EpiWarps = 8;                      // warps 0-7: epilogue (lane quadrant w % 4, column half w / 4)
constexpr int k8CvtWarp0 = 8;                      // warps 8-19: three groups of four converter warps
constexpr int k8CvtGroups = 3;
constexpr int k8LoadWarp = k8CvtWarp0 + 4 * k8CvtGroups;  // raw weight bulk copies
constexpr int k8BWarp = k8LoadWarp + 1;                   // activation tile bulk copies
constexpr int k8MmaWarp = k8BWarp + 1;                    // MMA issue
constexpr int k8Threads = (k8MmaWarp + 1) * 32;
constexpr int k8N = 128;                           // tokens per tile
constexpr int k8StepBytes = 4352;                  // one 64-K step of a 128-row MXFP4 block (codes + scales)
constexpr int k8RawBytes = 2 * k8StepBytes;        // one 128-K block
constexpr int k8ABytes = 16384;                    // 128 rows x 128 E4M3 codes
constexpr int k8BTileBytes = kMx8TileBytes;        // 16 KB codes + 512 bytes of scales, as written
constexpr int k8BBytes = 17408;                    // its ring stage (a multiple of 1024)
constexpr int k8Stages = 5;                        // A / B / scale-factor ring
constexpr int k8RawStages = 6;
constexpr int k8RingBytes = k8Stages * (k8ABytes + k8BBytes) + k8RawStages * k8RawBytes;
constexpr int k8AccCols = k8N;                     // TMEM columns per accumulator
constexpr int k8SfCol0 = 2 * k8AccCols;            // scale-factor stages after the two accumulators
constexpr int k8SfCols = 8;                        // per stage: A 4 + B 4 (kept 4-column aligned)
constexpr int k8TmemCols = 512;
constexpr int k8Bars = 3 * k8Stages + 2 * k8RawStages + 4 + 1;
static_assert(k8BBytes % 1024 == 0 && k8ABytes % 1024 == 0 && k8BTileBytes <= k8BBytes, "stage alignment");
static_assert(k8SfCol0 + k8Stages * k8SfCols <= k8TmemCols, "TMEM budget");

// kind::mxf8f6f4: A and B E4M3 (type 0), K-major, N >> 3 at bit 17, UE8M0
// scales (bit 23), M >> 4 at bit 24; scale-factor data IDs at bits 4-5 (B)
// and 29-30 (A).
constexpr uint32_t kMx8Idesc = ((uint32_t)(k8N >> 3) << 17) | (1u << 23) | ((uint32_t)(128 >> 4) << 24);

__device__ __forceinline__ void tc_mma_mx8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate));
}

// TMEM store of 4 consecutive 32-bit columns of this warp's 32 lanes.
__device__ __forceinline__ void tc_st4(uint32_t taddr, uint4 v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Two E2M1 codes (a byte, low nibble first) -> two E4M3 codes (low byte first).
__device__ __forceinline__ uint32_t e2m1x2_to_e4m3x2(uint32_t h2) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h2));
  return r;
}

struct Mx8Item {
  int e, bp, s0, ntok;
};
__device__ __forceinline__ int4 mx8_record(const GroupedArgs &a, int w, int nblk) { return a.tiles[w / nblk]; }
__device__ __forceinline__ Mx8Item mx8_item(const int4 r, int w, int nblk) {
  Mx8Item it;
  it.e = r.x;
  it.s0 = r.y;
  it.ntok = r.z;
  it.bp = w % nblk;
  return it;
}

template <int STAGE>
__global__ void __launch_bounds__(k8Threads, 1) k_grouped_mx8(const GroupedArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = (uint32_t)__cvta_generic_to_shared(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;  // swizzled tiles need 1024-byte alignment
  uint8_t *base = smem_raw + (base_s - raw_s);
  const uint32_t ringA = base_s, ringB = base_s + k8Stages * k8ABytes;
  const uint32_t ringR = ringB + k8Stages * k8BBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(base + k8RingBytes);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + k8Bars);
  const uint32_t afull0 = (uint32_t)__cvta_generic_to_shared(bars);  // A tile and both scale words in TMEM
  const uint32_t bfull0 = afull0 + 8u * k8Stages;                    // B tile has landed
  const uint32_t empty0 = bfull0 + 8u * k8Stages;                    // the stage's MMAs have completed
  const uint32_t rfull0 = empty0 + 8u * k8Stages;                    // raw weight bytes have landed
  const uint32_t rempty0 = rfull0 + 8u * k8RawStages;                // a converter group has read them
  const uint32_t tfull0 = rempty0 + 8u * k8RawStages;                // 2
  const uint32_t tempty0 = tfull0 + 16u;                             // 2
  const uint32_t drain = tempty0 + 16u;                              // 1

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int i = 0; i < k8Stages; ++i) {
      mbar_init(afull0 + 8u * i, 4);
      mbar_init(bfull0 + 8u * i, 1);
      mbar_init(empty0 + 8u * i, 1);
    }
    for (int i = 0; i < k8RawStages; ++i) {
      mbar_init(rfull0 + 8u * i, 1);
      mbar_init(rempty0 + 8u * i, 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull0 + 8u * b, 1);
      mbar_init(tempty0 + 8u * b, k8EpiWarps);
    }
    mbar_init(drain, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == k8MmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(tmem_slot)),
                 "n"(k8TmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int K = a.K;
  const int nkb = K / 128;
  const int nblk = a.n_blocks;
  const int n_large = a.large[0];
  const int W = n_large > 0 ? a.large_tiles[n_large] * nblk : 0;
  // Items are dealt round-robin over the CTAs: neighbouring CTAs share token
  // tiles and weight blocks in L2.
  const int w0 = blockIdx.x, wstep = gridDim.x;
  const int4 rec0 = w0 < W ? mx8_record(a, w0, nblk) : make_int4(0, 0, 0, 0);
  const int n_items = w0 < W ? (W - w0 + wstep - 1) / wstep : 0;
  bool ok = true;

  if (warp >= k8CvtWarp0 && warp < k8CvtWarp0 + 4 * k8CvtGroups) {
    // ------------------------------------------------------ converters
    // Group g (warps 8 + 4g .. 11 + 4g) takes the 128-K blocks n with
    // n % 3 == g.  Warp quadrant q handles rows 32q .. 32q + 31 (16-row tiles
    // 2q and 2q + 1): from each 64-K step, lane (r, c) of a tile's fragment
    // chunk holds rows r and r + 8 at K pairs 16j + 2c and 16j + 8 + 2c.
    const int grp = (warp - k8CvtWarp0) >> 2, q = warp & 3;
    const int g = lane >> 2, c4 = lane & 3;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const int total = n_items * nkb;
    for (int n = grp; n < total && ok; n += k8CvtGroups) {
      const int r = n % k8RawStages, st = n % k8Stages;
      const uint32_t rph = (uint32_t)(n / k8RawStages) & 1u, sph = (uint32_t)(n / k8Stages) & 1u;
      // the warp decides together (the TMEM stores below are warp-wide)
      if (!__all_sync(0xffffffffu, mbar_wait(rfull0 + 8u * r, rph))) {
        ok = false;
        break;
      }
      const uint8_t *rawp = base + (ringR - base_s) + (size_t)r * k8RawBytes;
      uint4 cch[2][2];  // [step][tile]
#pragma unroll
      for (int s = 0; s < 2; ++s)
#pragma unroll
        for (int t = 0; t < 2; ++t)
          cch[s][t] = *reinterpret_cast<const uint4 *>(rawp + s * k8StepBytes + (2 * q + t) * 512 + lane * 16);
      // this lane's weight scale words: rows lane + 32c, bytes = the four 32-K blocks
      uint32_t sa[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int R = lane + 32 * c;
        const int off = 4096 + (R >> 4) * 32 + (R & 7) * 4 + 2 * ((R >> 3) & 1);
        const uint32_t lo = *reinterpret_cast<const uint16_t *>(rawp + off);
        const uint32_t hi = *reinterpret_cast<const uint16_t *>(rawp + k8StepBytes + off);
        sa[c] = lo | (hi << 16);
      }
      __syncwarp();  // every lane's reads of the raw stage are done
      if (lane == 0) mbar_arrive(rempty0 + 8u * r);
      // the B stage's scale words land with its tile; the stage is free once
      // the MMAs that read it k8Stages blocks ago have completed
      const bool got_b = mbar_wait(bfull0 + 8u * st, sph);
      const bool got_e = got_b && mbar_wait(empty0 + 8u * st, sph ^ 1u);
      if (!__all_sync(0xffffffffu, got_e)) {
        ok = false;
        break;
      }
      const uint4 sb = *reinterpret_cast<const uint4 *>(base + k8Stages * k8ABytes + (size_t)st * k8BBytes + 16384 +
                                                        lane * 16);
      uint8_t *tileA = base + (size_t)st * k8ABytes;
#pragma unroll
      for (int s = 0; s < 2; ++s)
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const uint32_t cw[4] = {cch[s][t].x, cch[s][t].y, cch[s][t].z, cch[s][t].w};
          // per word j: bytes (r0, h = 0), (r1, h = 0), (r0, h = 1), (r1, h = 1); a byte's
          // nibbles are e = 0, 1 (elements 16e + 8 (j & 1) + 4h + c of block j >> 1)
          uint32_t p[4][4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t h2[4];
            e2m1x8_to_f16x2x4(cw[j], h2);
#pragma unroll
            for (int i = 0; i < 4; ++i) p[j][i] = e2m1x2_to_e4m3x2(h2[i]);
          }
          const int r0 = 16 * (2 * q + t) + g;
#pragma unroll
          for (int half = 0; half < 2; ++half) {  // row r0 or r0 + 8
            const int row = r0 + 8 * half;
#pragma unroll
            for (int b = 0; b < 2; ++b) {  // 32-K block of the step
              // (j, h) bytes of e = 0 then of e = 1, in the order 2j + h
              const uint32_t w0v = p[2 * b][half] | (p[2 * b][2 + half] << 16);
              const uint32_t w1v = p[2 * b + 1][half] | (p[2 * b + 1][2 + half] << 16);
              const int kk = 64 * s + 32 * b + 8 * c4;  // byte within the row's 128
              const int off = (row >> 3) * 1024 + (row & 7) * 128 + ((((kk >> 4) ^ row) & 7) << 4) + (kk & 15);
              *reinterpret_cast<uint2 *>(tileA + off) =
                  make_uint2(__byte_perm(w0v, w1v, 0x6420), __byte_perm(w0v, w1v, 0x7531));
            }
          }
        }
      const uint32_t sf = tmem + lane_base + (uint32_t)(k8SfCol0 + st * k8SfCols);
      tc_st4(sf, make_uint4(sa[0], sa[1], sa[2], sa[3]));
      tc_st4(sf + 4, sb);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(afull0 + 8u * st);
    }
  } else if (warp == k8LoadWarp) {
    // ------------------------------------------------------ raw weight bytes
    // One bulk copy per 128-K block: the two packed 64-K steps of the item's
    // 128-row block are contiguous.
    int r = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, issued_parity = 0;
    int4 rec = rec0;
    for (int w = w0; w < W && ok; w += wstep) {
      const Mx8Item it = mx8_item(rec, w, nblk);
      if (w + wstep < W) rec = mx8_record(a, w + wstep, nblk);
      const uint8_t *src = a.codes + (size_t)it.e * a.codes_expert + (size_t)it.bp * (K / 64) * k8StepBytes;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!__all_sync(0xffffffffu, mbar_wait(rempty0 + 8u * r, phase ^ 1u))) {
          ok = false;
          break;
        }
        if (elect_one()) {
          mbar_expect_tx(rfull0 + 8u * r, k8RawBytes);
          bulk_g2s(ringR + (uint32_t)r * k8RawBytes, src + (size_t)kb * k8RawBytes, k8RawBytes, rfull0 + 8u * r);
        }
        __syncwarp();
        issued |= 1u << r;
        issued_parity = (issued_parity & ~(1u << r)) | (phase << r);
        if (++r == k8RawStages) {
          r = 0;
          phase ^= 1u;
        }
      }
    }
    // Never leave with a copy in flight into this CTA's shared memory.
    for (int i = 0; i < k8RawStages; ++i)
      if (issued & (1u << i)) mbar_wait(rfull0 + 8u * i, (issued_parity >> i) & 1u);
    __syncwarp();
  } else if (warp == k8BWarp) {
    // ------------------------------------------------------ activation tiles
    int st = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, issued_parity = 0;
    const uint8_t *act = reinterpret_cast<const uint8_t *>(a.act);
    pdl_wait();  // the activation tiles come from the preceding kernel
    int4 rec = rec0;
    for (int w = w0; w < W && ok; w += wstep) {
      const Mx8Item it = mx8_item(rec, w, nblk);
      if (w + wstep < W) rec = mx8_record(a, w + wstep, nblk);
      const uint8_t *tiles = act + (size_t)(it.s0 / k8N) * nkb * k8BTileBytes;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!__all_sync(0xffffffffu, mbar_wait(empty0 + 8u * st, phase ^ 1u))) {
          ok = false;
          break;
        }
        if (elect_one()) {
          mbar_expect_tx(bfull0 + 8u * st, k8BTileBytes);
          bulk_g2s(ringB + (uint32_t)st * k8BBytes, tiles + (size_t)kb * k8BTileBytes, k8BTileBytes, bfull0 + 8u * st);
        }
        __syncwarp();
        issued |= 1u << st;
        issued_parity = (issued_parity & ~(1u << st)) | (phase << st);
        if (++st == k8Stages) {
          st = 0;
          phase ^= 1u;
        }
      }
    }
    for (int i = 0; i < k8Stages; ++i)
      if (issued & (1u << i)) mbar_wait(bfull0 + 8u * i, (issued_parity >> i) & 1u);
    __syncwarp();
  } else if (warp == k8MmaWarp) {
    // ------------------------------------------------------ MMA issuer
    int st = 0, li = 0;
    uint32_t ph = 0;
    bool any = false;
    for (int w = w0; w < W && ok; w += wstep, ++li) {
      const int b = li & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(tempty0 + 8u * b, ((li >> 1) & 1) ^ 1u))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem + (uint32_t)(b * k8AccCols);
      for (int kb = 0; kb < nkb; ++kb) {
        const bool got = mbar_wait(afull0 + 8u * st, ph) && mbar_wait(bfull0 + 8u * st, ph);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (elect_one()) {
          const uint64_t da = umma_desc_sw128(ringA + (uint32_t)st * k8ABytes);
          const uint64_t db = umma_desc_sw128(ringB + (uint32_t)st * k8BBytes);
          const uint32_t sf = tmem + (uint32_t)(k8SfCol0 + st * k8SfCols);
#pragma unroll
          for (int j = 0; j < 4; ++j)  // K = 32 per MMA: 32 bytes of each operand row; scale byte j
            tc_mma_mx8(d, da + 2u * j, db + 2u * j, kMx8Idesc | ((uint32_t)j << 4) | ((uint32_t)j << 29), sf, sf + 4,
                       (kb > 0 || j > 0) ? 1u : 0u);
          tc_commit(empty0 + 8u * st);
        }
        __syncwarp();
        any = true;
        if (++st == k8Stages) {
          st = 0;
          ph ^= 1u;
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
    __syncwarp();
  } else {
    // ------------------------------------------------------ epilogue
    const int m = (warp & 3) * 32 + lane;  // accumulator row = TMEM lane
    const int cbase = (warp >> 2) * (k8N / 2);  // this warp's half of the 128 token columns
    pdl_wait();                      // row factors come from the preceding kernels
    int li = 0;
    int4 rec = rec0;
    for (int w = w0; w < W && ok; w += wstep, ++li) {
      const Mx8Item it = mx8_item(rec, w, nblk);
      if (w + wstep < W) rec = mx8_record(a, w + wstep, nblk);
      const int b = li & 1;
      const float gsel = a.globals[4 * it.e + ((STAGE == STAGE_GATED && (m & 15) >= 8) ? 1 : 0)];
      const float g2 = STAGE == STAGE_DOWN ? a.globals[4 * it.e + 2] : 1.f;
      // per column (one per lane and 32-column chunk, broadcast with shuffles):
      // for the down projection the topk weight times the global scale
      float c_l[2];
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const int nl = cbase + 32 * ch + lane;
        c_l[ch] = 1.f;
        if (STAGE == STAGE_DOWN) c_l[ch] = nl < it.ntok ? a.topk_weights[a.sorted_pair[it.s0 + nl]] * g2 : 0.f;
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
      for (int ch = 0; ch < 2; ++ch) {
        const int c0 = cbase + 32 * ch;
        if (c0 >= it.ntok) break;
        uint32_t raw[32];
        tc_ld32(tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(b * k8AccCols + c0), raw);
        if (STAGE == STAGE_GATED) {
          // rows 0-7 of each 16-row group are gate rows, 8-15 the matching up
          // rows; columns in pairs, one SiLU per lane per pair
          const bool up_lane = rr >= 8;
          const int hrow = tile * 8 + (rr & 7);
#pragma unroll
          for (int p = 0; p < 16; ++p) {
            const float x0 = __uint_as_float(raw[2 * p]) * gsel, x1 = __uint_as_float(raw[2 * p + 1]) * gsel;
            const float other = __shfl_xor_sync(0xffffffffu, up_lane ? x0 : x1, 8);
            const float gate = up_lane ? other : x0, up = up_lane ? x1 : other;
            const int n = c0 + 2 * p + (up_lane ? 1 : 0);
            if (n < it.ntok) outp[(size_t)(it.s0 + n) * a.n_rows + hrow] = silu_f32(gate) * up;
          }
        } else if (STAGE == STAGE_RELU2) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int n = c0 + j;
            const float r = fmaxf(__uint_as_float(raw[j]) * gsel, 0.f);
            if (n < it.ntok) outp[(size_t)(it.s0 + n) * a.n_rows + tile * 16 + rr] = r * r;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int n = c0 + j;
            const float v = __uint_as_float(raw[j]) * __shfl_sync(0xffffffffu, c_l[ch], j);
            if (n < it.ntok) store_partial(a, (size_t)(it.s0 + n) * a.n_rows + blk * 128 + m, v);
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
  if (warp == k8MmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(k8TmemCols));
}

static size_t mx8_smem_bytes() { return (size_t)k8RingBytes + 1024 + 8 * k8Bars + 16; }
static_assert(k8RingBytes + 1024 + 8 * k8Bars + 16 <= 227 * 1024, "shared memory budget");

bool mx8_tc_supported(int rows_total, int K) { return rows_total % 128 == 0 && K % 128 == 0; }

template <int STAGE>
static cudaError_t launch_mx8_one(const GroupedArgs &a, int rows_total, cudaStream_t s) {
  const size_t smem = mx8_smem_bytes();
  cudaError_t err = cudaFuncSetAttribute(k_grouped_mx8<STAGE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  int dev = 0, sms = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
  GroupedArgs g = a;
  g.n_blocks = rows_total / 128;
  return launch_pdl(k_grouped_mx8<STAGE>, dim3(sms), dim3(k8Threads), smem, s, g);
}

cudaError_t launch_grouped_mx8(int stage, const GroupedArgs &a, int rows_total, cudaStream_t s) {
  if (!mx8_tc_supported(rows_total, a.K)) return cudaErrorInvalidValue;
  switch (stage) {
    case STAGE_GATED: return launch_mx8_one<STAGE_GATED>(a, rows_total, s);
    case STAGE_RELU2: return launch_mx8_one<STAGE_RELU2>(a, rows_total, s);
    case STAGE_DOWN: return launch_mx8_one<STAGE_DOWN>(a, rows_total, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace bqmoe
