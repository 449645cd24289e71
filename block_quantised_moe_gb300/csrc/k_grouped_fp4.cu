// Grouped expert contractions with NVFP4 weights AND NVFP4 activations (W4A4)
// on the block-scaled FP4 tensor-core MMA, for experts with many pairs
// (prefill).
//
// moe.fused_moe's NVFP4-activation mode (b12x project page, section "What's in
// here"; vLLM docs "b12x Linear and MoE Backends", "Supported Configurations"):
// both operands stay E2M1 codes with E4M3 scales per 16 elements, so the MMA
// takes them as they are.  Two CTAs of a cluster form one MMA,
// `tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X`, M=256
// N=128 K=64, FP32 accumulation in TMEM:
//
//   D[256 weight rows x 128 tokens] += sum over 4 MMAs of (A * sA)(B * sB)^T per 256-K block
//
// Nothing is dequantised, so the kernel is bound by the rate at which operand
// bytes land in shared memory: a single CTA with M=128 drew 36 KB per 256-K
// block for 256 cycles of MMA and never got its ring of bulk copies to turn
// over fast enough.  On a pair each CTA draws its own weight rows and half of
// the token tile, 28 KB for the same MMA time.
//
// * A: each CTA's 128-row block of the weights' FP4 tiles (MOE_WFLAG_FP4_TILES):
//   a 16 KB 128-byte-swizzled tile per 256-K block plus its 2 KB of scales,
//   one bulk copy; the pair's blocks are 2p and 2p + 1.
// * B: the quantised activations of the item's 128 slots (x^ of each slot's
//   token for GEMM1, h^ for GEMM2), which the row quantiser writes as slot-major
//   tiles in the same layout (16 KB of codes + 2 KB of scales per 256-K block).
//   CTA r copies rows [64 r, 64 r + 64) of the codes (8 KB, whole 1 KB swizzle
//   atoms) and all 2 KB of scales.  Slots past the expert's last pair hold
//   stale values that only reach accumulator columns that are never read.
// * Scale factors: both tiles end in their rows' E4M3 scales as four 512-byte
//   blocks, one per 64-K step, already in the order the MMA reads them from
//   TMEM (32 lanes x 4 columns, lane i column c = the four scales of row
//   i + 32c).  Each CTA holds the scales of its own 128 weight rows and those
//   of all 128 token rows, at the same TMEM columns in both CTAs.  Four warps
//   per CTA, one per TMEM lane quadrant, move them into TMEM with tcgen05.st
//   (the MMA reads the same words in every quadrant).
// * A relay thread in each CTA turns "this CTA's stage is complete" (operands
//   landed, scale factors in TMEM) into one arrival on the leader's ready
//   barrier; the leader's MMA warp issues the stage's four MMAs from an
//   elected lane and releases it in both CTAs with one multicast commit.
// * Epilogue (both CTAs): D x the weights' FP32 global x the row's FP32
//   activation global, then SiLU(g)*u or ReLU^2 (GEMM1) or the topk_weight
//   (GEMM2); two 128-column accumulators, so it overlaps the next item's MMAs.
// * Items (128-token tile, pair of 128-row blocks) come from the per-tile
//   records the routing writes (expert, first slot, live tokens), dealt
//   round-robin over persistent clusters; each role loads the next item's
//   record while it works on the current one.  The copy and MMA roles run
//   their loops on the whole warp and issue from one elected lane.
// * One release barrier per ring stage, shared by the A, B and scale-factor
//   producers (the three rings advance together): one commit per stage (with
//   a commit per ring the single-CTA kernel's GEMM1 took 10 % longer).
// Every wait is a bounded mbarrier wait; a timeout sets the status flag, every
// CTA still reaches the final cluster barrier, and the leader drains its MMAs
// before the pair's TMEM is released.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "launch.h"
#include "sync.cuh"
#include "tcgen05.cuh"

namespace bqmoe {

constexpr int kP4EpiWarps = 8;                       // warps 0-7: epilogue (lane quadrant w % 4, column half w / 4)
constexpr int kP4SfWarp0 = 8;                        // warps 8-11: scale factors into TMEM
constexpr int kP4BWarp = 12;                         // activation tile bulk copies
constexpr int kP4AWarp = 13;                         // weight tile bulk copies
constexpr int kP4MmaWarp = 14;                       // MMA issue (leader CTA)
constexpr int kP4RelayWarp = 15;                     // stage-complete relay to the leader
constexpr int kP4Threads = (kP4RelayWarp + 1) * 32;
constexpr int kP4N = 128;                            // tokens per tile
constexpr int kP4TileBytes = 16384;                  // 128 rows x 256 K of E2M1
constexpr int kP4SfBytes = 2048;                     // their scales: 4 K steps x 512 bytes in TMEM order
constexpr int kP4AStageBytes = kP4TileBytes + kP4SfBytes;   // a CTA's weight tile and its scales
constexpr int kP4BHalfBytes = kP4TileBytes / 2;             // 64 token rows of codes
constexpr int kP4BStageBytes = kP4BHalfBytes + kP4SfBytes;  // ... and the scales of all 128 token rows
constexpr int kP4Stages = 8;
constexpr int kP4RingBytes = kP4Stages * (kP4AStageBytes + kP4BStageBytes);
constexpr int kP4AccCols = kP4N;                     // TMEM columns per accumulator (FP32, N tokens)
constexpr int kP4SfCol0 = 2 * kP4AccCols;            // scale-factor stages after the two accumulators
constexpr int kP4SfCols = 32;                        // per stage: A 16 + B 16 (4 K steps x 4 columns)
constexpr int kP4TmemCols = 512;
constexpr int kP4Bars = 5 * kP4Stages + 4 + 1;
static_assert(kP4AStageBytes % 1024 == 0 && kP4BStageBytes % 1024 == 0, "swizzled tiles need 1024-byte aligned stages");
static_assert(kP4SfCol0 + kP4Stages * kP4SfCols <= kP4TmemCols, "TMEM budget");
static_assert(kP4SfCols % 4 == 0 && kP4SfCol0 % 4 == 0, "scale-factor TMEM addresses are 4-column aligned");

// Instruction descriptor of kind::mxf4nvf4: A and B E2M1 (format 1), K-major,
// N >> 3 at bit 17, UE4M3 scales (bit 23 = 0), M >> 4 at bit 24 (M = 256 over
// the pair), K = 64.
constexpr uint32_t kP4Idesc = (1u << 7) | (1u << 10) | ((uint32_t)(kP4N >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);

struct F4Item {
  int e, bp, s0, ntok;
};
__device__ __forceinline__ int4 fp4_record(const GroupedArgs &a, int w, int nbp) { return a.tiles[w / nbp]; }
__device__ __forceinline__ F4Item fp4_item(const int4 r, int w, int nbp) {
  F4Item it;
  it.e = r.x;
  it.s0 = r.y;
  it.ntok = r.z;
  it.bp = w % nbp;
  return it;
}

__device__ __forceinline__ void tc2_mma_fp4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t sfa,
                                            uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(kP4Idesc), "r"(sfa), "r"(sfb), "r"(accumulate));
}

template <int STAGE>
__global__ void __launch_bounds__(kP4Threads, 1) k_grouped_fp4(const GroupedArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = (uint32_t)__cvta_generic_to_shared(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;  // swizzled tiles need 1024-byte alignment
  uint8_t *base = smem_raw + (base_s - raw_s);
  const uint32_t ringA = base_s, ringB = base_s + kP4Stages * kP4AStageBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(base + kP4RingBytes);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kP4Bars);
  const uint32_t afull0 = (uint32_t)__cvta_generic_to_shared(bars);  // this CTA's weight tile has landed
  const uint32_t bfull0 = afull0 + 8u * kP4Stages;                   // this CTA's activation half has landed
  const uint32_t sfull0 = bfull0 + 8u * kP4Stages;                   // this CTA's scale factors are in TMEM
  const uint32_t empty0 = sfull0 + 8u * kP4Stages;                   // the pair's MMAs have read the stage
  const uint32_t ready0 = empty0 + 8u * kP4Stages;                   // leader: both CTAs' stages complete
  const uint32_t tfull0 = ready0 + 8u * kP4Stages;                   // 2
  const uint32_t tempty0 = tfull0 + 16u;                             // 2 (leader)
  const uint32_t drain = tempty0 + 16u;                              // 1

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();  // 0: leader (issues the MMAs), 1: peer
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int i = 0; i < kP4Stages; ++i) {
      mbar_init(afull0 + 8u * i, 1);
      mbar_init(bfull0 + 8u * i, 1);
      mbar_init(sfull0 + 8u * i, 4);
      mbar_init(empty0 + 8u * i, 1);
      mbar_init(ready0 + 8u * i, 2);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull0 + 8u * b, 1);
      mbar_init(tempty0 + 8u * b, 2 * kP4EpiWarps);
    }
    mbar_init(drain, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kP4MmaWarp) {  // one warp of each CTA of the pair allocates, together
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(tmem_slot)),
                 "n"(kP4TmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int K = a.K;
  const int nkb = K / 256;
  const int nbp = a.n_blocks / 2;
  const int n_large = a.large[0];
  const int W = n_large > 0 ? a.large_tiles[n_large] * nbp : 0;
  // Items (large expert, 128-token tile, pair of 128-row blocks) dealt
  // round-robin over clusters, so that neighbouring pairs share token tiles
  // and weight blocks in L2.
  const int w0 = (int)cluster_id_x(), wstep = (int)cluster_count_x();
  const int4 rec0 = w0 < W ? fp4_record(a, w0, nbp) : make_int4(0, 0, 0, 0);
  bool ok = true;
  bool any_mma = false;
  const bool by_token = a.act_by_token != 0;

  if (warp == kP4AWarp) {
    // ------------------------------------------------------ weight tiles
    {
      int slot = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;
      int4 rec = rec0;
      for (int w = w0; w < W && ok; w += wstep) {
        const F4Item it = fp4_item(rec, w, nbp);
        if (w + wstep < W) rec = fp4_record(a, w + wstep, nbp);
        const int blk = 2 * it.bp + (int)rank;
        const uint8_t *tiles = a.codes + (size_t)it.e * a.codes_expert + (size_t)blk * nkb * kP4AStageBytes;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!__all_sync(0xffffffffu, mbar_wait(empty0 + 8u * slot, phase ^ 1u))) {
            ok = false;
            break;
          }
          // the tile's codes and, right after them, its scale words in TMEM order
          if (elect_one()) {
            mbar_expect_tx(afull0 + 8u * slot, kP4AStageBytes);
            bulk_g2s(ringA + (uint32_t)slot * kP4AStageBytes, tiles + (size_t)kb * kP4AStageBytes, kP4AStageBytes,
                     afull0 + 8u * slot);
          }
          __syncwarp();
          issued |= 1u << slot;
          issued_parity = (issued_parity & ~(1u << slot)) | (phase << slot);
          if (++slot == kP4Stages) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
      // Never leave with a copy in flight into this CTA's shared memory.
      for (int i = 0; i < kP4Stages; ++i)
        if (issued & (1u << i)) mbar_wait(afull0 + 8u * i, (issued_parity >> i) & 1u);
    }
    __syncwarp();
  } else if (warp == kP4BWarp) {
    // ------------------------------------------------------ activation tiles
    // The activation rows of an item's 128 slots are one slot-major tile per
    // 256-K block (written by the row quantiser; expert groups are padded to
    // 128 slots, so a tile never straddles two experts).  This CTA's half of
    // the rows and all the scales: two bulk copies on one barrier.
    {
      int slot = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;
      const uint8_t *act = reinterpret_cast<const uint8_t *>(a.act);
      pdl_wait();  // the activation tiles come from the preceding kernel
      int4 rec = rec0;
      for (int w = w0; w < W && ok; w += wstep) {
        const F4Item it = fp4_item(rec, w, nbp);
        if (w + wstep < W) rec = fp4_record(a, w + wstep, nbp);
        const uint8_t *tiles = act + (size_t)(it.s0 / kP4N) * nkb * kP4AStageBytes;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!__all_sync(0xffffffffu, mbar_wait(empty0 + 8u * slot, phase ^ 1u))) {
            ok = false;
            break;
          }
          if (elect_one()) {
            const uint8_t *src = tiles + (size_t)kb * kP4AStageBytes;
            const uint32_t dst = ringB + (uint32_t)slot * kP4BStageBytes, bar = bfull0 + 8u * slot;
            mbar_expect_tx(bar, kP4BStageBytes);
            bulk_g2s(dst, src + rank * kP4BHalfBytes, kP4BHalfBytes, bar);
            bulk_g2s(dst + kP4BHalfBytes, src + kP4TileBytes, kP4SfBytes, bar);
          }
          __syncwarp();
          issued |= 1u << slot;
          issued_parity = (issued_parity & ~(1u << slot)) | (phase << slot);
          if (++slot == kP4Stages) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
      for (int i = 0; i < kP4Stages; ++i)
        if (issued & (1u << i)) mbar_wait(bfull0 + 8u * i, (issued_parity >> i) & 1u);
    }
    __syncwarp();
  } else if (warp >= kP4SfWarp0 && warp < kP4SfWarp0 + 4) {
    // ------------------------------------------------------ scale factors -> TMEM
    // Warp 8 + q writes lane quadrant q of this CTA's TMEM; every quadrant gets
    // the same words: per 64-K step t, this lane's 16 bytes of the weight
    // tile's and of the activation tile's scale blocks.
    const int q = warp - kP4SfWarp0;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    int slot = 0;
    uint32_t phase = 0;
    for (int w = w0; w < W && ok; w += wstep) {
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait(empty0 + 8u * slot, phase ^ 1u) || !mbar_wait(afull0 + 8u * slot, phase) ||
            !mbar_wait(bfull0 + 8u * slot, phase)) {
          ok = false;
          break;
        }
        const uint8_t *sfa = base + slot * kP4AStageBytes + kP4TileBytes + lane * 16;
        const uint8_t *sfb = base + kP4Stages * kP4AStageBytes + slot * kP4BStageBytes + kP4BHalfBytes + lane * 16;
        uint32_t ra[16], rb[16];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint4 va = *reinterpret_cast<const uint4 *>(sfa + 512 * t);
          const uint4 vb = *reinterpret_cast<const uint4 *>(sfb + 512 * t);
          ra[4 * t + 0] = va.x; ra[4 * t + 1] = va.y; ra[4 * t + 2] = va.z; ra[4 * t + 3] = va.w;
          rb[4 * t + 0] = vb.x; rb[4 * t + 1] = vb.y; rb[4 * t + 2] = vb.z; rb[4 * t + 3] = vb.w;
        }
        tc_fence_after();
        const uint32_t col = tmem + lane_base + (uint32_t)(kP4SfCol0 + slot * kP4SfCols);
        tc_st16(col, ra);
        tc_st16(col + 16, rb);
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sfull0 + 8u * slot);
        if (++slot == kP4Stages) {
          slot = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == kP4RelayWarp) {
    // ------------------------------------------------------ relay (both CTAs)
    // One thread per CTA turns "this CTA's stage is complete" into one arrival
    // on the leader's ready barrier.  The scale-factor warps arrive on sfull
    // only after they have seen both tiles land and their TMEM stores
    // complete, so sfull covers the whole stage.  The peer's arrival is
    // relaxed (a release at cluster scope would wait for every access the SM
    // has in flight, the next stages' copies included); the leader's MMAs
    // read the peer's stage only after it, when its writes have completed.
    if (lane == 0) {
      const uint32_t ready_leader = mapa(ready0, 0);
      int slot = 0;
      uint32_t phase = 0;
      for (int w = w0; w < W && ok; w += wstep) {
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(sfull0 + 8u * slot, phase)) {
            ok = false;
            break;
          }
          if (rank == 0)
            mbar_arrive(ready0 + 8u * slot);
          else
            mbar_arrive_remote_relaxed(ready_leader + 8u * slot);
          if (++slot == kP4Stages) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == kP4MmaWarp) {
    // ------------------------------------------------------ MMA issuer (leader CTA)
    if (rank == 0) {
      int sa = 0, li = 0;
      uint32_t pa = 0;
      for (int w = w0; w < W && ok; w += wstep, ++li) {
        const int b = li & 1;
        if (!__all_sync(0xffffffffu, mbar_wait_c(tempty0 + 8u * b, ((li >> 1) & 1) ^ 1u))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(b * kP4AccCols);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!__all_sync(0xffffffffu, mbar_wait_c(ready0 + 8u * sa, pa))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
            const uint64_t da = umma_desc_sw128(ringA + (uint32_t)sa * kP4AStageBytes);
            const uint64_t db = umma_desc_sw128(ringB + (uint32_t)sa * kP4BStageBytes);
            const uint32_t sf = tmem + (uint32_t)(kP4SfCol0 + sa * kP4SfCols);
#pragma unroll
            for (int j = 0; j < 4; ++j)  // K = 64 per MMA: 32 bytes of each operand row
              tc2_mma_fp4(d, da + 2u * j, db + 2u * j, sf + 4u * j, sf + 16u + 4u * j, (kb > 0 || j > 0) ? 1u : 0u);
            tc2_commit_both(empty0 + 8u * sa);  // frees both CTAs' stage once these MMAs have read it
          }
          __syncwarp();
          any_mma = true;
          if (++sa == kP4Stages) {
            sa = 0;
            pa ^= 1u;
          }
        }
        if (!ok) break;
        if (elect_one()) tc2_commit_both(tfull0 + 8u * b);
        __syncwarp();
      }
      // Every MMA of the pair completes before either CTA releases its shared
      // memory or the pair's tensor memory.
      if (any_mma) {
        if (elect_one()) tc2_commit_both(drain);
      } else if (lane == 0) {
        mbar_arrive(drain);
        mbar_arrive_remote(mapa(drain, 1));
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------ epilogue (both CTAs)
    // Each CTA's eight warps read its 128 rows of the accumulator (lane
    // quadrant warp % 4, column half warp / 4) and hand the buffer back to the
    // leader's MMA warp.
    const int m = (warp & 3) * 32 + lane;  // accumulator row = TMEM lane
    const int cbase = (warp >> 2) * (kP4N / 2);  // this warp's half of the 128 token columns
    constexpr int kCh = kP4N / 2 / 32;
    const uint32_t tempty_leader = mapa(tempty0, 0);
    // Per column (one per lane and 32-column chunk, broadcast with shuffles):
    // the activation row's FP32 global, times the topk weight and the global
    // scale for the down projection; per row the expert's global scale of the
    // gate / up / single matrix.  Item record -> the tile's pairs -> their
    // factors are three dependent global loads; they run as a pipeline over the
    // items (the record three items ahead, the pairs two, the factors one), so
    // each load has a whole item's epilogue to return.
    auto pairs_of = [&](const F4Item &it, int (&p)[kCh]) {
#pragma unroll
      for (int ch = 0; ch < kCh; ++ch) {
        const int nl = cbase + 32 * ch + lane;
        p[ch] = nl < it.ntok ? a.sorted_pair[it.s0 + nl] : -1;
      }
    };
    auto factors_of = [&](const F4Item &it, const int (&p)[kCh], float (&c)[kCh], float &gs) {
      gs = a.globals[4 * it.e + ((STAGE == STAGE_GATED && (m & 15) >= 8) ? 1 : 0)];
      const float g2 = STAGE == STAGE_DOWN ? a.globals[4 * it.e + 2] : 1.f;
#pragma unroll
      for (int ch = 0; ch < kCh; ++ch) {
        const int nl = cbase + 32 * ch + lane;
        c[ch] = 0.f;
        if (p[ch] >= 0) {
          const float f = a.act_g[by_token ? (int64_t)(p[ch] / a.top_k) : (int64_t)(it.s0 + nl)];
          c[ch] = STAGE == STAGE_DOWN ? f * (a.topk_weights[p[ch]] * g2) : f;
        }
      }
    };
    pdl_wait();                      // activation globals come from the preceding kernel
    F4Item it0{}, it1{};             // the current item and the next
    int p1[kCh];                     // the next item's pairs
    float c0[kCh], gs0 = 1.f;        // the current item's factors
    int4 rec2 = make_int4(0, 0, 0, 0);  // record of the item after next
#pragma unroll
    for (int ch = 0; ch < kCh; ++ch) {
      p1[ch] = -1;
      c0[ch] = 0.f;
    }
    if (w0 < W) {
      it0 = fp4_item(rec0, w0, nbp);
      int p0[kCh];
      pairs_of(it0, p0);
      factors_of(it0, p0, c0, gs0);
      if (w0 + wstep < W) {
        it1 = fp4_item(fp4_record(a, w0 + wstep, nbp), w0 + wstep, nbp);
        pairs_of(it1, p1);
      }
      if (w0 + 2 * wstep < W) rec2 = fp4_record(a, w0 + 2 * wstep, nbp);
    }
    int li = 0;
    for (int w = w0; w < W && ok; w += wstep, ++li) {
      const F4Item it = it0;
      const float gsel = gs0;
      float c_l[kCh];
#pragma unroll
      for (int ch = 0; ch < kCh; ++ch) c_l[ch] = c0[ch];
      // the next items' loads, consumed one item later
      float c1[kCh], gs1 = 1.f;
      F4Item it2{};
      int p2[kCh];
#pragma unroll
      for (int ch = 0; ch < kCh; ++ch) {
        c1[ch] = 0.f;
        p2[ch] = -1;
      }
      if (w + wstep < W) factors_of(it1, p1, c1, gs1);
      if (w + 2 * wstep < W) {
        it2 = fp4_item(rec2, w + 2 * wstep, nbp);
        pairs_of(it2, p2);
      }
      if (w + 3 * wstep < W) rec2 = fp4_record(a, w + 3 * wstep, nbp);
      const int b = li & 1;
      if (!mbar_wait(tfull0 + 8u * b, (li >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int blk = 2 * it.bp + (int)rank;
      const int tile = 8 * blk + (m >> 4), rr = m & 15;
      float *__restrict__ outp = a.out;
#pragma unroll
      for (int ch = 0; ch < kCh; ++ch) {
        const int c0 = cbase + 32 * ch;
        uint32_t raw[32];
        tc_ld32(tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(b * kP4AccCols + c0), raw);
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
      // relaxed: the accumulator has been read (tcgen05.wait::ld), and this
      // warp's output stores need not complete before the MMA reuses it
      if (lane == 0) mbar_arrive_remote_relaxed(tempty_leader + 8u * b);
      it0 = it1;
      gs0 = gs1;
      it1 = it2;
#pragma unroll
      for (int ch = 0; ch < kCh; ++ch) {
        c0[ch] = c1[ch];
        p1[ch] = p2[ch];
      }
    }
  }

  if (!ok && lane == 0) atomicOr(&a.status[ST_FLAGS], ST_FLAG_TIMEOUT);
  pdl_wait();  // completion implies the predecessor's (a no-op for threads that already waited)
  if (warp == kP4MmaWarp && lane == 0) {
    if (!mbar_wait_c(drain, 0)) atomicOr(&a.status[ST_FLAGS], ST_FLAG_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // neither CTA leaves while the pair's MMAs or remote arrivals may touch it
  tc_fence_after();
  if (warp == kP4MmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kP4TmemCols));
}

static size_t fp4_smem_bytes() { return (size_t)kP4RingBytes + 1024 + 8 * kP4Bars + 16; }
static_assert(kP4RingBytes + 1024 + 8 * kP4Bars + 16 <= 227 * 1024, "shared memory budget");

bool fp4_tc_supported(int rows_total, int K) { return rows_total % 256 == 0 && K % 256 == 0; }

template <int STAGE>
static cudaError_t launch_fp4_one(const GroupedArgs &a, int rows_total, cudaStream_t s) {
  auto kern = k_grouped_fp4<STAGE>;
  const size_t smem = fp4_smem_bytes();
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  // as many co-resident CTA pairs as the device holds (clusters are placed
  // within a GPC, so this can be below half the SM count)
  int clusters = 0;
  {
    cudaLaunchConfig_t cfg = {};
    int dev = 0, sms = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
    cfg.gridDim = dim3(sms / 2 * 2);
    cfg.blockDim = dim3(kP4Threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((err = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg)) != cudaSuccess) return err;
    clusters = std::min(clusters, sms / 2);
  }
  if (clusters <= 0) return cudaErrorInvalidConfiguration;
  GroupedArgs g = a;
  g.n_blocks = rows_total / 128;
  return launch_pdl_cluster(kern, dim3(2 * clusters), dim3(kP4Threads), smem, 2, s, g);
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
