// Grouped expert contractions on CTA pairs of the 5th-generation tensor cores
// (tcgen05.mma.cta_group::2, M = 256), for experts that receive many tokens.
//
// moe.fused_moe's W4A16 mode (BF16 activations against FP4 weights dequantised
// in the kernel) and its MXFP4 experts (b12x project page, section "What's in
// here").  The contraction of an expert is a dense GEMM once it sees more than
// a few dozen tokens.  On one SM an M=128 N=128 K=16 MMA reads 8 KB of
// operands from shared memory while the producers write the dequantised
// weight tile and the activation tile through the same port, so a single-CTA
// kernel is held by shared-memory bandwidth well below the tensor pipe's rate.
// Here two CTAs of a cluster form one MMA: each holds 128 weight rows (its A
// half) and half of the token tile (its B half), and the leader CTA issues
// M=256 N<=256 K=16 MMAs that read both CTAs' shared memory, so every byte
// written to shared memory feeds twice the FLOPs:
//
//   D[256 weight rows x N tokens] += A[256 x 64] * B[N x 64]^T per 64-K block
//
// * A: each CTA's 128-row block of the packed experts (the same fragment-order
//   bytes the decode kernel streams), loaded into registers four of its
//   k-blocks ahead by eight producer warps in two groups that produce
//   alternate k-blocks (one warp's chain of conversions, stores and proxy
//   fence per k-block is latency bound), dequantised to FP16 (NVFP4: E2M1 x
//   E4M3 is exact) or BF16 (MXFP4: E2M1 x 2^X is exact) and written in the
//   UMMA K-major 128-byte-swizzled layout; a 6-stage ring.  The K order of
//   both operands within a 64-element step is the pair order (below), in
//   which a producer lane's two rows take four 16-byte stores.
// * B: the tile's activation rows are consecutive slots of the expert-sorted
//   list (GEMM1's x rows are gathered into slot order beforehand, GEMM2's h
//   rows already are, both written in the pair order), so a CTA's B half of a
//   k-block is one 2-D tensor copy (TMA, 128 rows x 64 columns, 128-byte
//   swizzle); a 6-stage ring.
// * Token tiles: an expert with c pairs is cut into ceil(c / 256) tiles of
//   equal size (rounded up to 16), so no tile is a nearly empty remainder;
//   the MMA's N is the tile's size rounded up to 16.
// * A relay thread in each CTA turns "this CTA's operands of two k-blocks are
//   in shared memory" into one arrival on the leader's ready barrier; the
//   leader's MMA thread waits on that one barrier, issues 8 MMAs into one of
//   two TMEM accumulators (2 x 256 columns) and releases both CTAs' two
//   stages with one multicast tcgen05.commit.  K is a multiple of 128.
// * Each CTA's eight epilogue warps (lane quadrant, column half) read its 128
//   rows of the accumulator (SiLU(gate)*up, ReLU^2, or the topk_weight scaling
//   of the down projection) while the next tile's MMAs run, and hand the
//   buffer back with a relaxed arrive.
// * Work items are (large expert, token tile, pair of 128-row blocks), dealt
//   round-robin over persistent clusters (one CTA per SM).
// * Every wait is a bounded mbarrier wait; on a timeout the kernel sets the
//   status flag, every CTA still reaches the final cluster barrier, and the
//   leader drains its MMAs before the pair's tensor memory is released.
#include <algorithm>
#include <mutex>
#include <cstdio>
#include <cstdlib>

#include "common.cuh"
#include "dequant.cuh"
#include "internal.h"
#include "launch.h"
#include "sync.cuh"
#include "tcgen05.cuh"
#include "tmap.h"

namespace bqmoe {

constexpr int k2EpiWarps = 8, k2AWarps = 8, k2BWarps = 1;
constexpr int k2MmaWarp = k2EpiWarps + k2AWarps + k2BWarps;  // warp 17
constexpr int k2RelayWarp = k2MmaWarp + 1;                     // warp 18
constexpr int k2LoadWarp = k2RelayWarp + 1;                     // warp 19
constexpr int k2Threads = (k2LoadWarp + 1) * 32;
constexpr int k2MaxN = 256;                 // tokens per pair tile
constexpr int k2HalfRows = k2MaxN / 2;      // B rows per CTA
constexpr int k2ABytes = 128 * 64 * 2;      // one 128 x 64 16-bit block
constexpr int k2BBytes = k2HalfRows * 64 * 2;
// Rings: the packed weight bytes of a k-block (one contiguous run per 128-row
// block) arrive by bulk copies into a raw ring that runs up to k2RawStages
// k-blocks ahead of the A warps, which dequantise from it into the A ring; the
// activation tiles arrive by tensor copies into the B ring.
constexpr int k2AStages = 6;
constexpr int k2BStages = 6;
// The MMA thread consumes the stages two k-blocks at a time: one wait on the
// leader's ready barrier and one commit per pair of stages (A and B stages 2q
// and 2q + 1 share the empty barrier of pair q), which halves the per-k-block
// synchronisation on the issuing thread.
constexpr int k2Pairs = k2AStages / 2;
constexpr int k2RStages = 4;                // ready barriers, by pair of k-blocks
static_assert(k2AStages == k2BStages && k2AStages % 2 == 0 && k2RStages > k2Pairs, "paired stages");
constexpr int k2RawStages = 6;             // packed weight bytes of a k-block, by k-block
constexpr int k2RawBytes = 4608;            // bytes of one 64-K step of a 128-row block (NVFP4; MXFP4: 4352)
constexpr int k2AGroups = 2;                // A warp groups producing alternate k-blocks
constexpr int k2AThreadsPerGroup = k2AWarps * 32 / k2AGroups;
constexpr int k2RingBytes = k2AStages * k2ABytes + k2BStages * k2BBytes + k2RawStages * k2RawBytes;
constexpr int k2AccCols = k2MaxN;           // TMEM columns per accumulator buffer
constexpr int k2TmemCols = 2 * k2AccCols;   // double buffered
constexpr int k2Bars = k2AStages + k2BStages + k2Pairs + k2RStages + 4 + 1 + 2 * k2RawStages;
static_assert(k2AWarps * 32 == 256 && 256 % (k2AGroups * 32) == 0, "8 fragment chunks per k-block over the A groups");

// Named barrier 1 over the eight epilogue warps (threads 0..255).
__device__ __forceinline__ void epi_bar_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// The same barrier, returning whether every epilogue thread passed `v`.
__device__ __forceinline__ bool epi_bar_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 1, 256, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// 2-D tiled tensor copy global -> shared with completion (bytes) on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// Arrive on `bar` once all of this thread's earlier cp.async copies have landed
// (the arrival is not counted in advance: the barrier's count includes it).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc2_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// One fragment chunk of a packed 64-K step (16 code bytes of lane `ln` of
// 16-row tile `tile`, and the lane group's block scales), dequantised to
// 16-bit values (NVFP4: E2M1 x E4M3 in FP16, exact; MXFP4: E2M1 x 2^X in BF16,
// exact) and stored in the pair kernel's K order in the 128-byte-swizzled
// K-major tile.
template <int WF>
__device__ __forceinline__ void dequant_chunk_store(uint8_t *tileA, uint4 cch, uint2 sch, int tile, int ln) {
  const int g = ln >> 2, c4 = ln & 3;
  const int r0 = 16 * tile + g, r1 = r0 + 8;
  const uint32_t cw[4] = {cch.x, cch.y, cch.z, cch.w};
  uint32_t o[4][4];  // 16-bit pairs of mma j: (r0, k), (r1, k), (r0, k + 8), (r1, k + 8)
  if (WF == W_NVFP4) {
    uint32_t sp[4];
    e4m3x4_to_f16x2x2(sch.x, sp[0], sp[1]);
    e4m3x4_to_f16x2x2(sch.y, sp[2], sp[3]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t s_lo = sp[2 * (j >> 1)], s_hi = sp[2 * (j >> 1) + 1];
      uint32_t af[4];
      e2m1x8_to_f16x2x4(cw[j], af);
      o[j][0] = hmul2(af[0], s_lo);
      o[j][1] = hmul2(af[1], s_hi);
      o[j][2] = hmul2(af[2], s_lo);
      o[j][3] = hmul2(af[3], s_hi);
    }
  } else {
    const uint32_t sw = sch.x;  // (r0 block 0, r0 block 1, r1 block 0, r1 block 1)
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
  // Lane c of a quad holds, of rows r0 and r1, the 16 values of slot positions
  // 16 j + 8 h + 2 c + e (word j, pair h, element e); the pair kernel's K order
  // puts them at 16 c + 4 j + 2 h + e, so each row's 16 values are two
  // contiguous 16-byte chunks (the activation rows are written in that order).
  auto put = [&](int r, int ch, uint4 v) {
    *reinterpret_cast<uint4 *>(tileA + (r >> 3) * 1024 + (r & 7) * 128 + (((ch ^ r) & 7) << 4)) = v;
  };
  put(r0, 2 * c4, make_uint4(o[0][0], o[0][2], o[1][0], o[1][2]));
  put(r0, 2 * c4 + 1, make_uint4(o[2][0], o[2][2], o[3][0], o[3][2]));
  put(r1, 2 * c4, make_uint4(o[0][1], o[0][3], o[1][1], o[1][3]));
  put(r1, 2 * c4 + 1, make_uint4(o[2][1], o[2][3], o[3][1], o[3][3]));
}

// ------------------------------------------------------------------ work items

struct Tc2Item {
  int e, s0, ntok, n, bp;  // expert, first slot, live tokens, MMA N, row-block pair
};

// Items (token tile of a large expert, row-block pair), in that order: item w
// is row-block pair w % nbp of tile w / nbp, whose record the routing wrote
// (expert, first slot, live tokens).  The MMA's N is the live tokens rounded
// up to 16.  Every role loads the next item's record while it works on the
// current one, so no dependent global load sits between two items.
__device__ __forceinline__ int4 tc2_record(const GroupedArgs &a, int w, int nbp) { return a.tiles[w / nbp]; }
__device__ __forceinline__ Tc2Item tc2_item(const int4 r, int w, int nbp) {
  Tc2Item it;
  it.e = r.x;
  it.s0 = r.y;
  it.ntok = r.z;
  it.n = max(16, (r.z + 15) & ~15);
  it.bp = w % nbp;
  return it;
}

// ------------------------------------------------------------------ kernel

template <int STAGE, int WF>
__global__ void __launch_bounds__(k2Threads, 1) k_grouped_tc2(const GroupedArgs a,
                                                              const __grid_constant__ CUtensorMap bmap) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base for the swizzled tiles (the same offset in both CTAs)
  const uint32_t raw_s = (uint32_t)__cvta_generic_to_shared(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t *base = smem_raw + (base_s - raw_s);
  const uint32_t ringA = base_s, ringB = base_s + k2AStages * k2ABytes;
  const uint32_t ringR = ringB + k2BStages * k2BBytes;
  const uint8_t *rawR = base + (ringR - base_s);
  uint64_t *bars = reinterpret_cast<uint64_t *>(base + k2RingBytes);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + k2Bars);
  // per-column factor of the epilogue, two items deep: [2][k2MaxN]
  float *colinfo = reinterpret_cast<float *>(base + k2RingBytes + 8 * k2Bars + 16);
  const uint32_t afull0 = (uint32_t)__cvta_generic_to_shared(bars);  // this CTA's A tile is written
  const uint32_t bfull0 = afull0 + 8u * k2AStages;                   // this CTA's B tile has landed
  const uint32_t empty0 = bfull0 + 8u * k2BStages;                   // the pair's MMAs have read a pair of stages
  const uint32_t ready0 = empty0 + 8u * k2Pairs;                     // leader: both CTAs' operands of a pair
  const uint32_t tfull0 = ready0 + 8u * k2RStages;                   // 2
  const uint32_t tempty0 = tfull0 + 16u;                             // 2
  const uint32_t drain = tempty0 + 16u;                              // 1
  const uint32_t rfull0 = drain + 8u;                                // raw weight bytes have landed
  const uint32_t rempty0 = rfull0 + 8u * k2RawStages;                // the A group has read them

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();  // 0: leader (issues the MMAs), 1: peer
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int i = 0; i < k2AStages; ++i) {
      mbar_init(afull0 + 8u * i, k2AWarps / k2AGroups);
      mbar_init(bfull0 + 8u * i, 1);
    }
    for (int i = 0; i < k2Pairs; ++i) mbar_init(empty0 + 8u * i, 1);
    for (int i = 0; i < k2RStages; ++i) mbar_init(ready0 + 8u * i, 2);
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull0 + 8u * b, 1);
      mbar_init(tempty0 + 8u * b, 2 * k2EpiWarps);
    }
    mbar_init(drain, 1);
    for (int i = 0; i < k2RawStages; ++i) {
      mbar_init(rfull0 + 8u * i, 1);
      mbar_init(rempty0 + 8u * i, k2AWarps / k2AGroups);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == k2MmaWarp) {  // one warp of each CTA of the pair allocates, together
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(tmem_slot)),
                 "n"(k2TmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int K = a.K;
  const int nk = K / 64;
  const int nbp = a.n_blocks / 2;
  const int n_large = a.large[0];
  const int W = n_large > 0 ? a.large_tiles[n_large] * nbp : 0;
  // Items are dealt round-robin over clusters: at any moment the pairs work on
  // neighbouring items, which share token tiles and weight blocks in L2.
  const int w0 = (int)cluster_id_x(), wstep = (int)cluster_count_x();
  const int4 rec0 = w0 < W ? tc2_record(a, w0, nbp) : make_int4(0, 0, 0, 0);
  bool ok = true;
  bool any_mma = false;

  if (warp >= k2EpiWarps && warp < k2EpiWarps + k2AWarps) {
    // ------------------------------------------------------ A producers
    // The A warps form k2AGroups groups; group q produces the k-blocks n with
    // n % k2AGroups == q, so several stages are dequantised at once (one
    // warp's chain of loads, conversions, stores and fence per k-block is
    // latency bound).  Thread tg of a group takes fragment chunks tg + 128 i of
    // its k-blocks (16-row tile chunk / 32, lane chunk % 32) from the raw ring:
    // 16 code bytes and the lane group's block scales, dequantised to 16-bit
    // values written at their slot positions in the swizzled tile.
    constexpr int CPT = k2AGroups;                   // chunks per thread per k-block
    const int t = threadIdx.x - k2EpiWarps * 32;    // 0..255
    const int grp = t / (k2AThreadsPerGroup), tg = t % k2AThreadsPerGroup;
    const int ln = tg & 31;
    const int n_items = w0 < W ? (W - w0 + wstep - 1) / wstep : 0;
    const int total = n_items * nk;
    for (int n = grp; n < total && ok; n += k2AGroups) {
      const int r = n % k2RawStages;
      if (!mbar_wait(rfull0 + 8u * r, (uint32_t)(n / k2RawStages) & 1u)) {
        ok = false;
        break;
      }
      const uint8_t *step = rawR + (size_t)r * k2RawBytes;
      uint4 cch[CPT];
      uint2 sch[CPT];
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        const int tile = (tg >> 5) + (k2AThreadsPerGroup / 32) * i;
        cch[i] = *reinterpret_cast<const uint4 *>(step + tile * 512 + ln * 16);
        if (WF == W_NVFP4) sch[i] = *reinterpret_cast<const uint2 *>(step + 4096 + tile * 64 + (ln >> 2) * 8);
        else sch[i] = make_uint2(*reinterpret_cast<const uint32_t *>(step + 4096 + tile * 32 + (ln >> 2) * 4), 0u);
      }
      const int slot = n % k2AStages;
      const bool got = mbar_wait(empty0 + 8u * (slot >> 1), ((uint32_t)(n / k2AStages) & 1u) ^ 1u);
      __syncwarp();  // every lane's reads of the raw stage are done
      if (lane == 0) mbar_arrive(rempty0 + 8u * r);
      if (!got) {
        ok = false;
        break;
      }
      uint8_t *tileA = base + (size_t)slot * k2ABytes;
#pragma unroll
      for (int i = 0; i < CPT; ++i)
        dequant_chunk_store<WF>(tileA, cch[i], sch[i], (tg >> 5) + (k2AThreadsPerGroup / 32) * i, ln);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(afull0 + 8u * slot);
    }
  } else if (warp >= k2EpiWarps + k2AWarps && warp < k2MmaWarp) {
    // ------------------------------------------------------ B producer
    // The tile's activation rows are consecutive slots of the expert-sorted
    // list (GEMM1: x rows gathered into slot order beforehand; GEMM2: h rows),
    // so a stage's B half is one 2-D tensor copy: rows [s0 + rank * N/2, +128)
    // x columns [64 kb, +64).  Rows past the tile's live tokens feed only MMA
    // columns that the epilogue discards; rows past the tensor read as zeros.
    // The whole warp runs the loop; one elected lane issues the copies.
    {
      int slot = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;  // per slot: has a copy, parity of its last phase
      pdl_wait();  // activation rows come from the preceding kernels
      int4 rec = rec0;
      for (int w = w0; w < W && ok; w += wstep) {
        const Tc2Item it = tc2_item(rec, w, nbp);
        if (w + wstep < W) rec = tc2_record(a, w + wstep, nbp);
        const int y = it.s0 + (int)rank * (it.n >> 1);
        for (int kb = 0; kb < nk; ++kb) {
          if (!__all_sync(0xffffffffu, mbar_wait(empty0 + 8u * (slot >> 1), phase ^ 1u))) {
            ok = false;
            break;
          }
          const uint32_t bar = bfull0 + 8u * slot;
          if (elect_one()) {
            mbar_expect_tx(bar, k2BBytes);
            tma_load_2d(ringB + (uint32_t)slot * k2BBytes, &bmap, kb * 64, y, bar);
          }
          __syncwarp();
          issued |= 1u << slot;
          issued_parity = (issued_parity & ~(1u << slot)) | (phase << slot);
          if (++slot == k2BStages) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
      // Never leave with a tensor copy in flight into this CTA's shared memory.
      for (int i = 0; i < k2BStages; ++i)
        if (issued & (1u << i)) mbar_wait(bfull0 + 8u * i, (issued_parity >> i) & 1u);
    }
    __syncwarp();
  } else if (warp == k2MmaWarp) {
    // ------------------------------------------------------ MMA issuer (leader CTA)
    // The whole warp runs the loop (waits, counters, descriptors), so every
    // operand of the MMAs is warp-uniform, and one elected lane issues the
    // MMAs and commits.  Issued from a single-thread branch instead, each
    // cta_group::2 MMA cost about 130 cycles of issue whatever its N, which
    // capped the tensor pipe at half its rate for N near 128.
    if (rank == 0) {
      constexpr uint32_t fmt = WF == W_MXFP4 ? 1u : 0u;  // operand type: 0 = F16, 1 = BF16
      const uint32_t idesc0 = (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(256 >> 4) << 24);
      int q = 0, li = 0;  // pairs of k-blocks consumed over the launch
      int4 rec = rec0;
      for (int w = w0; w < W && ok; w += wstep, ++li) {
        const Tc2Item it = tc2_item(rec, w, nbp);
        if (w + wstep < W) rec = tc2_record(a, w + wstep, nbp);
        const uint32_t idesc = idesc0 | ((uint32_t)(it.n >> 3) << 17);
        const int b = li & 1;
        if (!__all_sync(0xffffffffu, mbar_wait_c(tempty0 + 8u * b, ((li >> 1) & 1) ^ 1u))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem + (uint32_t)(b * k2AccCols);
        for (int kp = 0; kp < nk; kp += 2, ++q) {
          if (!__all_sync(0xffffffffu, mbar_wait(ready0 + 8u * (q % k2RStages), (uint32_t)(q / k2RStages) & 1u))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int slot = (2 * q + h) % k2AStages;
              const uint64_t da = umma_desc_sw128(ringA + (uint32_t)slot * k2ABytes);
              const uint64_t db = umma_desc_sw128(ringB + (uint32_t)slot * k2BBytes);
#pragma unroll
              for (int j = 0; j < 4; ++j)  // K = 16 per MMA: advance the start address by 32 bytes
                tc2_mma_f16(d0, da + 2u * j, db + 2u * j, idesc, (kp > 0 || h > 0 || j > 0) ? 1u : 0u);
            }
            tc2_commit_both(empty0 + 8u * (q % k2Pairs));  // frees both CTAs' stages once these MMAs have read them
          }
          __syncwarp();
          any_mma = true;
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
  } else if (warp == k2RelayWarp) {
    // ------------------------------------------------------ relay (both CTAs)
    // One thread per CTA turns "this CTA's stage is full" (its A warps'
    // arrivals and its B tensor copy) into one arrival on the leader's ready
    // barrier, so the MMA thread waits on a single barrier per pair.  The
    // relay has observed the stage's writes (acquire) before it arrives; the
    // peer's arrival is relaxed, because a release at cluster scope here
    // would wait for every memory access the SM has in flight (the tensor
    // copies and weight loads of the next stages) and stall the pipeline by
    // about half a microsecond per pair.  The leader's MMAs read the peer's
    // stage only after that arrival, when its writes have completed.
    if (lane == 0) {
      const uint32_t ready_leader = mapa(ready0, 0);
      int q = 0;
      for (int w = w0; w < W && ok; w += wstep) {
        for (int kp = 0; kp < nk && ok; kp += 2, ++q) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int n = 2 * q + h, slot = n % k2AStages;
            const uint32_t ph = (uint32_t)(n / k2AStages) & 1u;
            if (!mbar_wait(afull0 + 8u * slot, ph) || !mbar_wait(bfull0 + 8u * slot, ph)) {
              ok = false;
              break;
            }
          }
          if (!ok) break;
          if (rank == 0)
            mbar_arrive(ready0 + 8u * (q % k2RStages));
          else
            mbar_arrive_remote_relaxed(ready_leader + 8u * (q % k2RStages));
        }
      }
    }
    __syncwarp();
  } else if (warp == k2LoadWarp) {
    // ------------------------------------------------------ raw weight loader
    // One bulk copy per k-block of this CTA's 128-row block of the item's
    // expert: the packed codes and scales of a 64-K step are contiguous.
    // The whole warp runs the loop; one elected lane issues the copies.
    {
      constexpr uint32_t SB = WF == W_NVFP4 ? 4608u : 4352u;
      int r = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;  // per slot: has a copy, parity of its last phase
      int4 rec = rec0;
      for (int w = w0; w < W && ok; w += wstep) {
        const Tc2Item it = tc2_item(rec, w, nbp);
        if (w + wstep < W) rec = tc2_record(a, w + wstep, nbp);
        const int blk = 2 * it.bp + (int)rank;
        const uint8_t *src = a.codes + (size_t)it.e * a.codes_expert + (size_t)blk * nk * SB;
        for (int kb = 0; kb < nk; ++kb) {
          if (!__all_sync(0xffffffffu, mbar_wait(rempty0 + 8u * r, phase ^ 1u))) {
            ok = false;
            break;
          }
          const uint32_t bar = rfull0 + 8u * r;
          if (elect_one()) {
            mbar_expect_tx(bar, SB);
            bulk_g2s(ringR + (uint32_t)r * k2RawBytes, src + (size_t)kb * SB, SB, bar);
          }
          __syncwarp();
          issued |= 1u << r;
          issued_parity = (issued_parity & ~(1u << r)) | (phase << r);
          if (++r == k2RawStages) {
            r = 0;
            phase ^= 1u;
          }
        }
      }
      // Never leave with a bulk copy in flight into this CTA's shared memory.
      for (int i = 0; i < k2RawStages; ++i)
        if (issued & (1u << i)) mbar_wait(rfull0 + 8u * i, (issued_parity >> i) & 1u);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------ epilogue (both CTAs)
    // Each column's factor (activation factor; for the down projection times
    // the topk weight and the expert's global scale) is fetched one item ahead
    // into shared memory by the 256 epilogue threads (slot -> pair -> factors:
    // dependent global loads whose latency then overlaps the previous item's
    // epilogue) and read back as broadcast vector loads.  The eight warps decide
    // together (barrier with an AND vote) whether to go on, so none waits at
    // the barrier for a warp that has stopped.
    const int m = (warp & 3) * 32 + lane;    // accumulator row = TMEM lane (quadrant warp % 4)
    const int cbase = (warp >> 2) * (k2MaxN / 2);  // this warp's half of the tile's columns
    const int et = threadIdx.x;              // 0..255: the column whose factor this thread fetches
    const uint32_t tempty_leader = mapa(tempty0, 0);
    float *__restrict__ outp = a.out;
    int pn;
    auto fetch_pairs = [&](const Tc2Item &it) { pn = et < it.ntok ? a.sorted_pair[it.s0 + et] : -1; };
    float cn, gn = 1.f;
    auto fetch_factors = [&](const Tc2Item &it) {
      // the expert's global scale of this thread's rows (gate / up / single
      // matrix), applied in the epilogue; the down projection's goes into the
      // column factor
      gn = a.globals[4 * it.e + ((STAGE == STAGE_GATED && (m & 15) >= 8) ? 1 : 0)];
      const float g2 = STAGE == STAGE_DOWN ? a.globals[4 * it.e + 2] : 1.f;
      cn = 0.f;
      if (pn >= 0) {
        const int sl = it.s0 + et;
        const float f = a.act_g ? a.act_g[a.act_by_token ? (int64_t)(pn / a.top_k) : (int64_t)sl] : 1.f;
        cn = STAGE == STAGE_DOWN ? f * (a.topk_weights[pn] * g2) : f;
      }
    };
    auto put_factors = [&](int buf) { colinfo[buf * k2MaxN + et] = cn; };
    pdl_wait();  // row factors come from the preceding kernels
    Tc2Item it_next{};
    float gsel_next = 1.f;
    int4 rec = make_int4(0, 0, 0, 0);  // record of the item after next
    if (w0 < W) {
      it_next = tc2_item(rec0, w0, nbp);
      if (w0 + wstep < W) rec = tc2_record(a, w0 + wstep, nbp);
      fetch_pairs(it_next);
      fetch_factors(it_next);
      put_factors(0);
      gsel_next = gn;
    }
    epi_bar_sync();
    int li = 0;
    for (int w = w0; w < W && ok; w += wstep, ++li) {
      const Tc2Item it = it_next;
      const float gsel = gsel_next;
      const bool more = w + wstep < W;
      if (more) {
        it_next = tc2_item(rec, w + wstep, nbp);
        if (w + 2 * wstep < W) rec = tc2_record(a, w + 2 * wstep, nbp);
        fetch_pairs(it_next);
      }
      const int b = li & 1;
      const bool got = mbar_wait(tfull0 + 8u * b, (li >> 1) & 1);
      if (more) fetch_factors(it_next);
      if (got) {
        tc_fence_after();
        const int blk = 2 * it.bp + (int)rank;
        const int tile = 8 * blk + (m >> 4), rr = m & 15;
        const float *colc = colinfo + b * k2MaxN;
        for (int c0 = cbase; c0 < min(it.n, cbase + k2MaxN / 2); c0 += 32) {
          uint32_t raw[32];
          tc_ld32(tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(b * k2AccCols + c0), raw);
          float v[32];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 c4 = *reinterpret_cast<const float4 *>(colc + c0 + 4 * q);
            v[4 * q + 0] = __uint_as_float(raw[4 * q + 0]) * c4.x;
            v[4 * q + 1] = __uint_as_float(raw[4 * q + 1]) * c4.y;
            v[4 * q + 2] = __uint_as_float(raw[4 * q + 2]) * c4.z;
            v[4 * q + 3] = __uint_as_float(raw[4 * q + 3]) * c4.w;
          }
          if (STAGE == STAGE_GATED) {
            // Rows 0-7 of each 16-row group are gate rows, 8-15 the matching up
            // rows.  Columns go in pairs: a gate lane finishes the even column
            // (its up value from lane + 8), an up lane the odd one (its gate
            // value from lane - 8), so every lane evaluates one SiLU per pair.
            const bool up_lane = rr >= 8;
            const int hrow = tile * 8 + (rr & 7);
            float hv[16];
#pragma unroll
            for (int p = 0; p < 16; ++p) {
              const float x0 = v[2 * p] * gsel, x1 = v[2 * p + 1] * gsel;
              const float other = __shfl_xor_sync(0xffffffffu, up_lane ? x0 : x1, 8);
              const float gate = up_lane ? other : x0, up = up_lane ? x1 : other;
              const float h = silu_f32(gate) * up;
              const int n = c0 + 2 * p + (up_lane ? 1 : 0);
              const bool live = n < it.ntok;
              if (live) outp[(size_t)(it.s0 + n) * a.n_rows + hrow] = h;
              hv[p] = live ? fabsf(h) : 0.f;
            }
            if (a.out_amax != nullptr) {
              // reduce-scatter max over the 16 lanes holding the same column
              // parity (lane bits 4, 2, 1, 0): lane l ends with pair
              // (bit 4 of l) * 8 + (l & 7), column parity bit 3 of l
#pragma unroll
              for (int hs = 8, k = 0; hs >= 1; hs >>= 1, ++k) {
                const int step = k == 0 ? 16 : hs;
                const bool upper = (lane & step) != 0;
#pragma unroll
                for (int j = 0; j < hs; ++j) {
                  const float send = upper ? hv[j] : hv[j + hs];
                  const float keep = upper ? hv[j + hs] : hv[j];
                  hv[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, step));
                }
              }
              const int n = c0 + 2 * (((lane >> 4) & 1) * 8 + (lane & 7)) + ((lane >> 3) & 1);
              if (n < it.ntok)
                atomicMax(reinterpret_cast<unsigned *>(a.out_amax) + it.s0 + n, __float_as_uint(hv[0]));
            }
          } else if (STAGE == STAGE_RELU2) {
            float hv[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int n = c0 + j;
              const bool live = n < it.ntok;
              const float r = fmaxf(v[j] * gsel, 0.f);
              if (live) outp[(size_t)(it.s0 + n) * a.n_rows + tile * 16 + rr] = r * r;
              hv[j] = live ? r * r : 0.f;
            }
            if (a.out_amax != nullptr) {
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
              if (n < it.ntok)
                atomicMax(reinterpret_cast<unsigned *>(a.out_amax) + it.s0 + n, __float_as_uint(hv[0]));
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
      }
      if (more) {
        put_factors((li + 1) & 1);
        gsel_next = gn;
      }
      ok = epi_bar_and(got);  // buffer li + 1 is complete; buffer li is no longer read
    }
  }

  if (!ok && lane == 0) atomicOr(&a.status[ST_FLAGS], ST_FLAG_TIMEOUT);
  pdl_wait();  // completion implies the predecessor's (a no-op for threads that already waited)
  if (warp == k2MmaWarp && lane == 0) {
    if (!mbar_wait_c(drain, 0)) atomicOr(&a.status[ST_FLAGS], ST_FLAG_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // neither CTA leaves while the pair's MMAs or remote arrivals may touch it
  tc_fence_after();
  if (warp == k2MmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(k2TmemCols));
}

constexpr int k2ColBytes = 2 * k2MaxN * 4;
static size_t tc2_smem_bytes() { return (size_t)k2RingBytes + 1024 + 8 * k2Bars + 16 + k2ColBytes; }
static_assert(k2RingBytes + 1024 + 8 * k2Bars + 16 + k2ColBytes <= 227 * 1024, "shared memory budget");
static_assert((8 * k2Bars + 16) % 16 == 0, "column factors are 16-byte aligned");

bool tc2_supported(int rows_total, int K) { return rows_total % 256 == 0 && K % 128 == 0; }

template <int STAGE, int WF>
static cudaError_t launch_tc2_one(const GroupedArgs &a, int rows_total, int64_t b_rows, cudaStream_t s) {
  auto kern = k_grouped_tc2<STAGE, WF>;
  const size_t smem = tc2_smem_bytes();
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
    cfg.blockDim = dim3(k2Threads);
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
  CUtensorMap bmap;
  if ((err = encode_rows16_sw128(&bmap, a.act, (uint64_t)b_rows, (uint64_t)a.K, k2HalfRows)) != cudaSuccess)
    return err;
  return launch_pdl_cluster(kern, dim3(2 * clusters), dim3(k2Threads), smem, 2, s, g, bmap);
}

template <int WF>
static cudaError_t launch_tc2_wf(int stage, const GroupedArgs &a, int rows_total, int64_t b_rows, cudaStream_t s) {
  switch (stage) {
    case STAGE_GATED: return launch_tc2_one<STAGE_GATED, WF>(a, rows_total, b_rows, s);
    case STAGE_RELU2: return launch_tc2_one<STAGE_RELU2, WF>(a, rows_total, b_rows, s);
    case STAGE_DOWN: return launch_tc2_one<STAGE_DOWN, WF>(a, rows_total, b_rows, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_grouped_tc2(int stage, int wfmt, const GroupedArgs &a, int rows_total, int64_t b_rows,
                               cudaStream_t s) {
  if (!tc2_supported(rows_total, a.K)) return cudaErrorInvalidValue;
  if (wfmt == W_NVFP4) return launch_tc2_wf<W_NVFP4>(stage, a, rows_total, b_rows, s);
  if (wfmt == W_MXFP4) return launch_tc2_wf<W_MXFP4>(stage, a, rows_total, b_rows, s);
  return cudaErrorInvalidValue;
}

// ------------------------------------------------------------ tensor maps

cudaError_t encode_rows16_sw128(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  using Encode = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static Encode encode = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<Encode>(f);
  });
  if (!encode) return cudaErrorNotSupported;
  if (rows == 0) rows = 1;
  const cuuint64_t dim[2] = {cols, rows};
  const cuuint64_t stride[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(base), dim, stride, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// ------------------------------------------- token rows -> expert-sorted slot rows
//
// dst[s] = src[sorted_pair[s] / top_k] for every live slot s < offsets[E] (one
// warp per row), so that the pair kernel's activation tiles are contiguous
// rows, in the pair kernel's K order (the source rows are in the slot order;
// pair_order_flush transposes every 64-element step's 32 pairs as a 4 x 8
// matrix).  Padding slots are left as they are (they feed only discarded MMA
// columns).
__global__ void __launch_bounds__(256) k_gather_slot_rows(const uint4 *__restrict__ src, const int32_t *__restrict__ sorted,
                                                          const int32_t *__restrict__ n_live, int top_k, int row_chunks,
                                                          uint4 *__restrict__ dst) {
  __shared__ __align__(16) uint32_t sbuf_all[8][8 * kPairStride];
  uint32_t *sbuf = sbuf_all[threadIdx.x >> 5];
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t live = *n_live;
  const int steps = row_chunks / 8;  // 64-element steps of 8 16-byte chunks
  for (int64_t s = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); s < live; s += (int64_t)gridDim.x * 8) {
    const int p = sorted[s];
    if (p < 0) continue;
    const uint4 *a = src + (int64_t)(p / top_k) * row_chunks;
    uint4 *b = dst + s * row_chunks;
    for (int st0 = 0; st0 < steps; st0 += 8) {
      const int ns = min(8, steps - st0);
      // the eight steps' 64 chunks, two per lane, coalesced
      uint4 v[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = lane + 32 * h;
        if (c < 8 * ns) v[h] = __ldg(a + 8 * st0 + c);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = lane + 32 * h;
        if (c < 8 * ns) *reinterpret_cast<uint4 *>(sbuf + (c >> 3) * kPairStride + 4 * (c & 7)) = v[h];
      }
      __syncwarp();
      pair_order_flush(sbuf, b + 8 * st0, ns, lane);
      __syncwarp();
    }
  }
}

cudaError_t launch_gather_slot_rows(const void *src, const int32_t *sorted, const int32_t *n_live, int top_k,
                                    int cols16, int64_t cap_rows, void *dst, cudaStream_t s) {
  if (cap_rows <= 0) return cudaSuccess;
  if (cols16 % 64) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t err;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
  const int grid = (int)std::min<int64_t>((cap_rows + 7) / 8, (int64_t)sms * 8);
  return launch_pdl(k_gather_slot_rows, dim3(grid), dim3(256), 0, s, reinterpret_cast<const uint4 *>(src), sorted,
                    n_live, top_k, cols16 / 8, reinterpret_cast<uint4 *>(dst));
}

}  // namespace bqmoe
