// Grouped expert contractions on CTA pairs of the 5th-generation tensor cores
// (tcgen05.mma.cta_group::2, M = 256), for experts that receive many tokens.
//
// moe.fused_moe's W4A16 mode (BF16 activations against FP4 weights dequantised
// in the kernel) and its MXFP4 experts (b12x project page, section "What's in
// here").  The contraction of an expert is a dense GEMM once it sees more than
// a few dozen tokens.  On one SM an M=128 N=128 K=16 MMA reads 8 KB of
// operands from shared memory while the producers write the dequantised
// weight tile and the gathered activation tile through the same port, so a
// single-CTA kernel is held by shared-memory bandwidth well below the tensor
// pipe's rate.  Here two CTAs of a cluster form one MMA: each holds 128 weight
// rows (its A half) and half of the token tile (its B half), and the leader
// CTA issues M=256 N<=256 K=16 MMAs that read both CTAs' shared memory, so
// every byte written to shared memory feeds twice the FLOPs:
//
//   D[256 weight rows x N tokens] += A[256 x 64] * B[N x 64]^T per 64-K block
//
// * A: each CTA's 128-row block of the packed experts (the same fragment-order
//   bytes the decode kernel streams), loaded four k-blocks ahead into
//   registers by eight producer warps, dequantised to FP16 (NVFP4: E2M1 x E4M3
//   is exact) or BF16 (MXFP4: E2M1 x 2^X is exact) and written in the UMMA
//   K-major 128-byte-swizzled layout.
// * B: N/2 activation rows per CTA (FP16 slot-order rows with a power-of-two
//   factor, or BF16), gathered by two producer warps with cp.async and
//   zero-filled past the tile's last token.
// * Token tiles: an expert with c pairs is cut into ceil(c / 256) tiles of
//   equal size (rounded up to 16), so no tile is a nearly empty remainder;
//   the MMA's N is the tile's size rounded up to 16.
// * The leader's MMA thread waits for both CTAs' producers (they arrive on the
//   leader's mbarriers across the cluster), issues 4 MMAs per k-block into one
//   of two TMEM accumulators (2 x 256 columns) and releases the stages of both
//   CTAs with a multicast tcgen05.commit; each CTA's four epilogue warps read
//   their 128 rows of the accumulator (SiLU(gate)*up, ReLU^2, or the
//   topk_weight scaling of the down projection) while the next tile's MMAs run.
// * Work items are (large expert, token tile, pair of 128-row blocks), dealt
//   round-robin over persistent clusters (one CTA per SM).
// * Every wait is a bounded mbarrier wait; on a timeout the kernel sets the
//   status flag, every CTA still reaches the final cluster barrier, and the
//   leader drains its MMAs before the pair's tensor memory is released.
#include <algorithm>

#include "common.cuh"
#include "dequant.cuh"
#include "internal.h"
#include "launch.h"
#include "sync.cuh"
#include "tcgen05.cuh"

namespace bqmoe {

constexpr int k2EpiWarps = 4, k2AWarps = 8, k2BWarps = 2;
constexpr int k2MmaWarp = k2EpiWarps + k2AWarps + k2BWarps;  // warp 14
constexpr int k2Threads = (k2MmaWarp + 1) * 32;
constexpr int k2MaxN = 256;                 // tokens per pair tile
constexpr int k2HalfRows = k2MaxN / 2;      // B rows per CTA
constexpr int k2ABytes = 128 * 64 * 2;      // one 128 x 64 16-bit block
constexpr int k2BBytes = k2HalfRows * 64 * 2;
constexpr int k2AStages = 4;
constexpr int k2BStages = 6;
constexpr int k2BLag = 4;                   // cp.async stages a B thread keeps in flight
constexpr int k2APrefetch = 4;              // k-blocks of packed A bytes an A thread keeps in flight
constexpr int k2RingBytes = k2AStages * k2ABytes + k2BStages * k2BBytes;
constexpr int k2AccCols = k2MaxN;           // TMEM columns per accumulator buffer
constexpr int k2TmemCols = 2 * k2AccCols;   // double buffered
constexpr int k2BRows = k2HalfRows * 8 / (k2BWarps * 32);  // 16-byte chunks per B thread per k-block
constexpr int k2Bars = 2 * k2AStages + 2 * k2BStages + 4 + 1;
static_assert(k2AWarps * 32 == 8 * 32, "one fragment chunk per A thread per k-block");

// ------------------------------------------------------------ cluster helpers

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Shared-memory address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_c(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait with cluster-scope acquire (arrivals come from the peer CTA
// and from the pair's tensor-core commits); false on timeout.
__device__ __forceinline__ bool mbar_wait_c(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait_c(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_c(bar, parity)) return true;
    if ((it & 255u) == 0 && globaltimer_ns() - t0 > kWaitNs) return false;
  }
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ void tc2_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
// Arrive (once the pair's earlier MMAs have completed) on the mbarrier at the
// same offset in both CTAs of the pair.
__device__ __forceinline__ void tc2_commit_both(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}

// ------------------------------------------------------------------ work items

struct Tc2Item {
  int e, s0, ntok, n, bp;  // expert, first slot, live tokens, MMA N, row-block pair
};

// Items (large expert i, token tile, row-block pair), in that order;
// tiles[i] is the per-expert prefix of ceil(count / 256).  An expert's tiles
// have equal sizes (a multiple of 16), the last one possibly shorter.
struct Tc2Cursor {
  int i = 0;
  __device__ __forceinline__ void seek(const GroupedArgs &a, int w, int nbp) {
    int lo = 0, hi = a.large[0] - 1;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (a.large_tiles[mid + 1] * nbp > w) hi = mid;
      else lo = mid + 1;
    }
    i = lo;
  }
  __device__ __forceinline__ Tc2Item at(const GroupedArgs &a, int w, int nbp) {
    while (a.large_tiles[i + 1] * nbp <= w) ++i;
    Tc2Item it;
    it.e = a.large[1 + i];
    const int nt = a.large_tiles[i + 1] - a.large_tiles[i];
    const int local = w - a.large_tiles[i] * nbp;
    const int tile = local / nbp;
    it.bp = local % nbp;
    const int cnt = a.counts[it.e];
    const int tsz = (((cnt + nt - 1) / nt) + 15) & ~15;
    it.s0 = a.offsets[it.e] + tile * tsz;
    it.ntok = max(0, min(tsz, cnt - tile * tsz));
    it.n = max(16, (it.ntok + 15) & ~15);
    return it;
  }
};

// ------------------------------------------------------------------ kernel

template <int STAGE, int WF>
__global__ void __launch_bounds__(k2Threads, 1) k_grouped_tc2(const GroupedArgs a) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base for the swizzled tiles (the same offset in both CTAs)
  const uint32_t raw_s = (uint32_t)__cvta_generic_to_shared(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t *base = smem_raw + (base_s - raw_s);
  const uint32_t ringA = base_s, ringB = base_s + k2AStages * k2ABytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(base + k2RingBytes);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + k2Bars);
  const uint32_t afull0 = (uint32_t)__cvta_generic_to_shared(bars);
  const uint32_t aempty0 = afull0 + 8u * k2AStages;
  const uint32_t bfull0 = aempty0 + 8u * k2AStages;
  const uint32_t bempty0 = bfull0 + 8u * k2BStages;
  const uint32_t tfull0 = bempty0 + 8u * k2BStages;  // 2
  const uint32_t tempty0 = tfull0 + 16u;             // 2
  const uint32_t drain = tempty0 + 16u;              // 1

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();  // 0: leader (issues the MMAs), 1: peer
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int i = 0; i < k2AStages; ++i) {
      mbar_init(afull0 + 8u * i, 2 * k2AWarps);
      mbar_init(aempty0 + 8u * i, 1);
    }
    for (int i = 0; i < k2BStages; ++i) {
      mbar_init(bfull0 + 8u * i, 2 * k2BWarps);
      mbar_init(bempty0 + 8u * i, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull0 + 8u * b, 1);
      mbar_init(tempty0 + 8u * b, 2 * k2EpiWarps);
    }
    mbar_init(drain, 1);
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
  Tc2Cursor cur;
  if (w0 < W) cur.seek(a, w0, nbp);
  bool ok = true;
  bool any_mma = false;

  if (warp >= k2EpiWarps && warp < k2EpiWarps + k2AWarps) {
    // ------------------------------------------------------ A producers
    // Lane t holds fragment chunk t of the k-block (16-row tile t / 32, lane
    // t % 32): 16 code bytes and its lane group's block scales, dequantised to
    // 16-bit values written at their slot positions in the swizzled tile.
    constexpr int SB = WF == W_NVFP4 ? 4608 : 4352;  // bytes of one 64-K step of a block
    const int t = threadIdx.x - k2EpiWarps * 32;    // 0..255
    const int tile = t >> 5, ln = t & 31;
    const int g = ln >> 2, c4 = ln & 3;
    const int r0 = 16 * tile + g, r1 = r0 + 8;
    const uint32_t afull_leader = mapa(afull0, 0);
    int slot = 0;
    uint32_t phase = 0;
    uint4 pch[k2APrefetch];
    uint2 psc[k2APrefetch];
    auto load = [&](const Tc2Item &it, int kb, uint4 &c, uint2 &s) {
      const int blk = 2 * it.bp + (int)rank;
      const uint8_t *step = a.codes + (size_t)it.e * a.codes_expert + ((size_t)blk * nk + kb) * SB;
      c = __ldg(reinterpret_cast<const uint4 *>(step + tile * 512 + ln * 16));
      if (WF == W_NVFP4) s = __ldg(reinterpret_cast<const uint2 *>(step + 4096 + tile * 64 + (ln >> 2) * 8));
      else s = make_uint2(__ldg(reinterpret_cast<const uint32_t *>(step + 4096 + tile * 32 + (ln >> 2) * 4)), 0u);
    };
    Tc2Cursor pcur = cur;  // cursor of the prefetch (k2APrefetch k-blocks ahead)
    int pw = w0, pkb = 0;
    bool pv = pw < W;
    Tc2Item pit;
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
    for (int d = 0; d < k2APrefetch; ++d) {
      if (pv) load(pit, pkb, pch[d], psc[d]);
      advance();
    }
    for (int w = w0; w < W && ok; w += wstep) {
      for (int kb = 0; kb < nk; ++kb) {
        const uint4 cch = pch[0];
        const uint2 sch = psc[0];
#pragma unroll
        for (int d = 0; d + 1 < k2APrefetch; ++d) {
          pch[d] = pch[d + 1];
          psc[d] = psc[d + 1];
        }
        if (pv) load(pit, pkb, pch[k2APrefetch - 1], psc[k2APrefetch - 1]);
        advance();
        if (!mbar_wait_c(aempty0 + 8u * slot, phase ^ 1u)) {
          ok = false;
          break;
        }
        uint8_t *tileA = base + (size_t)slot * k2ABytes;
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
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int k = 16 * j + 2 * c4;
          *reinterpret_cast<uint32_t *>(tileA + sw128_elem(r0, k)) = o[j][0];
          *reinterpret_cast<uint32_t *>(tileA + sw128_elem(r1, k)) = o[j][1];
          *reinterpret_cast<uint32_t *>(tileA + sw128_elem(r0, k + 8)) = o[j][2];
          *reinterpret_cast<uint32_t *>(tileA + sw128_elem(r1, k + 8)) = o[j][3];
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(afull_leader + 8u * slot);
        if (++slot == k2AStages) {
          slot = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp >= k2EpiWarps + k2AWarps && warp < k2MmaWarp) {
    // ------------------------------------------------------ B producers
    const int t = threadIdx.x - (k2EpiWarps + k2AWarps) * 32;  // 0..63
    const int cc = t & 7;                                      // 16-byte chunk of the row
    constexpr int kRowStep = k2BWarps * 32 / 8;                // rows between a thread's chunks
    const bool by_token = a.act_by_token != 0;
    const uint32_t bfull_leader = mapa(bfull0, 0);
    int slot = 0, issued = 0;
    uint32_t phase = 0;
    const __half *act = reinterpret_cast<const __half *>(a.act);
    pdl_wait();  // activation rows come from the preceding kernels
    for (int w = w0; w < W && ok; w += wstep) {
      const Tc2Item it = cur.at(a, w, nbp);
      const int half = it.n >> 1;  // rows of this CTA's B half
      int rid[k2BRows];
#pragma unroll
      for (int i = 0; i < k2BRows; ++i) {
        const int r = (t >> 3) + kRowStep * i;
        const int n = (int)rank * half + r;  // token of the tile
        rid[i] = (r < half && n < it.ntok) ? (by_token ? a.sorted_pair[it.s0 + n] / a.top_k : it.s0 + n)
                                           : (r < half ? -1 : -2);
      }
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait_c(bempty0 + 8u * slot, phase ^ 1u)) {
          ok = false;
          break;
        }
        const uint32_t stB = ringB + (uint32_t)slot * k2BBytes;
#pragma unroll
        for (int i = 0; i < k2BRows; ++i) {
          if (rid[i] == -2) continue;  // beyond the rows the MMA reads
          const int r = (t >> 3) + kRowStep * i;
          const uint32_t dst = stB + (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + (((cc ^ r) & 7) << 4));
          const __half *src = act + (int64_t)(rid[i] < 0 ? 0 : rid[i]) * K + kb * 64 + cc * 8;
          cp_async16(dst, src, rid[i] >= 0);
        }
        cp_async_commit();
        ++issued;
        if (issued > k2BLag) {  // the stage issued k2BLag steps ago has landed: hand it to the MMA
          cp_async_wait_group<k2BLag>();
          fence_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(bfull_leader + 8u * ((slot + k2BStages - k2BLag) % k2BStages));
        }
        if (++slot == k2BStages) {
          slot = 0;
          phase ^= 1u;
        }
      }
    }
    cp_async_wait_group<0>();
    fence_async_smem();
    __syncwarp();
    if (ok && lane == 0) {  // the last k2BLag stages
      for (int back = issued < k2BLag ? issued : k2BLag; back >= 1; --back)
        mbar_arrive_remote(bfull_leader + 8u * ((slot + k2BStages - back) % k2BStages));
    }
  } else if (warp == k2MmaWarp) {
    // ------------------------------------------------------ MMA issuer (leader CTA)
    if (rank == 0 && lane == 0) {
      constexpr uint32_t fmt = WF == W_MXFP4 ? 1u : 0u;  // operand type: 0 = F16, 1 = BF16
      const uint32_t idesc0 = (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(256 >> 4) << 24);
      int sa = 0, sb = 0, li = 0;
      uint32_t pa = 0, pb = 0;
      for (int w = w0; w < W && ok; w += wstep, ++li) {
        const Tc2Item it = cur.at(a, w, nbp);
        const uint32_t idesc = idesc0 | ((uint32_t)(it.n >> 3) << 17);
        const int b = li & 1;
        if (!mbar_wait_c(tempty0 + 8u * b, ((li >> 1) & 1) ^ 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem + (uint32_t)(b * k2AccCols);
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_c(afull0 + 8u * sa, pa) || !mbar_wait_c(bfull0 + 8u * sb, pb)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t da = umma_desc_sw128(ringA + (uint32_t)sa * k2ABytes);
          const uint64_t db = umma_desc_sw128(ringB + (uint32_t)sb * k2BBytes);
#pragma unroll
          for (int j = 0; j < 4; ++j)  // K = 16 per MMA: advance the start address by 32 bytes
            tc2_mma_f16(d0, da + 2u * j, db + 2u * j, idesc, (kb > 0 || j > 0) ? 1u : 0u);
          tc2_commit_both(aempty0 + 8u * sa);  // frees both CTAs' stages once these MMAs have read them
          tc2_commit_both(bempty0 + 8u * sb);
          any_mma = true;
          if (++sa == k2AStages) {
            sa = 0;
            pa ^= 1u;
          }
          if (++sb == k2BStages) {
            sb = 0;
            pb ^= 1u;
          }
        }
        if (!ok) break;
        tc2_commit_both(tfull0 + 8u * b);
      }
      // Every MMA of the pair completes before either CTA releases its shared
      // memory or the pair's tensor memory.
      if (any_mma) {
        tc2_commit_both(drain);
      } else {
        mbar_arrive(drain);
        mbar_arrive_remote(mapa(drain, 1));
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------ epilogue (both CTAs)
    const int m = warp * 32 + lane;  // accumulator row = TMEM lane
    const float *gl_all = a.globals;
    const uint32_t tempty_leader = mapa(tempty0, 0);
    pdl_wait();  // row factors come from the preceding kernels
    int li = 0;
    for (int w = w0; w < W && ok; w += wstep, ++li) {
      const Tc2Item it = cur.at(a, w, nbp);
      const int b = li & 1;
      if (!mbar_wait_c(tfull0 + 8u * b, (li >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float *gl = gl_all + 4 * it.e;
      const int blk = 2 * it.bp + (int)rank;
      const int tile = 8 * blk + (m >> 4), rr = m & 15;
      for (int c0 = 0; c0 < it.n; c0 += 32) {
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
        tc_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(b * k2AccCols + c0), raw);
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
              hv[j] = live ? fabsf(h) : 0.f;
            }
          } else if (STAGE == STAGE_RELU2) {
            const float r = fmaxf(v * gl[0], 0.f);
            if (live) a.out[(size_t)s * a.n_rows + tile * 16 + rr] = r * r;
            hv[j] = live ? r * r : 0.f;
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
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(tempty_leader + 8u * b);
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

static size_t tc2_smem_bytes() { return (size_t)k2RingBytes + 1024 + 8 * k2Bars + 16; }
static_assert(k2RingBytes + 1024 + 8 * k2Bars + 16 <= 227 * 1024, "shared memory budget");

bool tc2_supported(int rows_total, int K) { return rows_total % 256 == 0 && K % 64 == 0; }

template <int STAGE, int WF>
static cudaError_t launch_tc2_one(const GroupedArgs &a, int rows_total, cudaStream_t s) {
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
  return launch_pdl_cluster(kern, dim3(2 * clusters), dim3(k2Threads), smem, 2, s, g);
}

template <int WF>
static cudaError_t launch_tc2_wf(int stage, const GroupedArgs &a, int rows_total, cudaStream_t s) {
  switch (stage) {
    case STAGE_GATED: return launch_tc2_one<STAGE_GATED, WF>(a, rows_total, s);
    case STAGE_RELU2: return launch_tc2_one<STAGE_RELU2, WF>(a, rows_total, s);
    case STAGE_DOWN: return launch_tc2_one<STAGE_DOWN, WF>(a, rows_total, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_grouped_tc2(int stage, int wfmt, const GroupedArgs &a, int rows_total, cudaStream_t s) {
  if (!tc2_supported(rows_total, a.K)) return cudaErrorInvalidValue;
  if (wfmt == W_NVFP4) return launch_tc2_wf<W_NVFP4>(stage, a, rows_total, s);
  if (wfmt == W_MXFP4) return launch_tc2_wf<W_MXFP4>(stage, a, rows_total, s);
  return cudaErrorInvalidValue;
}

}  // namespace bqmoe
