// Body of the register-dequant grouped kernel (see k_grouped_mma.cu), as a
// device function shared by its stand-alone launches and by the single-launch
// decode forward.
#pragma once

#include "common.cuh"
#include "dequant.cuh"
#include "internal.h"
#include "sync.cuh"

namespace bqmoe {

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The same with a zero accumulator input (a fresh partial sum).
__device__ __forceinline__ void mma_16816_zc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x2(uint32_t addr, uint32_t &r0, uint32_t &r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

// ------------------------------------------------------------ grouped kernel
//
// Persistent, one CTA per SM: warp 8 is the producer, warps 0-7 the consumers.
// The work list is every (expert with pairs, 128-row block) of the stage; CTA c
// takes a contiguous range of it, so consecutive units usually share an expert
// and its staged activations.  The producer streams each unit's packed bytes
// (4608 per 64-K step: codes + scales of the whole 128-row block) with 1-D bulk
// copies (cp.async.bulk, completion on an mbarrier) into a ring of shared-memory
// stages, up to the ring's depth ahead of the consumers, across unit
// boundaries.  Consumer warp w dequantises tile w of each step straight into
// mma fragments.  Every mbarrier wait is bounded: on timeout the status word
// gets MOE timeout flag, the warp stops, and the producer waits (bounded) for
// its own copies in flight before the CTA exits.

constexpr int kConsumers = 8;
constexpr int kTmaThreads = (kConsumers + 1) * 32;
// One 64-K step of a 128-row block: 4096 code bytes + block scales (NVFP4 512,
// MXFP4 256).  Ring stages are sized for the larger.
template <int WF>
constexpr int step_bytes() { return WF == W_NVFP4 ? 4608 : 4352; }
constexpr int kStepBytes = 4608;
constexpr int kSPS = 4;           // K steps per ring stage
constexpr int kStageBytes = kStepBytes * kSPS;
constexpr int kMaxStages = 8;
constexpr int kQueue = 8;         // item ids handed from the producer to the consumers
constexpr int kQEntry = 8 + 2 * 16;  // ints per queue entry: unit, item fields, rows[16], weights[16]
// Two 9-warp CTAs per SM put five warps on some SM sub-partitions, whose
// register files hold 16K registers each: 5 x 32 x 96 <= 16384.
constexpr int kMmaMaxRegs = 96;
// Barrier among the consumer warps only (the producer never joins), built on an
// mbarrier so that its wait is bounded too.  Lane 0 of each warp arrives after
// the warp's own shared-memory writes and cp.async copies are complete.
__device__ __forceinline__ bool consumer_sync(uint32_t cbar, uint32_t &cphase) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(cbar);
  const bool ok = mbar_wait(cbar, cphase);
  cphase ^= 1u;
  __syncwarp();
  return ok;
}

// A work item is (active expert i, pass, 128-row block), ordered that way, so
// consecutive items share staged activations.  passes[] is the per-expert
// prefix of passes written by the routing kernel.
struct Item {
  int e, pass, blk, cnt, off;
};

struct ItemCursor {
  int i = 0;  // active-expert index of the current item
  // Called by all 32 lanes of a warp.  i = the smallest i < n_active with
  // passes[i+1] * nblk > w (else n_active - 1): passes is a non-decreasing
  // prefix, so that is the number of entries at or below w, counted over the
  // whole list in one round of independent loads (n_active <= kMaxExperts).
  __device__ __forceinline__ void seek(const GroupedArgs &a, int w, int nblk, int n_active) {
    const int lane = threadIdx.x & 31;
    int cnt = 0;
#pragma unroll
    for (int j = 0; j < kMaxExperts / 32; ++j) {
      const int e = lane + 32 * j;
      if (e < n_active && a.passes[e + 1] * nblk <= w) ++cnt;
    }
    cnt = __reduce_add_sync(0xffffffffu, cnt);
    i = min(cnt, n_active - 1);
  }
  __device__ __forceinline__ Item at(const GroupedArgs &a, int w, int nblk) {
    while (a.passes[i + 1] * nblk <= w) ++i;
    Item it;
    it.e = a.active[1 + i];
    const int local = w - a.passes[i] * nblk;
    it.pass = local / nblk;
    it.blk = local % nblk;
    it.cnt = a.counts[it.e];
    it.off = a.offsets[it.e];
    return it;
  }
};

// The grouped kernel's body, shared by the stand-alone launches (PDL: with the
// programmatic-dependent-launch protocol) and the phases of the single-launch
// decode forward (CTA `cta` of `ncta`, shared memory at `smem`, 1024-byte
// aligned).  Every thread of the CTA calls it.
template <int WF, int SRC, int STAGE, int NT, bool PDL>
__device__ __forceinline__ void grouped_mma_run(const GroupedArgs &a, int nst, int ngroups, uint8_t *smem, int cta,
                                                int ncta) {
  constexpr int NTOK = 8 * NT;
  const int K = a.K;
  const int pitch = 2 * K + 16;  // bytes per staged activation row; +16 keeps ldmatrix conflict-free
  uint8_t *ring = smem;
  __half *xs = reinterpret_cast<__half *>(smem + (size_t)nst * kStageBytes);
  float *fac = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(xs) + (size_t)NTOK * pitch);
  int64_t *rows = reinterpret_cast<int64_t *>(fac + NTOK);
  float *wts = reinterpret_cast<float *>(rows + NTOK);  // GEMM2: topk weight x down global per staged token
  // full[nst], empty[nst], consumer barrier, item queue full[kQueue] / empty[kQueue]
  uint64_t *bars = reinterpret_cast<uint64_t *>(wts + NTOK);
  // item queue entries: unit id (-1: no more), then the item's expert, pass, row
  // block, pair count and sorted offset (the producer has them, the consumers
  // would otherwise re-read the routing arrays at every item)
  volatile int *qitem = reinterpret_cast<volatile int *>(bars + 2 * nst + 1 + 2 * kQueue);
  const uint32_t ring_s = (uint32_t)__cvta_generic_to_shared(ring);
  const uint32_t full0 = (uint32_t)__cvta_generic_to_shared(bars);
  const uint32_t empty0 = full0 + 8u * nst;
  const uint32_t cbar = empty0 + 8u * nst;
  const uint32_t qfull0 = cbar + 8u, qempty0 = qfull0 + 8u * kQueue;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // With BF16 x, routing stages the x rows and triggers its dependents on
  // entry, and GEMM1 follows it directly: GEMM1 then waits before its first
  // read of a routing output and triggers only after that wait, so every later
  // kernel still starts after routing has completed.  Otherwise (GEMM2, or
  // GEMM1 behind the activation quantisers, whose routing never triggered
  // early) the kernel triggers on entry and the producer streams weights while
  // the predecessor finishes.
  const bool wait_first = PDL && SRC == SRC_X16 && a.wait_first;
  if (PDL && !wait_first) pdl_trigger();
  if (threadIdx.x == 0) {
    for (int i = 0; i < nst; ++i) {
      mbar_init(full0 + 8u * i, 1);
      mbar_init(empty0 + 8u * i, kConsumers);
    }
    mbar_init(cbar, kConsumers);
    for (int i = 0; i < kQueue; ++i) {
      mbar_init(qfull0 + 8u * i, 1);
      mbar_init(qempty0 + 8u * i, kConsumers);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (wait_first) {
    pdl_wait();
    pdl_trigger();
  }

  const int nsteps = K / 64;
  const int nblk = a.n_blocks;
  const int n_active = a.active[0];
  const int W = n_active > 0 ? a.passes[n_active] * nblk : 0;
  // CTA group g = CTA index % ngroups (the CTAs that share an SM when the grid
  // is ctas-per-SM x SMs) owns the contiguous items [u0, u1) and its CTAs take
  // them one at a time from the group's counter, so a CTA the warp scheduler
  // serves less simply takes fewer items; neighbouring items share staged
  // activations.
  const int grp = cta % ngroups;
  const int u0 = (int)((int64_t)grp * W / ngroups);
  const int u1 = (int)((int64_t)(grp + 1) * W / ngroups);
  int32_t *const ctr = a.work + grp;
  const int stages_per_pass = (nsteps + kSPS - 1) / kSPS;
  ItemCursor cur;
  if (u0 < u1) cur.seek(a, u0, nblk, n_active);

  if (warp == kConsumers) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int slot = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;  // per-slot: has a copy, parity of its last phase
      bool ok = true;
      int q = 0;
      uint32_t qph = 0;
      // the CTA's first item is its rank in the group (no atomic on the way to
      // the first copy); later ones come from the counter, past those
      const int rank = cta / ngroups;
      const int in_grp = (ncta - 1 - grp) / ngroups + 1;
      int u = u0 + rank;
      int last_e = -1, last_pass = -1;
      constexpr bool by_token_src = SRC == SRC_X16;
      for (;;) {
        if (u >= u1) u = -1;
        Item w;
        if (u >= 0) w = cur.at(a, u, nblk);
        // hand the item to the consumers (-1: no more)
        if (!mbar_wait(qempty0 + 8u * q, qph ^ 1u)) {
          ok = false;
          break;
        }
        if (u >= 0) {
          volatile int *qe = qitem + kQEntry * q;
          qe[1] = w.e;
          qe[2] = w.pass;
          qe[3] = w.blk;
          qe[4] = w.cnt;
          qe[5] = w.off;
          if (w.e != last_e || w.pass != last_pass) {
            // the pass's activation rows (token or slot ids, -1 past the
            // expert's pairs) and, for the down projection, topk_weight x g_down
            const int s0 = w.off + w.pass * NTOK;
            const int ntok = min(NTOK, w.off + w.cnt - s0);
            int pr[NTOK];
#pragma unroll
            for (int n = 0; n < NTOK; ++n) pr[n] = n < ntok ? a.sorted_pair[s0 + n] : -1;
            const float gd = STAGE == STAGE_DOWN ? a.globals[4 * w.e + 2] : 0.f;
#pragma unroll
            for (int n = 0; n < NTOK; ++n) {
              qe[8 + n] = pr[n] < 0 ? -1 : (by_token_src ? pr[n] / a.top_k : s0 + n);
              float wt = 0.f;
              if (STAGE == STAGE_DOWN && pr[n] >= 0) wt = a.topk_weights[pr[n]] * gd;
              reinterpret_cast<volatile float *>(qe)[8 + NTOK + n] = wt;
            }
            last_e = w.e;
            last_pass = w.pass;
          }
        }
        qitem[kQEntry * q] = u;
        mbar_arrive(qfull0 + 8u * q);
        if (++q == kQueue) {
          q = 0;
          qph ^= 1u;
        }
        if (u < 0) break;
        const int un = u0 + in_grp + atomicAdd(ctr, 1);  // the next item, fetched while this one streams
        const uint8_t *base = a.codes + (size_t)w.e * a.codes_expert + (size_t)w.blk * nsteps * step_bytes<WF>();
        for (int st = 0; st < stages_per_pass; ++st) {
          if (!mbar_wait(empty0 + 8u * slot, phase ^ 1u)) {
            ok = false;
            break;
          }
          const uint32_t bytes = (uint32_t)min(kSPS, nsteps - st * kSPS) * step_bytes<WF>();
          mbar_expect_tx(full0 + 8u * slot, bytes);
          bulk_g2s(ring_s + (uint32_t)slot * kStageBytes, base + (size_t)st * kSPS * step_bytes<WF>(), bytes,
                   full0 + 8u * slot);
          issued |= 1u << slot;
          issued_parity = (issued_parity & ~(1u << slot)) | (phase << slot);
          if (++slot == nst) {
            slot = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        u = un;
      }
      if (!ok) atomicOr(&a.status[ST_FLAGS], ST_FLAG_TIMEOUT);
      // Never leave with a copy in flight into this CTA's shared memory.
      for (int i = 0; i < nst; ++i)
        if (issued & (1u << i)) mbar_wait(full0 + 8u * i, (issued_parity >> i) & 1u);
    }
    if (PDL) pdl_wait();  // the producer only read routing outputs and weights; complete after the predecessor
    return;
  }

  // ------------------------------------------------------------- consumers
  const uint32_t xs_base = (uint32_t)__cvta_generic_to_shared(xs);
  // ldmatrix row addresses: lanes 0-7 rows 0-7 at k, 8-15 rows 0-7 at k+8,
  // 16-23 rows 8-15 at k, 24-31 rows 8-15 at k+8.
  const int lrow = (lane & 7) + ((lane >> 4) << 3);
  const uint32_t b_addr = xs_base + lrow * pitch + ((lane >> 3) & 1) * 16;
  const int r = lane >> 2;
  int slot = 0;
  uint32_t phase = 0;
  int staged_e = -1, staged_pass = -1;
  uint32_t cphase = 0;
  bool ok = true;
  if (PDL) pdl_wait();  // activations / h come from the preceding kernels

  int q = 0;
  uint32_t qph = 0;
  while (ok) {
    if (!mbar_wait(qfull0 + 8u * q, qph)) {
      ok = false;
      break;
    }
    const volatile int *qe = qitem + kQEntry * q;
    const uint32_t qe_bar = qempty0 + 8u * q;
    const int u = qe[0];
    Item w;
    w.e = qe[1];
    w.pass = qe[2];
    w.blk = qe[3];
    w.cnt = qe[4];
    w.off = qe[5];
    if (++q == kQueue) {
      q = 0;
      qph ^= 1u;
    }
    if (u < 0) {
      __syncwarp();
      if (lane == 0) mbar_arrive(qe_bar);
      break;
    }
    const int tile = w.blk * kConsumers + warp;  // 16-row tile of this warp
    // the expert's globals, loaded while the item's K loop runs
    const float gl0 = a.globals[4 * w.e], gl1 = a.globals[4 * w.e + 1];
    {
      const int pass = w.pass;
      const int s0 = w.off + pass * NTOK;
      const int ntok = min(NTOK, w.off + w.cnt - s0);
      if (w.e != staged_e || pass != staged_pass) {
        // Stage NTOK activation rows as FP16 (warp j: rows j, j+8, ...).
        if (!consumer_sync(cbar, cphase)) {  // everyone is done with the previous rows
          ok = false;
          break;
        }
        if (threadIdx.x < NTOK) {  // the rows and weights the producer looked up
          rows[threadIdx.x] = qe[8 + threadIdx.x];
          wts[threadIdx.x] = reinterpret_cast<const volatile float *>(qe)[8 + NTOK + threadIdx.x];
        }
        if (!consumer_sync(cbar, cphase)) {
          ok = false;
          break;
        }
        for (int j = warp; j < NTOK; j += kConsumers) {
          const int64_t rid = rows[j];
          uint8_t *dst = reinterpret_cast<uint8_t *>(xs) + (size_t)j * pitch;
          if (SRC == SRC_X16) {
            const __half *src = reinterpret_cast<const __half *>(a.act) + (rid < 0 ? 0 : rid) * K;
            const uint32_t d0 = (uint32_t)__cvta_generic_to_shared(dst);
            for (int k = lane * 8; k < K; k += 256) cp_async16(d0 + 2 * k, src + k, rid >= 0);
            if (lane == 0) fac[j] = rid < 0 ? 0.f : a.act_g[rid];
            continue;
          }
          if (rid < 0) {
            for (int k = lane * 8; k < K; k += 256) *reinterpret_cast<uint4 *>(dst + 2 * k) = make_uint4(0, 0, 0, 0);
            if (lane == 0) fac[j] = 0.f;
            continue;
          }
          float f;
          if (SRC == SRC_H_NVFP4) {
            f = a.act_g[rid];
          } else if (SRC == SRC_H_F32) {
            f = stage_factor(a.act_g[rid]);  // the |h| maximum GEMM1 recorded for this pair
          } else {
            float m = 0.f;
            for (int k = lane * 8; k < K; k += 256) {
              float v[8];
              src_load8<SRC>(a.act, a.act_scales, rid, k, K, v);
#pragma unroll
              for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
            }
            f = stage_factor(warp_max(m));
          }
          const float inv = SRC == SRC_H_NVFP4 ? 1.f : __frcp_rn(f);
          if (WF == W_NVFP4 || NT == 1)  // (MXFP4 with 16-token passes would spill)
            stage_row_slots_x2<SRC>(a.act, a.act_scales, rid, K, inv, reinterpret_cast<__half *>(dst), lane, 32);
          else
            stage_row_slots<SRC>(a.act, a.act_scales, rid, K, inv, reinterpret_cast<__half *>(dst), lane, 32);
          if (lane == 0) fac[j] = f;
        }
        if (SRC == SRC_X16) cp_async_wait_all();
        if (!consumer_sync(cbar, cphase)) {
          ok = false;
          break;
        }
        staged_e = w.e;
        staged_pass = pass;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(qe_bar);  // done with this queue entry

      // Two accumulator sets (even / odd k16 sub-steps) halve the dependent mma chain.
      float acc[NT][4], acc2[NT][4];
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[j][c] = acc2[j][c] = 0.f;

      for (int st = 0; st < stages_per_pass; ++st) {
        if (!mbar_wait(full0 + 8u * slot, phase)) {
          ok = false;
          break;
        }
        // This warp's fragment chunks of the stage, and the B row address of its first step.
        const uint8_t *stage = ring + (size_t)slot * kStageBytes + warp * 512 + lane * 16;
        const uint32_t bq = b_addr + (uint32_t)(st * kSPS * 64 * 2);
        const int nq = min(kSPS, nsteps - st * kSPS);
        auto step = [&](int i4) {
          constexpr int SB = step_bytes<WF>();
          const uint4 c = *reinterpret_cast<const uint4 *>(stage + i4 * SB);
          const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
          if (WF == W_NVFP4) {
            const uint2 sc = *reinterpret_cast<const uint2 *>(stage + i4 * SB + 4096 - warp * 448 - lane * 16 + r * 8);
            // f16x2 scale multipliers: (block 0, block 1) and (block 2, block 3) of rows r and r + 8
            uint32_t spairs[4];
            e4m3x4_to_f16x2x2(sc.x, spairs[0], spairs[1]);
            e4m3x4_to_f16x2x2(sc.y, spairs[2], spairs[3]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t s_lo = spairs[2 * (i >> 1)];      // row r
              const uint32_t s_hi = spairs[2 * (i >> 1) + 1];  // row r + 8
              uint32_t af[4];
              e2m1x8_to_f16x2x4(cw[i], af);
              af[0] = hmul2(af[0], s_lo);
              af[1] = hmul2(af[1], s_hi);
              af[2] = hmul2(af[2], s_lo);
              af[3] = hmul2(af[3], s_hi);
              const uint32_t kb = bq + (uint32_t)(i4 * 64 + i * 16) * 2;
              float(&ac)[NT][4] = (i & 1) ? acc2 : acc;
              if (NT == 2) {
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4(kb, b0, b1, b2, b3);
                mma_16816(ac[0], af, b0, b1);
                mma_16816(ac[NT - 1], af, b2, b3);
              } else {
                uint32_t b0, b1;
                ldmatrix_x2(kb, b0, b1);
                mma_16816(ac[0], af, b0, b1);
              }
            }
          } else {
            // MXFP4: mma 0-1 and 2-3 of the step each lie in one 32-element block
            // (slot order); the E2M1 codes go in unscaled (exact in FP16) and the
            // block's E8M0 scale 2^X multiplies the two mmas' FP32 partial sum.
            const uint32_t sw = *reinterpret_cast<const uint32_t *>(stage + i4 * SB + 4096 - warp * 480 - lane * 16 + r * 4);
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
              const float s_lo = e8m0_to_f32((sw >> (8 * hb)) & 0xFFu);        // row r
              const float s_hi = e8m0_to_f32((sw >> (16 + 8 * hb)) & 0xFFu);   // row r + 8
              float t[NT][4];
#pragma unroll
              for (int ii = 0; ii < 2; ++ii) {
                const int i = 2 * hb + ii;
                uint32_t af[4];
                e2m1x8_to_f16x2x4(cw[i], af);
                const uint32_t kb = bq + (uint32_t)(i4 * 64 + i * 16) * 2;
                if (NT == 2) {
                  uint32_t b0, b1, b2, b3;
                  ldmatrix_x4(kb, b0, b1, b2, b3);
                  if (ii == 0) {
                    mma_16816_zc(t[0], af, b0, b1);
                    mma_16816_zc(t[NT - 1], af, b2, b3);
                  } else {
                    mma_16816(t[0], af, b0, b1);
                    mma_16816(t[NT - 1], af, b2, b3);
                  }
                } else {
                  uint32_t b0, b1;
                  ldmatrix_x2(kb, b0, b1);
                  if (ii == 0) mma_16816_zc(t[0], af, b0, b1);
                  else mma_16816(t[0], af, b0, b1);
                }
              }
              float(&ac)[NT][4] = hb ? acc2 : acc;
#pragma unroll
              for (int j = 0; j < NT; ++j) {
                ac[j][0] = fmaf(s_lo, t[j][0], ac[j][0]);
                ac[j][1] = fmaf(s_lo, t[j][1], ac[j][1]);
                ac[j][2] = fmaf(s_hi, t[j][2], ac[j][2]);
                ac[j][3] = fmaf(s_hi, t[j][3], ac[j][3]);
              }
            }
          }
        };
        if (nq == kSPS) {  // full stage: constant offsets
#pragma unroll
          for (int i4 = 0; i4 < kSPS; ++i4) step(i4);
        } else {
          for (int i4 = 0; i4 < nq; ++i4) step(i4);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8u * slot);
        if (++slot == nst) {
          slot = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[j][c] += acc2[j][c];

      // Epilogue.  Thread owns rows r and r+8 of its tile, tokens n = 2*(lane%4) + {0,1} of each n8 tile.
#pragma unroll
      for (int j = 0; j < NT; ++j) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int n = j * 8 + 2 * (lane & 3) + c;
          const bool live = n < ntok;
          const int s = s0 + n;
          const float f = live ? fac[n] : 0.f;
          const float lo = acc[j][c] * f, hi = acc[j][2 + c] * f;
          float hmax = 0.f;
          if (STAGE == STAGE_GATED) {
            const float h = silu_f32(lo * gl0) * (hi * gl1);
            if (live) a.out[(size_t)s * a.n_rows + tile * 8 + r] = h;
            hmax = fabsf(h);
          } else if (STAGE == STAGE_RELU2) {
            const float v0 = fmaxf(lo * gl0, 0.f), v1 = fmaxf(hi * gl0, 0.f);
            if (live) {
              a.out[(size_t)s * a.n_rows + tile * 16 + r] = v0 * v0;
              a.out[(size_t)s * a.n_rows + tile * 16 + r + 8] = v1 * v1;
            }
            hmax = fmaxf(v0 * v0, v1 * v1);
          } else if (live) {
            const float wt = wts[n];
            store_partial(a, (size_t)s * a.n_rows + tile * 16 + r, wt * lo);
            store_partial(a, (size_t)s * a.n_rows + tile * 16 + r + 8, wt * hi);
          }
          if (STAGE != STAGE_DOWN && a.out_amax != nullptr) {
            // max over the 8 lanes holding this token, then one atomic per warp; a max of
            // non-negative floats is exact and order-free, so the result is deterministic.
            hmax = fmaxf(hmax, __shfl_xor_sync(0xffffffffu, hmax, 4));
            hmax = fmaxf(hmax, __shfl_xor_sync(0xffffffffu, hmax, 8));
            hmax = fmaxf(hmax, __shfl_xor_sync(0xffffffffu, hmax, 16));
            if (live && r == 0) atomicMax(reinterpret_cast<unsigned *>(a.out_amax) + s, __float_as_uint(hmax));
          }
        }
      }
    }
  }
  if (!ok && lane == 0) atomicOr(&a.status[ST_FLAGS], ST_FLAG_TIMEOUT);
}


// Shared-memory bytes of the grouped kernel for reduction length K, NT n8 token
// tiles per pass and nst ring stages.
inline size_t grouped_mma_smem_bytes(int K, int NT, int nst) {
  return (size_t)nst * kStageBytes + (size_t)8 * NT * (2 * K + 16) + 8 * NT * (4 + 8 + 4) + 16 * (size_t)nst + 8 +
         (16 + 4 * kQEntry) * kQueue;
}

}  // namespace bqmoe
