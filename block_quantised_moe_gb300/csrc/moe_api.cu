// C ABI of libmoe: host-side planning, binding and the run sequence.
// The contract (plan -> scratch -> bind -> run; plan may allocate host state,
// bind only records pointers, run only launches) follows the b12x project page,
// section "Using it"; fixed workspace capacity and live counts kept out of the
// plan follow "b12x has moved to FlashInfer", section "Technical layout and
// contracts".
#include <algorithm>
#include <mutex>
#include <new>

#include "common.cuh"
#include "internal.h"
#include "launch.h"
#include "moe.h"
#include "sync.cuh"
#include "unified.cuh"

using namespace bqmoe;

struct moe_weight_plan_s {
  WeightLayout L;
};

struct moe_plan_s {
  WeightLayout L;
  int K = 0, max_tokens = 0, afmt = 0, pad = 16;
  bool tc_on = false;  // experts with >= large_min pairs run on the tcgen05 kernel
  bool fp4_on = false; // ... on the block-scaled FP4 kernel (W4A4 with the weights' FP4 tiles)
  bool mx8_on = false; // ... on the block-scaled FP8 kernel (MXFP4 weights x MXFP8 activations)
  bool tc2_on = false; // ... otherwise on the CTA-pair kernel (token tiles of up to 256)
  bool unified_ok = false;  // decode plan the single-launch forward supports
  bool unified_on = false;  // ... and moe_run uses it (MOE_OPT_SINGLE_LAUNCH)
  bool out_f32 = false;     // FP32 output (MOE_OPT_OUT_F32)
  int large_min = 0x7FFFFFFF;
  ScratchLayout S;
};

struct moe_binding_s {
  moe_plan_s P;
  uint8_t *scratch = nullptr;
  const uint8_t *packed = nullptr;
  const void *x = nullptr;
  const int32_t *ids = nullptr;
  const float *w = nullptr;
  int T = 0;
  void *out = nullptr;
  int32_t launches = 0;  // kernels enqueued by the last forward on this binding
};

namespace bqmoe {
int &launch_counter() {
  thread_local int n = 0;
  return n;
}
}  // namespace bqmoe

namespace {

constexpr int kMaxTopK = 16;
constexpr int kPad = 16;        // expert groups are padded to this many pairs
constexpr int kFp4Tile = 128;   // ... and to this many with the block-scaled FP4 kernel
constexpr int kLargeMin = 32;  // pairs from which an expert runs on the tcgen05 kernel

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

template <typename T>
T *at(uint8_t *base, size_t off) {
  return reinterpret_cast<T *>(base + off);
}

}  // namespace

extern "C" {

const char *moe_status_str(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CAPACITY: return "MOE_ERR_CAPACITY";
    case MOE_ERR_SCRATCH_TOO_SMALL: return "MOE_ERR_SCRATCH_TOO_SMALL";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
  }
  return "MOE_ERR_UNKNOWN";
}

moe_status moe_plan_weights(const moe_weight_desc *d, moe_weight_plan *out, size_t *packed_bytes) {
  if (!d || !out || !packed_bytes) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (d->num_experts < 1 || d->hidden <= 0 || d->intermediate <= 0) return MOE_ERR_INVALID_ARG;
  if (d->wfmt != MOE_W_NVFP4 && d->wfmt != MOE_W_MXFP4) return MOE_ERR_INVALID_ARG;
  if (d->act != MOE_ACT_SILU_GATED && d->act != MOE_ACT_RELU2) return MOE_ERR_INVALID_ARG;
  if (d->flags & ~MOE_WFLAG_FP4_TILES) return MOE_ERR_INVALID_ARG;
  if (d->num_experts > kMaxExperts || d->hidden % 128 || d->intermediate % 64) return MOE_ERR_UNSUPPORTED;
  WeightLayout L;
  L.E = d->num_experts;
  L.H = d->hidden;
  L.I = d->intermediate;
  L.wfmt = d->wfmt;
  L.act = d->act;
  L.bs = d->wfmt == MOE_W_NVFP4 ? 16 : 32;
  L.n13 = d->act == MOE_ACT_SILU_GATED ? 2 * L.I : L.I;
  L.off_c13 = 0;  // codes and scales interleaved per 128-row block and 64-K step
  L.off_c2 = align_up(L.off_c13 + (size_t)L.E * L.blk13_expert());
  L.off_g = align_up(L.off_c2 + (size_t)L.E * L.blk2_expert());
  L.off_t13 = L.off_t2 = align_up(L.off_g + (size_t)L.E * 4 * sizeof(float));
  if (d->flags & MOE_WFLAG_FP4_TILES) {
    if (d->wfmt != MOE_W_NVFP4) return MOE_ERR_UNSUPPORTED;
    L.fp4_tiles = L.n13 % 128 == 0 && L.H % 256 == 0 && L.I % 256 == 0;
    if (!L.fp4_tiles) return MOE_ERR_UNSUPPORTED;
    L.off_t2 = align_up(L.off_t13 + (size_t)L.E * L.t13_expert());
  }
  L.total = L.fp4_tiles ? align_up(L.off_t2 + (size_t)L.E * L.t2_expert()) : L.off_t13;
  moe_weight_plan p = new (std::nothrow) moe_weight_plan_s{L};
  if (!p) return MOE_ERR_CAPACITY;
  *out = p;
  *packed_bytes = L.total;
  return MOE_OK;
}

moe_status moe_prepare_weights(moe_weight_plan wp, const void *w13_codes, const void *w13_scales,
                               const float *w13_global, const void *w2_codes, const void *w2_scales,
                               const float *w2_global, void *packed, cudaStream_t stream) {
  if (!wp || !w13_codes || !w13_scales || !w2_codes || !w2_scales || !packed) return MOE_ERR_INVALID_ARG;
  const WeightLayout &L = wp->L;
  const bool nv = L.wfmt == MOE_W_NVFP4;
  if (nv != (w13_global != nullptr) || nv != (w2_global != nullptr)) return MOE_ERR_INVALID_ARG;
  for (const void *p : {w13_codes, w13_scales, w2_codes, w2_scales, (const void *)packed})
    if (!aligned(p, 16)) return MOE_ERR_INVALID_ARG;
  if (nv && (!aligned(w13_global, 4) || !aligned(w2_global, 4))) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_pack(L, w13_codes, w13_scales, w13_global, w2_codes, w2_scales, w2_global,
                                 static_cast<uint8_t *>(packed), stream));
}

moe_status moe_is_supported(const moe_caps *c) {
  if (!c || !c->wplan) return MOE_ERR_INVALID_ARG;
  if (c->top_k < 1 || c->max_tokens < 1) return MOE_ERR_INVALID_ARG;
  if (c->afmt != MOE_A_BF16 && c->afmt != MOE_A_NVFP4 && c->afmt != MOE_A_MXFP8) return MOE_ERR_INVALID_ARG;
  if (c->top_k > kMaxTopK) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)c->max_tokens * c->top_k > (int64_t)1 << 30) return MOE_ERR_UNSUPPORTED;
  // Supported pairs (vLLM docs "b12x Linear and MoE Backends", "Supported
  // Configurations"): NVFP4 weights with BF16, NVFP4 or MXFP8 activations;
  // MXFP4 weights with BF16 or MXFP8 activations.
  if (c->wplan->L.wfmt == MOE_W_MXFP4 && c->afmt == MOE_A_NVFP4) return MOE_ERR_UNSUPPORTED;
  // The tensor-core kernel works on 128-row blocks of each weight matrix.
  if (c->wplan->L.n13 % 128 != 0) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status moe_plan(const moe_caps *c, moe_plan_t *out, size_t *scratch_bytes, int32_t *m_tile) {
  if (!out || !scratch_bytes) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  moe_status st = moe_is_supported(c);
  if (st != MOE_OK) return st;
  moe_plan_s P;
  P.L = c->wplan->L;
  P.K = c->top_k;
  P.max_tokens = c->max_tokens;
  P.afmt = c->afmt;
  P.pad = kPad;
  const WeightLayout &L = P.L;
  const int64_t Pmax = (int64_t)c->max_tokens * c->top_k;
  const int64_t T = c->max_tokens;
  ScratchLayout &S = P.S;
  // Plans for batches of 1024+ (token, slot) pairs send experts with at least
  // kLargeMin pairs to the tcgen05 kernels (dense tiles of 128 tokens): FP16
  // operands with row factors for NVFP4, BF16 operands for MXFP4 (E2M1 * 2^X and
  // E4M3 * 2^X are exact in BF16, not in FP16), and, for W4A4 with the weights'
  // FP4 tiles, both operands as E2M1 codes on the block-scaled FP4 MMA; MXFP4
  // weights with MXFP8 activations run on the block-scaled FP8 MMA (weights
  // widened to E4M3, both operands' E8M0 scales as they are).  The block-scaled
  // kernels read their activation rows as slot-major 128-row tiles, so their
  // plans pad every expert's group to 128 slots.
  P.tc_on = Pmax >= 1024 && tc2_supported(L.n13, L.H) && tc2_supported(L.H, L.I);
  P.fp4_on = P.tc_on && P.afmt == MOE_A_NVFP4 && L.fp4_tiles && fp4_tc_supported(L.n13, L.H) &&
             fp4_tc_supported(L.H, L.I);
  P.mx8_on = P.tc_on && L.wfmt == MOE_W_MXFP4 && P.afmt == MOE_A_MXFP8 && mx8_tc_supported(L.n13, L.H) &&
             mx8_tc_supported(L.H, L.I);
  if (P.fp4_on || P.mx8_on) P.pad = kFp4Tile;
  P.tc2_on = P.tc_on && !P.fp4_on && !P.mx8_on;
  P.unified_ok = !P.tc_on && unified_supported(L.wfmt, P.afmt, (int)Pmax, L.E, P.K);
  P.unified_on = false;  // opt-in: measured slower than the PDL-overlapped launches (see moe.h)
  S.cap_sorted = round_up(Pmax + (int64_t)L.E * (P.pad - 1), P.pad);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  S.status = take(16);
  S.counts = take(4 * (size_t)L.E);
  S.offsets = take(4 * (size_t)(L.E + 1));
  S.sorted = take(4 * (size_t)S.cap_sorted);
  S.pair_pos = take(4 * (size_t)Pmax);
  S.active = take(4 * (size_t)(L.E + 1));
  S.passes = take(4 * (size_t)(L.E + 1));
  S.large = take(4 * (size_t)(L.E + 1));
  S.large_tiles = take(4 * (size_t)(L.E + 1));
  // tiles of at least 128 tokens: at most one more per large expert than P / 128
  S.tiles = take(16 * ((size_t)Pmax / 128 + (size_t)L.E + 1));
  S.route_hist = take(4 * (size_t)route_chunks((int)Pmax) * (L.E + 1));
  S.work = take(4 * 2 * (size_t)kWorkSlots);
  S.gbar = take(16);
  if (P.afmt == MOE_A_NVFP4) {
    S.xq_codes = take((size_t)T * L.H / 2);
    S.xq_scales = take((size_t)T * L.H / 16);
    S.xq_g = take(4 * (size_t)T);
  } else if (P.afmt == MOE_A_MXFP8) {
    S.xq_codes = take((size_t)T * L.H);
    S.xq_scales = take((size_t)T * L.H / 32);
  }
  S.h = take(4 * (size_t)S.cap_sorted * L.I);
  if (P.afmt == MOE_A_NVFP4) {
    S.hq_codes = take((size_t)S.cap_sorted * L.I / 2);
    S.hq_scales = take((size_t)S.cap_sorted * L.I / 16);
    S.hq_g = take(4 * (size_t)S.cap_sorted);
  } else if (P.afmt == MOE_A_MXFP8) {
    S.hq_codes = take((size_t)S.cap_sorted * L.I);
    S.hq_scales = take((size_t)S.cap_sorted * L.I / 32);
  }
  S.x16 = take(2 * (size_t)T * L.H);
  S.xfac = take(4 * (size_t)T);
  S.hamax = take(4 * (size_t)S.cap_sorted);
  if (P.tc_on) {
    P.large_min = kLargeMin;
    if (P.fp4_on) {
      // activation tiles: per 128 slots and 256-K block, 16 KB of codes + 2 KB of scales
      S.xt = take((size_t)(S.cap_sorted / kFp4Tile) * (L.H / 256) * WeightLayout::kFp4TileBytes);
      S.ht = take((size_t)(S.cap_sorted / kFp4Tile) * (L.I / 256) * WeightLayout::kFp4TileBytes);
    } else if (P.mx8_on) {
      // activation tiles: per 128 slots and 128-K block, 16 KB of codes + 512 bytes of scales
      S.xt = take((size_t)(S.cap_sorted / kFp4Tile) * (L.H / 128) * kMx8TileBytes);
      S.ht = take((size_t)(S.cap_sorted / kFp4Tile) * (L.I / 128) * kMx8TileBytes);
    } else {
      if (L.wfmt == MOE_W_MXFP4) S.xb16 = take(2 * (size_t)T * L.H);
      if (P.tc2_on) S.xs16 = take(2 * (size_t)S.cap_sorted * L.H);
      S.h16 = take(2 * (size_t)S.cap_sorted * L.I);
      if (L.wfmt == MOE_W_NVFP4) S.h16fac = take(4 * (size_t)S.cap_sorted);
    }
  }
  // GEMM2 partials: BF16 when the tcgen05 kernels run (many tokens: the partials'
  // write + read dominate the non-GEMM traffic), FP32 otherwise.
  S.part = take((P.tc_on ? 2 : 4) * (size_t)S.cap_sorted * L.H);
  S.total = o;
  moe_plan_t p = new (std::nothrow) moe_plan_s(P);
  if (!p) return MOE_ERR_CAPACITY;
  *out = p;
  *scratch_bytes = S.total;
  if (m_tile) *m_tile = P.pad;
  return MOE_OK;
}

moe_status moe_plan_set_option(moe_plan_t plan, int32_t option, int32_t value) {
  if (!plan) return MOE_ERR_INVALID_ARG;
  if (option == MOE_OPT_SINGLE_LAUNCH) {
    if (value != 0 && value != 1) return MOE_ERR_INVALID_ARG;
    if (value == 1 && (!plan->unified_ok || plan->out_f32)) return MOE_ERR_UNSUPPORTED;
    plan->unified_on = value == 1;
    return MOE_OK;
  }
  if (option == MOE_OPT_OUT_F32) {
    if (value != 0 && value != 1) return MOE_ERR_INVALID_ARG;
    if (value == 1 && plan->unified_on) return MOE_ERR_UNSUPPORTED;
    plan->out_f32 = value == 1;
    return MOE_OK;
  }
  return MOE_ERR_INVALID_ARG;
}

moe_status moe_bind(moe_plan_t plan, void *scratch, size_t scratch_bytes, const void *packed, const void *x,
                    const int32_t *topk_ids, const float *topk_weights, int32_t num_tokens, void *out,
                    moe_binding *out_binding) {
  if (!out_binding) return MOE_ERR_INVALID_ARG;
  *out_binding = nullptr;
  if (!plan || num_tokens < 0) return MOE_ERR_INVALID_ARG;
  if (num_tokens > plan->max_tokens) return MOE_ERR_CAPACITY;
  if (!scratch || !aligned(scratch, 256)) return MOE_ERR_INVALID_ARG;
  if (scratch_bytes < plan->S.total) return MOE_ERR_SCRATCH_TOO_SMALL;
  if (num_tokens > 0) {
    if (!packed || !x || !topk_ids || !topk_weights || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned(packed, 256) || !aligned(x, 16) || !aligned(out, 16) || !aligned(topk_ids, 4) ||
        !aligned(topk_weights, 4))
      return MOE_ERR_INVALID_ARG;
  }
  moe_binding b = new (std::nothrow) moe_binding_s;
  if (!b) return MOE_ERR_CAPACITY;
  b->P = *plan;
  b->scratch = static_cast<uint8_t *>(scratch);
  b->packed = static_cast<const uint8_t *>(packed);
  b->x = x;
  b->ids = topk_ids;
  b->w = topk_weights;
  b->T = num_tokens;
  b->out = out;
  *out_binding = b;
  return MOE_OK;
}

static moe_status run_forward(moe_binding b, cudaStream_t stream, cudaEvent_t *ev);

// The single-launch decode forward (unified.cuh) on the binding's buffers;
// `withhold` >= 0 is the failure-detection self-test (CTA 0 withholds its
// arrival at that grid barrier).
static moe_status run_unified(moe_binding b, cudaStream_t stream, int withhold) {
  const moe_plan_s &P = b->P;
  const WeightLayout &L = P.L;
  const ScratchLayout &S = P.S;
  uint8_t *sc = b->scratch;
  const int T = b->T, K = P.K, E = L.E, H = L.H, I = L.I;
  const bool wide = (int64_t)P.max_tokens * K > (int64_t)8 * E;
  const int ntok = mma_tokens_per_pass(H, I, wide);
  UnifiedArgs u{};
  u.x = static_cast<const __nv_bfloat16 *>(b->x);
  u.ids = b->ids;
  u.T = T;
  u.K = K;
  u.E = E;
  u.H = H;
  u.I = I;
  u.pad = P.pad;
  u.ntok = ntok;
  u.ro = RouteOut{at<int32_t>(sc, S.counts), at<int32_t>(sc, S.offsets), at<int32_t>(sc, S.sorted),
                  at<int32_t>(sc, S.pair_pos), at<int32_t>(sc, S.active), at<int32_t>(sc, S.passes),
                  at<int32_t>(sc, S.large), at<int32_t>(sc, S.large_tiles), at<int32_t>(sc, S.status), nullptr, 0,
                  at<int32_t>(sc, S.work), 2 * kWorkSlots};
  u.x16 = at<__half>(sc, S.x16);
  u.xfac = at<float>(sc, S.xfac);
  u.hamax = at<float>(sc, S.hamax);
  u.cap_sorted = S.cap_sorted;
  const bool a16 = P.afmt == MOE_A_BF16;
  if (!a16) {
    u.xq_codes = at<uint8_t>(sc, S.xq_codes);
    u.xq_scales = at<uint8_t>(sc, S.xq_scales);
    u.xq_g = P.afmt == MOE_A_NVFP4 ? at<float>(sc, S.xq_g) : nullptr;
    u.hq_codes = at<uint8_t>(sc, S.hq_codes);
    u.hq_scales = at<uint8_t>(sc, S.hq_scales);
    u.hq_g = P.afmt == MOE_A_NVFP4 ? at<float>(sc, S.hq_g) : nullptr;
  }
  GroupedArgs a{};
  a.counts = u.ro.counts;
  a.offsets = u.ro.offsets;
  a.sorted_pair = u.ro.sorted_pair;
  a.active = u.ro.active;
  a.passes = u.ro.passes;
  a.large = u.ro.large;
  a.large_tiles = u.ro.large_tiles;
  a.status = u.ro.status;
  a.top_k = K;
  a.topk_weights = b->w;
  a.globals = reinterpret_cast<const float *>(b->packed + L.off_g);
  a.I = I;
  a.tiny = (int64_t)P.max_tokens * K * 8 <= E;
  GroupedArgs g1 = a;  // GEMM1: staged x rows -> h (+ the per-pair |h| maxima for BF16 activations)
  g1.codes = b->packed + L.off_c13;
  g1.codes_expert = L.blk13_expert();
  g1.K = H;
  g1.n_rows = I;
  g1.n_blocks = L.n13 / 128;
  g1.act = u.x16;
  g1.act_g = u.xfac;
  g1.out_amax = a16 ? u.hamax : nullptr;
  g1.out = at<float>(sc, S.h);
  g1.work = u.ro.work;
  GroupedArgs g2 = a;  // GEMM2: h (or its re-quantised codes) -> FP32 partials x topk weight
  g2.codes = b->packed + L.off_c2;
  g2.codes_expert = L.blk2_expert();
  g2.K = I;
  g2.n_rows = H;
  g2.n_blocks = H / 128;
  g2.act = a16 ? static_cast<const void *>(g1.out) : static_cast<const void *>(u.hq_codes);
  g2.act_scales = a16 ? nullptr : u.hq_scales;
  g2.act_g = a16 ? u.hamax : u.hq_g;
  g2.out = at<float>(sc, S.part);
  g2.out_bf16 = 0;
  g2.work = u.ro.work + kWorkSlots;
  u.g1 = g1;
  u.g2 = g2;
  u.part = g2.out;
  u.out = static_cast<__nv_bfloat16 *>(b->out);
  u.gbar = at<int32_t>(sc, S.gbar);
  u.withhold = withhold;
  const int stage1 = L.act == MOE_ACT_SILU_GATED ? STAGE_GATED : STAGE_RELU2;
  return cuda_status(launch_unified(L.wfmt, P.afmt, stage1, ntok, a.tiny, u, stream));
}

static moe_status run_impl(moe_binding b, cudaStream_t stream, cudaEvent_t *ev) {
  launch_counter() = 0;
  const moe_status st = run_forward(b, stream, ev);
  b->launches = launch_counter();
  return st;
}

static moe_status run_forward(moe_binding b, cudaStream_t stream, cudaEvent_t *ev) {
  // Inside stream capture the stage events become event-record nodes of the
  // graph, so a replayed graph still times its stages.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (ev && cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return MOE_ERR_CUDA;
  const unsigned ev_flags = cap == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
  auto mark = [&](int i) { return ev ? cudaEventRecordWithFlags(ev[i], stream, ev_flags) : cudaSuccess; };
  if (b->T == 0) {
    for (int i = 0; ev && i <= MOE_NUM_STAGES; ++i)
      if (mark(i) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  const moe_plan_s &P = b->P;
  const WeightLayout &L = P.L;
  const ScratchLayout &S = P.S;
  uint8_t *sc = b->scratch;
  const int T = b->T, K = P.K, E = L.E, H = L.H, I = L.I;
  int32_t *status = at<int32_t>(sc, S.status);
  int32_t *counts = at<int32_t>(sc, S.counts);
  int32_t *offsets = at<int32_t>(sc, S.offsets);
  int32_t *sorted = at<int32_t>(sc, S.sorted);
  int32_t *pair_pos = at<int32_t>(sc, S.pair_pos);
  float *h = at<float>(sc, S.h);
  float *part = at<float>(sc, S.part);
  cudaError_t err;
  if (P.unified_on && ev == nullptr) return run_unified(b, stream, -1);

  if ((err = mark(MOE_STAGE_ROUTE)) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t *active = at<int32_t>(sc, S.active);
  int32_t *passes = at<int32_t>(sc, S.passes);
  // one n8 token tile per pass when the plan expects at most 8 pairs per expert
  const bool wide = (int64_t)P.max_tokens * K > (int64_t)8 * E;
  const int ntok = mma_tokens_per_pass(H, I, wide);
  int32_t *large = at<int32_t>(sc, S.large);
  int32_t *large_tiles = at<int32_t>(sc, S.large_tiles);
  // With BF16 activations on the tensor-core path, extra CTAs of the routing
  // launch stage x as FP16 rows and clear the per-pair |h| maxima.
  RouteStaging stg{static_cast<const __nv_bfloat16 *>(b->x), T, H, at<__half>(sc, S.x16), at<float>(sc, S.xfac),
                   at<float>(sc, S.hamax), S.cap_sorted};
  const bool staged = P.afmt == MOE_A_BF16;
  if ((err = launch_route(b->ids, T * K, E, P.pad, ntok, P.large_min, P.tc2_on ? 256 : 128, counts, offsets, sorted,
                          pair_pos, active,
                          passes, large, large_tiles, at<int4>(sc, S.tiles), P.tc2_on ? 1 : 0, status,
                          at<int32_t>(sc, S.route_hist),
                          at<int32_t>(sc, S.work),
                          2 * kWorkSlots, staged ? &stg : nullptr,
                          stream)) != cudaSuccess)
    return MOE_ERR_CUDA;

  GroupedArgs a{};
  a.counts = counts;
  a.offsets = offsets;
  a.sorted_pair = sorted;
  a.active = active;
  a.passes = passes;
  a.large = large;
  a.large_tiles = large_tiles;
  a.tiles = at<int4>(sc, S.tiles);
  a.status = status;
  a.top_k = K;
  a.topk_weights = b->w;
  a.globals = reinterpret_cast<const float *>(b->packed + L.off_g);
  a.I = I;

  // activation quantiser (x) for NVFP4 / MXFP8 activations
  if ((err = mark(MOE_STAGE_QUANT_X)) != cudaSuccess) return MOE_ERR_CUDA;
  int src1 = SRC_X_BF16;
  a.act = b->x;
  if (P.afmt == MOE_A_NVFP4) {
    err = launch_quant_rows_nvfp4(b->x, true, T, H, at<uint8_t>(sc, S.xq_codes), at<uint8_t>(sc, S.xq_scales),
                                  at<float>(sc, S.xq_g), nullptr, nullptr, stream,
                                  P.fp4_on ? at<uint8_t>(sc, S.xt) : nullptr, pair_pos, K);
    src1 = SRC_X_NVFP4;
    a.act = at<uint8_t>(sc, S.xq_codes);
    a.act_scales = at<uint8_t>(sc, S.xq_scales);
    a.act_g = at<float>(sc, S.xq_g);
  } else if (P.afmt == MOE_A_MXFP8) {
    err = launch_quant_blocks(Q_MXFP8, b->x, true, T, H, 1, nullptr, at<uint8_t>(sc, S.xq_codes),
                              at<uint8_t>(sc, S.xq_scales), nullptr, nullptr, stream,
                              P.mx8_on ? at<uint8_t>(sc, S.xt) : nullptr, pair_pos, K);
    src1 = SRC_X_MXFP8;
    a.act = at<uint8_t>(sc, S.xq_codes);
    a.act_scales = at<uint8_t>(sc, S.xq_scales);
  }
  if (err != cudaSuccess) return MOE_ERR_CUDA;
  const bool nv = L.wfmt == MOE_W_NVFP4;
  // Staged B operand of the register-dequant kernel: x^ as FP16 slot-order rows
  // + per-row factor (done by the routing launch for BF16 x); also clears the
  // per-pair |h| maxima.
  if (!staged) {
    err = launch_stage_x16(src1, a.act, a.act_scales, a.act_g, T, H, at<__half>(sc, S.x16), at<float>(sc, S.xfac),
                           at<float>(sc, S.hamax), S.cap_sorted, stream);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
  }
  const void *x_src = a.act;  // BF16 x or x^ codes, for the MXFP4 tcgen05 staging
  const uint8_t *x_src_scales = a.act_scales;
  a.act = at<__half>(sc, S.x16);
  a.act_scales = nullptr;
  a.act_g = at<float>(sc, S.xfac);
  a.out_amax = P.afmt == MOE_A_BF16 ? at<float>(sc, S.hamax) : nullptr;

  // GEMM1 + activation -> h (its activation staging for the tensor-core kernels
  // is timed with the activation quantiser's stage)
  a.codes = b->packed + L.off_c13;
  a.codes_expert = L.blk13_expert();
  a.K = H;
  a.n_rows = I;
  a.out = h;
  const int stage1 = L.act == MOE_ACT_SILU_GATED ? STAGE_GATED : STAGE_RELU2;
  if (!nv && P.tc2_on) {  // MXFP4 tcgen05 operands: x or x^ as BF16 slot-order rows, factor 1
    err = launch_stage_h16(P.afmt == MOE_A_MXFP8 ? SRC_H_MXFP8 : SRC_X_BF16, x_src, x_src_scales, nullptr, H, T,
                           nullptr, at<__half>(sc, S.xb16), nullptr, true, false, stream);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (P.tc2_on) {  // the pair kernel reads GEMM1's activation rows in slot order, one tensor copy per stage
    err = launch_gather_slot_rows(nv ? static_cast<const void *>(at<__half>(sc, S.x16))
                                     : static_cast<const void *>(at<__half>(sc, S.xb16)),
                                  sorted, offsets + E, K, H, S.cap_sorted, at<__half>(sc, S.xs16), stream);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (mark(MOE_STAGE_GEMM1) != cudaSuccess) return MOE_ERR_CUDA;
  a.work = at<int32_t>(sc, S.work);
  a.tiny = (int64_t)P.max_tokens * K * 8 <= E;
  a.wait_first = staged ? 1 : 0;  // routing (which staged x) triggered GEMM1 early
  err = launch_grouped_mma(L.wfmt, SRC_X16, stage1, a, L.n13, E, ntok, stream);
  if (err == cudaSuccess && P.tc_on) {
    GroupedArgs t = a;
    t.act_by_token = 1;
    if (P.mx8_on) {
      t.act = at<uint8_t>(sc, S.xt);  // x^ as slot-major MX FP8 tiles
      t.act_scales = nullptr;
      t.act_g = nullptr;
      t.out_amax = nullptr;
      err = launch_grouped_mx8(stage1, t, L.n13, stream);
    } else if (P.fp4_on) {
      t.codes = b->packed + L.off_t13;
      t.codes_expert = L.t13_expert();
      t.act = at<uint8_t>(sc, S.xt);  // x^ as slot-major FP4 tiles; per-token globals
      t.act_scales = nullptr;
      t.act_g = at<float>(sc, S.xq_g);
      t.out_amax = nullptr;
      err = launch_grouped_fp4(stage1, t, L.n13, stream);
    } else {
      if (!nv) {
        t.act = at<__half>(sc, S.xb16);
        t.act_g = nullptr;
      }
      t.act = at<__half>(sc, S.xs16);
      err = launch_grouped_tc2(stage1, L.wfmt, t, L.n13, S.cap_sorted, stream);
    }
  }
  a.out_amax = nullptr;
  a.wait_first = 0;
  if (err != cudaSuccess) return MOE_ERR_CUDA;

  // re-quantise h for NVFP4 / MXFP8 activations (rows past offsets[E] are skipped)
  if ((err = mark(MOE_STAGE_QUANT_H)) != cudaSuccess) return MOE_ERR_CUDA;
  int src2 = SRC_H_F32;
  a.act = h;
  a.act_scales = nullptr;
  a.act_g = at<float>(sc, S.hamax);
  if (P.afmt == MOE_A_NVFP4) {
    err = launch_quant_rows_nvfp4(h, false, S.cap_sorted, I, at<uint8_t>(sc, S.hq_codes),
                                  at<uint8_t>(sc, S.hq_scales), at<float>(sc, S.hq_g), offsets + E, sorted, stream,
                                  P.fp4_on ? at<uint8_t>(sc, S.ht) : nullptr, nullptr, 0);
    src2 = SRC_H_NVFP4;
    a.act = at<uint8_t>(sc, S.hq_codes);
    a.act_scales = at<uint8_t>(sc, S.hq_scales);
    a.act_g = at<float>(sc, S.hq_g);
  } else if (P.afmt == MOE_A_MXFP8) {
    err = launch_quant_blocks(Q_MXFP8, h, false, S.cap_sorted, I, 1, nullptr, at<uint8_t>(sc, S.hq_codes),
                              at<uint8_t>(sc, S.hq_scales), offsets + E, sorted, stream,
                              P.mx8_on ? at<uint8_t>(sc, S.ht) : nullptr, nullptr, 0);
    src2 = SRC_H_MXFP8;
    a.act = at<uint8_t>(sc, S.hq_codes);
    a.act_scales = at<uint8_t>(sc, S.hq_scales);
    a.act_g = nullptr;
  }
  if (err != cudaSuccess) return MOE_ERR_CUDA;

  // GEMM2 * topk_weight -> partials, then the ordered combine
  if (P.tc2_on) {  // 16-bit slot-order rows of h (or of its re-quantised codes) for the CTA-pair GEMM2
    err = launch_stage_h16(src2, a.act, a.act_scales, a.act_g, I, S.cap_sorted, offsets + E, at<__half>(sc, S.h16),
                           nv ? at<float>(sc, S.h16fac) : nullptr, !nv, true, stream);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
  }
  a.codes = b->packed + L.off_c2;
  a.codes_expert = L.blk2_expert();
  a.K = I;
  a.n_rows = H;
  a.out = part;
  a.out_bf16 = P.tc_on ? 1 : 0;
  if (mark(MOE_STAGE_GEMM2) != cudaSuccess) return MOE_ERR_CUDA;
  a.work = at<int32_t>(sc, S.work) + kWorkSlots;
  err = launch_grouped_mma(L.wfmt, src2, STAGE_DOWN, a, H, E, ntok, stream);
  if (err == cudaSuccess && P.tc_on && P.mx8_on) {
    GroupedArgs t = a;  // h^ as slot-major MX FP8 tiles
    t.act = at<uint8_t>(sc, S.ht);
    t.act_scales = nullptr;
    t.act_g = nullptr;
    t.act_by_token = 0;
    err = launch_grouped_mx8(STAGE_DOWN, t, H, stream);
  } else if (err == cudaSuccess && P.tc_on && P.fp4_on) {
    GroupedArgs t = a;  // h^ as slot-major FP4 tiles; per-slot globals
    t.codes = b->packed + L.off_t2;
    t.codes_expert = L.t2_expert();
    t.act = at<uint8_t>(sc, S.ht);
    t.act_scales = nullptr;
    t.act_by_token = 0;
    err = launch_grouped_fp4(STAGE_DOWN, t, H, stream);
  } else if (err == cudaSuccess && P.tc_on) {
    GroupedArgs t = a;
    t.act = at<__half>(sc, S.h16);
    t.act_scales = nullptr;
    t.act_g = nv ? at<float>(sc, S.h16fac) : nullptr;
    t.act_by_token = 0;
    err = launch_grouped_tc2(STAGE_DOWN, L.wfmt, t, H, S.cap_sorted, stream);
  }
  if (err != cudaSuccess) return MOE_ERR_CUDA;
  if (mark(MOE_STAGE_COMBINE) != cudaSuccess) return MOE_ERR_CUDA;
  if ((err = launch_combine(part, P.tc_on, H, pair_pos, T, K, b->out, P.out_f32, stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (mark(MOE_NUM_STAGES) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_run(moe_binding b, cudaStream_t stream) {
  if (!b) return MOE_ERR_INVALID_ARG;
  return run_impl(b, stream, nullptr);
}

moe_status moe_run_timed(moe_binding b, cudaStream_t stream, cudaEvent_t *events) {
  if (!b || !events) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i <= MOE_NUM_STAGES; ++i)
    if (!events[i]) return MOE_ERR_INVALID_ARG;
  return run_impl(b, stream, events);
}

moe_status moe_launch_count(moe_binding b, int32_t *n) {
  if (!b || !n) return MOE_ERR_INVALID_ARG;
  *n = b->launches;
  return MOE_OK;
}

moe_status moe_run_host(moe_binding b, const void *x_host, const int32_t *ids_host, const float *weights_host,
                        void *out_host, cudaStream_t stream) {
  if (!b) return MOE_ERR_INVALID_ARG;
  if (b->T == 0) return MOE_OK;
  if (!x_host || !ids_host || !weights_host || !out_host) return MOE_ERR_INVALID_ARG;
  const size_t T = b->T, H = b->P.L.H, K = b->P.K;
  if (cudaMemcpyAsync(const_cast<void *>(b->x), x_host, T * H * 2, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
      cudaMemcpyAsync(const_cast<int32_t *>(b->ids), ids_host, T * K * 4, cudaMemcpyHostToDevice, stream) !=
          cudaSuccess ||
      cudaMemcpyAsync(const_cast<float *>(b->w), weights_host, T * K * 4, cudaMemcpyHostToDevice, stream) !=
          cudaSuccess)
    return MOE_ERR_CUDA;
  moe_status st = moe_run(b, stream);
  if (st != MOE_OK) return st;
  if (cudaMemcpyAsync(out_host, b->out, T * H * (b->P.out_f32 ? 4 : 2), cudaMemcpyDeviceToHost, stream) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return cuda_status(cudaStreamSynchronize(stream));
}

moe_status moe_device_status(moe_binding b, cudaStream_t stream, int32_t *status) {
  if (!b || !status) return MOE_ERR_INVALID_ARG;
  int32_t st[4] = {0, 0, 0, 0};
  if (b->T > 0) {
    if (cudaMemcpyAsync(st, b->scratch + b->P.S.status, 16, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  }
  for (int i = 0; i < 4; ++i) status[i] = st[i];
  return (st[ST_FLAGS] & ST_FLAG_TIMEOUT) ? MOE_ERR_TIMEOUT : MOE_OK;
}

moe_status moe_debug_hidden(moe_binding b, cudaStream_t stream, float *h, int32_t rows_cap, int32_t *rows) {
  if (!b || !h || !rows || rows_cap < 0) return MOE_ERR_INVALID_ARG;
  *rows = 0;
  if (b->T == 0) return MOE_OK;
  const ScratchLayout &S = b->P.S;
  int32_t n = 0;
  if (cudaMemcpyAsync(&n, b->scratch + S.offsets + sizeof(int32_t) * b->P.L.E, sizeof n, cudaMemcpyDeviceToHost,
                      stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (n > rows_cap) return MOE_ERR_CAPACITY;
  if (cudaMemcpyAsync(h, b->scratch + S.h, sizeof(float) * (size_t)n * b->P.L.I, cudaMemcpyDeviceToHost, stream) !=
          cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  *rows = n;
  return MOE_OK;
}

namespace bqmoe {
// One thread waits, bounded, on an mbarrier that nothing arrives on, and
// records the timeout the way every kernel of the forward does.
__global__ void k_wait_timeout_probe(int32_t *status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = (uint32_t)__cvta_generic_to_shared(&bar);
  mbar_init(b, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  if (!mbar_wait(b, 0)) atomicOr(&status[ST_FLAGS], ST_FLAG_TIMEOUT);
}
}  // namespace bqmoe

moe_status moe_selftest_wait_timeout(cudaStream_t stream, int32_t *status_dev, int32_t *status) {
  if (!status_dev || !status) return MOE_ERR_INVALID_ARG;
  if (cudaMemsetAsync(status_dev, 0, 4 * sizeof(int32_t), stream) != cudaSuccess) return MOE_ERR_CUDA;
  bqmoe::k_wait_timeout_probe<<<1, 32, 0, stream>>>(status_dev);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  int32_t st[4] = {0, 0, 0, 0};
  if (cudaMemcpyAsync(st, status_dev, sizeof st, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  for (int i = 0; i < 4; ++i) status[i] = st[i];
  return (st[ST_FLAGS] & ST_FLAG_TIMEOUT) ? MOE_ERR_TIMEOUT : MOE_OK;
}

moe_status moe_selftest_grid_barrier_timeout(moe_binding b, cudaStream_t stream, int32_t *status) {
  if (!b || !status) return MOE_ERR_INVALID_ARG;
  if (!b->P.unified_on || b->T == 0) return MOE_ERR_UNSUPPORTED;
  launch_counter() = 0;
  const moe_status st = run_unified(b, stream, 1);  // barrier 1: after GEMM1
  b->launches = launch_counter();
  if (st != MOE_OK) return st;
  return moe_device_status(b, stream, status);
}

moe_status moe_debug_routing(moe_binding b, cudaStream_t stream, int32_t *counts, int32_t *offsets,
                             int32_t *pair_pos, int32_t *sorted_pair, int32_t sorted_cap) {
  if (!b || !counts || !offsets || !pair_pos || !sorted_pair || sorted_cap < 0) return MOE_ERR_INVALID_ARG;
  const int E = b->P.L.E;
  const size_t P = (size_t)b->T * b->P.K;
  uint8_t *sc = b->scratch;
  const ScratchLayout &S = b->P.S;
  if (b->T == 0) return MOE_OK;
  if (cudaMemcpyAsync(counts, sc + S.counts, 4 * (size_t)E, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaMemcpyAsync(offsets, sc + S.offsets, 4 * (size_t)(E + 1), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaMemcpyAsync(pair_pos, sc + S.pair_pos, 4 * P, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  const int32_t n = offsets[E];
  if (n < 0 || n > S.cap_sorted) return MOE_ERR_CUDA;
  if (sorted_cap < n) return MOE_ERR_CAPACITY;
  if (n > 0 && (cudaMemcpyAsync(sorted_pair, sc + S.sorted, 4 * (size_t)n, cudaMemcpyDeviceToHost, stream) !=
                    cudaSuccess ||
                cudaStreamSynchronize(stream) != cudaSuccess))
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_quantize(int32_t qfmt, int32_t gmode, int32_t src_bf16, const void *src, int64_t batch, int64_t rows,
                        int64_t cols, void *codes, void *scales, float *global, cudaStream_t stream) {
  if (qfmt != MOE_Q_NVFP4 && qfmt != MOE_Q_MXFP4 && qfmt != MOE_Q_MXFP8) return MOE_ERR_INVALID_ARG;
  if (batch < 0 || rows < 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
  if (batch == 0 || rows == 0) return MOE_OK;
  if (!src || !codes || !scales) return MOE_ERR_INVALID_ARG;
  if (!aligned(src, 16) || !aligned(codes, 16) || !aligned(scales, 4)) return MOE_ERR_INVALID_ARG;
  const bool bf = src_bf16 != 0;
  cudaError_t err;
  if (qfmt == MOE_Q_NVFP4) {
    if (cols % 16 || !global || !aligned(global, 4)) return MOE_ERR_INVALID_ARG;
    if (gmode == MOE_G_PER_ROW) {
      err = launch_quant_rows_nvfp4(src, bf, batch * rows, cols, static_cast<uint8_t *>(codes),
                                    static_cast<uint8_t *>(scales), global, nullptr, nullptr, stream);
    } else if (gmode == MOE_G_PER_TENSOR) {
      err = launch_amax_tensor(src, bf, batch, rows * cols, global, stream);
      if (err == cudaSuccess) err = launch_amax_to_global(global, batch, stream);
      if (err == cudaSuccess)
        err = launch_quant_blocks(Q_NVFP4, src, bf, batch * rows, cols, rows, global, static_cast<uint8_t *>(codes),
                                  static_cast<uint8_t *>(scales), nullptr, nullptr, stream);
    } else {
      return MOE_ERR_INVALID_ARG;
    }
  } else {
    if (cols % 32 || gmode != MOE_G_NONE || global) return MOE_ERR_INVALID_ARG;
    err = launch_quant_blocks(qfmt == MOE_Q_MXFP4 ? Q_MXFP4 : Q_MXFP8, src, bf, batch * rows, cols, 1, nullptr,
                              static_cast<uint8_t *>(codes), static_cast<uint8_t *>(scales), nullptr, nullptr,
                              stream);
  }
  return cuda_status(err);
}

void moe_destroy_weight_plan(moe_weight_plan p) { delete p; }
void moe_destroy_plan(moe_plan_t p) { delete p; }
void moe_destroy_binding(moe_binding b) { delete b; }

}  // extern "C"

// ------------------------------------------------------------------------
// Forward pass for callers that cannot allocate device memory.
//
// Some callers are handed only their input and output buffers: plugin and
// custom-op interfaces that pass no workspace, and applications whose memory
// pool owns the whole device, where an extra cudaMalloc would fail or fragment
// the pool.  moe_run_no_alloc runs the same kernels as moe_run but takes its
// scratch from the file-scope array below instead of a caller buffer.  The
// array is kNoAllocScratchBytes (MOE_NO_ALLOC_SCRATCH_BYTES, 32 MiB) on every
// device that loads this library and stays allocated until the process exits.
// Every call shares it and it keeps the contents of the last call; everything
// the kernels read before writing (the device status word) is cleared at the
// start of each call.  Calls that overlap on the GPU (on different streams, or
// from different host threads) race on the array.
namespace {

constexpr size_t kNoAllocScratchBytes = MOE_NO_ALLOC_SCRATCH_BYTES;
__device__ __align__(256) uint8_t g_no_alloc_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_no_alloc_mu;
struct NoAllocSlot {
  void *addr = nullptr;         // device address of the array in context `ctx`
  unsigned long long ctx = 0;   // unique id of that context (0: unknown)
};
NoAllocSlot g_no_alloc[kNoAllocMaxDevices];

// Unique id of the current CUDA context, through the driver entry points (the
// library does not link the driver API); 0 if it cannot be had.  A device
// reset or a torn-down primary context gives the next context a new id, so a
// stale device address is never reused.
unsigned long long current_ctx_id() {
  using GetCurrent = int (*)(void **);
  using GetId = int (*)(void *, unsigned long long *);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(f);
  });
  void *ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != 0 || ctx == nullptr || get_id(ctx, &id) != 0) return 0;
  return id;
}

// Device address of the array in the current device's context.  The first
// call in a context looks it up with cudaGetSymbolAddress (with that device
// current); the host-side symbol itself is only a stand-in and must never
// reach a kernel.
moe_status no_alloc_scratch(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_no_alloc_mu);
  NoAllocSlot &slot = g_no_alloc[dev];
  const unsigned long long ctx = current_ctx_id();
  if (slot.addr == nullptr || ctx == 0 || ctx != slot.ctx) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_no_alloc_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    slot.addr = p;
    slot.ctx = current_ctx_id();  // the lookup may have created the context
  }
  *out = slot.addr;
  return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_run_no_alloc(moe_plan_t plan, const void *packed, const void *x, const int32_t *topk_ids,
                                       const float *topk_weights, int32_t num_tokens, void *out,
                                       cudaStream_t stream) {
  if (!plan || num_tokens < 0) return MOE_ERR_INVALID_ARG;
  if (num_tokens > plan->max_tokens) return MOE_ERR_CAPACITY;
  if (plan->S.total > kNoAllocScratchBytes) return MOE_ERR_CAPACITY;  // plan needs more than the static array
  if (num_tokens > 0) {
    if (!packed || !x || !topk_ids || !topk_weights || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned(packed, 256) || !aligned(x, 16) || !aligned(out, 16) || !aligned(topk_ids, 4) ||
        !aligned(topk_weights, 4))
      return MOE_ERR_INVALID_ARG;
  }
  void *scratch = nullptr;
  moe_status st = no_alloc_scratch(&scratch);
  if (st != MOE_OK) return st;
  moe_binding_s b;  // on the stack: nothing is allocated, on the host or the device
  b.P = *plan;
  b.scratch = static_cast<uint8_t *>(scratch);
  b.packed = static_cast<const uint8_t *>(packed);
  b.x = x;
  b.ids = topk_ids;
  b.w = topk_weights;
  b.T = num_tokens;
  b.out = out;
  return run_impl(&b, stream, nullptr);
}

extern "C" moe_status moe_no_alloc_device_status(moe_plan_t plan, cudaStream_t stream, int32_t *status) {
  if (!plan || !status) return MOE_ERR_INVALID_ARG;
  void *scratch = nullptr;
  moe_status st = no_alloc_scratch(&scratch);
  if (st != MOE_OK) return st;
  int32_t w[4] = {0, 0, 0, 0};
  if (cudaMemcpyAsync(w, static_cast<uint8_t *>(scratch) + plan->S.status, sizeof w, cudaMemcpyDeviceToHost,
                      stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  for (int i = 0; i < 4; ++i) status[i] = w[i];
  return (w[ST_FLAGS] & ST_FLAG_TIMEOUT) ? MOE_ERR_TIMEOUT : MOE_OK;
}
