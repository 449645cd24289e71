// Host-side layouts and kernel launchers of libmoe (internal; not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace bqmoe {

constexpr size_t kAlign = 256;
// Work counters per grouped launch of the register-dequant kernel (one per CTA
// group; zeroed by the routing kernel at the start of every forward).
constexpr int kWorkSlots = 512;
// Largest expert count a layer may have (moe_plan_weights rejects more).
constexpr int kMaxExperts = 512;
inline size_t align_up(size_t v, size_t a = kAlign) { return (v + a - 1) / a * a; }

// Packed expert buffer written by the packer, segments on 256-byte boundaries:
//   c13  W13 (gate and up rows, or W1; N13 rows x H) codes and block scales,
//        interleaved per 128-row block and 64-wide K step in mma.m16n8k16
//        A-fragment order (see the packer)
//   c2   W2 (H rows x I), same layout
//   g    float [E][4] global scales (gate|w1, up, down, 1); all 1 for MXFP4
//   t13, t2  (MOE_WFLAG_FP4_TILES, NVFP4) per expert, 128-row block and
//        256-K block: a 16 KB 128-byte-swizzled tile of E2M1 codes, then the
//        block scales of the block's 128 rows as 2 KB in tensor-memory order
//        (see the packer)
struct WeightLayout {
  int E = 0, H = 0, I = 0, wfmt = 0, act = 0;
  int bs = 16;   // elements per block scale (16 NVFP4, 32 MXFP4)
  int n13 = 0;   // rows of W13
  bool fp4_tiles = false;
  size_t off_c13 = 0, off_c2 = 0, off_g = 0, off_t13 = 0, off_t2 = 0, total = 0;
  // FP4 tiles: bytes of one (128-row block, 256-K block) tile + its scales
  static constexpr size_t kFp4TileBytes = 16384 + 2048;
  size_t t13_expert() const { return (size_t)(n13 / 128) * (H / 256) * kFp4TileBytes; }
  size_t t2_expert() const { return (size_t)(H / 128) * (I / 256) * kFp4TileBytes; }
  // bytes of one expert's W13 / W2 segment (codes + block scales)
  size_t blk13_expert() const { return (size_t)n13 * H / 2 + (size_t)n13 * H / bs; }
  size_t blk2_expert() const { return (size_t)H * I / 2 + (size_t)H * I / bs; }
  // bytes of one 64-K step of a 128-row block
  int step_bytes() const { return 4096 + 128 * 64 / bs; }
};

// One slot-major MX FP8 activation tile (128 slots x 128 K) of the block-scaled
// FP8 kernel: 16 KB of E4M3 codes + 512 bytes of UE8M0 scales in TMEM order.
constexpr int kMx8TileBytes = 16384 + 512;

// Scratch owned by the caller and carved by the plan (offsets in bytes).
struct ScratchLayout {
  int64_t cap_sorted = 0;  // rows of the padded, expert-sorted pair list
  size_t status = 0, counts = 0, offsets = 0, sorted = 0, pair_pos = 0, active = 0, passes = 0, large = 0, large_tiles = 0;
  size_t tiles = 0;       // token-tile records of the large experts (int4 each)
  size_t route_hist = 0;  // per-chunk expert counts of the chunked routing sort
  size_t work = 0;        // 2 x kWorkSlots work counters of the register-dequant kernel (GEMM1, GEMM2)
  size_t xq_codes = 0, xq_scales = 0, xq_g = 0;
  size_t h = 0, hq_codes = 0, hq_scales = 0, hq_g = 0;
  size_t x16 = 0, xfac = 0, hamax = 0;  // tensor-core path: FP16 x, its factors, per-pair max |h|
  size_t h16 = 0, h16fac = 0;           // tcgen05 path: 16-bit h rows (and their FP16 factors)
  size_t xb16 = 0;                      // tcgen05 path, MXFP4: BF16 slot-order x rows
  size_t xt = 0, ht = 0;                // FP4 path: x^ / h^ as slot-major 128-row tiles (codes + scales)
  size_t xs16 = 0;                      // CTA-pair path: GEMM1's 16-bit x rows gathered into slot order
  size_t gbar = 0;                      // single-launch path: grid barrier words
  size_t part = 0, total = 0;
};

// Activation sources the grouped kernels can stage.
enum Src { SRC_X_BF16 = 0, SRC_X_NVFP4 = 1, SRC_X_MXFP8 = 2, SRC_H_F32 = 3, SRC_H_NVFP4 = 4, SRC_H_MXFP8 = 5,
           SRC_X16 = 6 /* FP16 rows + per-row factor, staged by launch_stage_x16 */ };
// Grouped-kernel stage.
enum Stage { STAGE_GATED = 0, STAGE_RELU2 = 1, STAGE_DOWN = 2 };

struct GroupedArgs {
  // expert weights of this stage
  const uint8_t *codes;  // expert 0 base of the packed segment (codes + block scales)
  size_t codes_expert;   // bytes per expert
  const float *globals;  // [E][4]
  int K;       // reduction length
  int n_blocks;  // 128-row blocks of the stage's weight matrix (set by the mma launcher)
  int n_rows;  // I (GEMM1 features) or H (GEMM2 rows)
  int I;       // intermediate (gated: up rows start at I)
  // activation source
  const void *act;            // bf16 x [T][H] | f32 h [cap][I] | codes | FP16 x16 [T][H]
  const uint8_t *act_scales;  // block scales (quantised sources)
  const float *act_g;         // per-row NVFP4 global | x16 factor | |h| maximum per pair (SRC_H_F32, mma)
  float *out_amax;            // GEMM1 on the mma path: per-pair max |h| (atomicMax), or null
  // routing
  const int32_t *counts, *offsets, *sorted_pair;
  const int32_t *active;  // [0] = number of experts with pairs, [1..] their ids (ascending)
  const int32_t *passes;  // [i] = passes of active experts before i (prefix, n_active + 1 entries)
  const int32_t *large;        // experts for the tcgen05 kernel: [0] = n, [1..] ids
  const int32_t *large_tiles;  // [i] = token tiles of large experts before i (prefix)
  const int4 *tiles;           // per token tile of the large experts: (expert, first slot, live tokens, 0)
                               // (balanced tiles of up to 256 for the CTA-pair kernel, 128 for the FP4 one)
  int act_by_token;            // tcgen05 kernel: B rows indexed by token (GEMM1) or by slot (GEMM2)
  int32_t *status;        // device status word (timeout flag)
  int32_t *work;          // register-dequant kernel: kWorkSlots zeroed item counters
  int tiny;               // register-dequant kernel: at most E/8 pairs (one deep-ring CTA per SM)
  int wait_first;         // register-dequant GEMM1: routing triggered early, wait before triggering
  int top_k;
  const float *topk_weights;
  // output: h [cap][I] (GEMM1) or partials [cap][H] (GEMM2)
  float *out;
  int out_bf16;  // GEMM2: the partials are BF16 (out reinterpreted), else FP32
};

// A GEMM2 partial (topk_weight x g_down x W2 h) into the FP32 or BF16 partial array.
__device__ __forceinline__ void store_partial(const GroupedArgs &a, size_t idx, float v) {
  if (a.out_bf16) reinterpret_cast<__nv_bfloat16 *>(a.out)[idx] = __float2bfloat16_rn(v);
  else a.out[idx] = v;
}

// Optional staging done by extra CTAs of the routing launch: BF16 x [T][H] ->
// FP16 rows + per-row factor, and clearing of `zero` (zero_n floats).
struct RouteStaging {
  const __nv_bfloat16 *x;
  int T, H;
  __half *x16;
  float *xfac, *zero;
  int64_t zero_n;
};

// ntok: tokens per pass of the register-dequant kernel; experts with at least
// large_min pairs go to the tcgen05 kernel in tiles of large_tile tokens.
// Above 1024 pairs the sort runs in route_chunks(P) chunks and needs
// chunk_hist: route_chunks(P) * (E + 1) ints of scratch.
int route_chunks(int P);
cudaError_t launch_route(const int32_t *ids, int P, int E, int pad, int ntok, int large_min, int large_tile,
                         int32_t *counts, int32_t *offsets, int32_t *sorted_pair, int32_t *pair_pos, int32_t *active,
                         int32_t *passes, int32_t *large, int32_t *large_tiles, int4 *tiles, int balanced,
                         int32_t *status, int32_t *chunk_hist, int32_t *work, int work_n, const RouteStaging *stg,
                         cudaStream_t s);

// Register-dequant tensor-core grouped kernel (experts with few pairs), NVFP4 or
// MXFP4 weights (wfmt); rows_total = rows of the stage's weight matrix (2I gated,
// I for ReLU^2, H for the down projection).  Tokens per pass (8, or 16 when
// `wide` and the staging fits); the routing kernel's pass prefix must use the
// same value.
int mma_tokens_per_pass(int H, int I, bool wide);
cudaError_t launch_grouped_mma(int wfmt, int src, int stage, const GroupedArgs &a, int rows_total, int E, int ntok,
                               cudaStream_t s);

cudaError_t launch_stage_x16(int src, const void *act, const uint8_t *act_scales, const float *act_g, int T, int K,
                             __half *x16, float *fac, float *zero, int64_t zero_n, cudaStream_t s);

// tcgen05 kernels for experts with many pairs, on CTA pairs
// (tcgen05.mma.cta_group::2, M = 256, token tiles of up to 256 from routing's
// large_tile = 256 prefix): NVFP4 weights (FP16 operands) or MXFP4 weights
// (BF16 operands), both from the packed fragment layout; rows_total a multiple
// of 256.
bool tc2_supported(int rows_total, int K);
// a.act: the activation rows in slot order, b_rows of a.K 16-bit values (GEMM1:
// x gathered with launch_gather_slot_rows; GEMM2: h16).
cudaError_t launch_grouped_tc2(int stage, int wfmt, const GroupedArgs &a, int rows_total, int64_t b_rows,
                               cudaStream_t s);
// dst[s] = src[sorted[s] / top_k] (rows of cols16 16-bit values) for the live
// slots s < *n_live; padding slots are skipped.
cudaError_t launch_gather_slot_rows(const void *src, const int32_t *sorted, const int32_t *n_live, int top_k,
                                    int cols16, int64_t cap_rows, void *dst, cudaStream_t s);
// Block-scaled FP4 tcgen05 kernel for NVFP4 weights with NVFP4 activations (the
// weights' FP4 tiles; a.act / act_scales / act_g = the quantised activations).
bool fp4_tc_supported(int rows_total, int K);
cudaError_t launch_grouped_fp4(int stage, const GroupedArgs &a, int rows_total, cudaStream_t s);
// Block-scaled FP8 kernel (kind::mxf8f6f4) for MXFP4 weights x MXFP8
// activations, experts with many pairs: the weights' packed fragments widened
// to E4M3 in shared memory, the activations as slot-major MX FP8 tiles
// (launch_quant_blocks with tiles), 128-token tiles from a.tiles.
bool mx8_tc_supported(int rows_total, int K);
cudaError_t launch_grouped_mx8(int stage, const GroupedArgs &a, int rows_total, cudaStream_t s);
// h (or its re-quantised codes) as 16-bit rows for the tcgen05 GEMM2: FP16 with a
// per-row factor, or BF16 with factor 1 (out_bf16; also MXFP8 x^ -> BF16 rows).
// rows_dev (device, nullable) caps the rows actually converted.  pair_order:
// the CTA-pair kernel's K order (h rows) instead of the slot order (x rows that
// the slot-order gather reorders).
cudaError_t launch_stage_h16(int src, const void *act, const uint8_t *act_scales, const float *act_g, int K,
                             int64_t rows, const int32_t *rows_dev, __half *h16, float *fac, bool out_bf16,
                             bool pair_order, cudaStream_t s);

// Single-launch decode forward (unified.cuh): supported formats and sizes,
// and the launch (args filled by the caller; nst / ngroups set here).
struct UnifiedArgs;
bool unified_supported(int wfmt, int afmt, int P, int E, int K);
cudaError_t launch_unified(int wfmt, int afmt, int stage1, int ntok, bool tiny, UnifiedArgs u, cudaStream_t s);

// Ordered per-token sum of the partials (FP32, or BF16 when part_bf16).
// out: BF16 [T][H], or FP32 with out_f32 (a rank's partial of a tensor-parallel layer).
cudaError_t launch_combine(const void *part, bool part_bf16, int H, const int32_t *pair_pos, int T, int K,
                           void *out, bool out_f32, cudaStream_t s);

// Quantisers.  `rows_dev`, when non-null, is a device int with the number of
// rows that are live; rows at or beyond it are skipped, and so are rows r with
// row_live[r] < 0 when row_live (the expert-sorted pair list) is non-null.
// With `tiles` (cols a multiple of 256) the codes and scales also go to the
// slot-major FP4 tiles of the block-scaled kernel: token row r to the slots
// tile_slots[r * top_k + k] (top_k > 0), or row r to slot r (top_k == 0).
cudaError_t launch_quant_rows_nvfp4(const void *src, bool src_bf16, int64_t rows, int64_t cols,
                                    uint8_t *codes, uint8_t *scales, float *g, const int32_t *rows_dev,
                                    const int32_t *row_live, cudaStream_t s, uint8_t *tiles = nullptr,
                                    const int32_t *tile_slots = nullptr, int top_k = 0);
// With `tiles` (MXFP8 only, cols a multiple of 128): also the slot-major MX FP8
// tiles of the block-scaled FP8 kernel, token row r to the slots
// tile_slots[r * top_k + k] (top_k > 0), or row r to slot r (top_k == 0).
cudaError_t launch_quant_blocks(int qfmt, const void *src, bool src_bf16, int64_t rows, int64_t cols,
                                int64_t rows_per_global, const float *g, uint8_t *codes, uint8_t *scales,
                                const int32_t *rows_dev, const int32_t *row_live, cudaStream_t s,
                                uint8_t *tiles = nullptr, const int32_t *tile_slots = nullptr, int top_k = 0);
cudaError_t launch_amax_tensor(const void *src, bool src_bf16, int64_t batch, int64_t elems, float *amax,
                               cudaStream_t s);
cudaError_t launch_amax_to_global(float *g, int64_t n, cudaStream_t s);

cudaError_t launch_pack(const WeightLayout &L, const void *w13_codes, const void *w13_scales,
                        const float *w13_global, const void *w2_codes, const void *w2_scales,
                        const float *w2_global, uint8_t *packed, cudaStream_t s);

}  // namespace bqmoe
