/*
 * moe.h -- C ABI of the GB300 (sm_103a) block-quantised fused MoE library.
 *
 * The operation is the fused routed-expert FFN over FP4 block-quantised expert
 * weights: the pages' moe.fused_moe, which runs a small-batch decode path, a
 * persistent-grid path and a W4A16 mode where BF16 activations meet FP4
 * weights dequantised inside the kernel (b12x project page (shadowgraph.io),
 * section "What's in here"):
 *
 *     y_t = sum_k  w_tk * W2_e( act( W13_e x^_t ) ),   e = topk_ids[t, k]
 *
 * with act = SiLU(gate) * up (gated) or max(., 0)^2 (non-gated ReLU^2; vLLM
 * docs "b12x Linear and MoE Backends", section "ModelOpt block codecs": the
 * routed experts carry no bias and use SiLU or a non-gated ReLU^2).  Supported
 * formats follow the same docs, section "Supported Configurations": NVFP4
 * weights with BF16, NVFP4 or MXFP8 activations; MXFP4 weights with BF16 or
 * MXFP8 activations.
 *
 * The calls mirror the pages' plan -> scratch -> bind -> run contract (b12x
 * project page, section "Using it"):
 *
 *   moe_plan_weights    host only; decides the packed layout of the experts.
 *   moe_prepare_weights one-time repack of the checkpoint tensors into that
 *                       layout on the GPU (the pages prepare the weights once
 *                       per model).
 *   moe_plan            host only; fixes every launch decision for a capacity
 *                       (max_tokens) and reports the scratch size.  Live token
 *                       counts are not part of a plan (b12x has moved to
 *                       FlashInfer, section "Technical layout and contracts":
 *                       the workspace has a fixed capacity and live request
 *                       counts never enter a compile key).
 *   moe_bind            host only; records pointers (on the pages, bind only
 *                       makes views of caller tensors and never allocates).
 *   moe_run             launches the kernels on the caller's stream; it never
 *                       allocates, synchronises or compiles, so it can be
 *                       captured in a CUDA graph (the pages' run is safe under
 *                       CUDA-graph capture).
 *
 * Ownership.  The caller owns all device memory: source weights, the packed
 * buffer, scratch, activations, ids, weights and the output.  The library owns
 * only the host-side plan and binding objects and allocates no device memory.
 *
 * Errors.  Every call returns a moe_status and never throws or aborts.  Argument
 * errors are found on the host before anything is launched.  Conditions found
 * on the device (out-of-range expert ids, which are dropped) are recorded in a
 * status word inside scratch and read back with moe_device_status.
 *
 * Shapes.  hidden must be a multiple of 128 and intermediate a multiple of 64;
 * moe_is_supported also requires the rows of W13 (2I gated, I for ReLU^2) to be
 * a multiple of 128 (the tensor-core kernels work on 128-row blocks).
 * All device pointers must be 16-byte aligned.
 */
#ifndef BQMOE_MOE_H
#define BQMOE_MOE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,       /* null pointer, bad size, misaligned pointer   */
  MOE_ERR_UNSUPPORTED = 2,       /* shape / format combination not implemented  */
  MOE_ERR_CAPACITY = 3,          /* num_tokens > max_tokens, or host buffer short */
  MOE_ERR_SCRATCH_TOO_SMALL = 4, /* scratch_bytes below what moe_plan reported   */
  MOE_ERR_CUDA = 5,              /* a CUDA runtime call or launch failed         */
  MOE_ERR_TIMEOUT = 6            /* a bounded device-side wait gave up           */
} moe_status;

/* Expert weight formats.
 * NVFP4: E2M1 codes, one E4M3 scale per 16 elements along K, one FP32 global
 *        scale per expert and per matrix (gate, up, down).
 * MXFP4: E2M1 codes, one E8M0 scale per 32 elements along K, no global. */
enum { MOE_W_NVFP4 = 1, MOE_W_MXFP4 = 2 };

/* Activation formats (what GEMM1 and GEMM2 consume).
 * BF16 : x as given, h kept in floating point ("W4A16").
 * NVFP4: x and h re-quantised per token row: E2M1 + E4M3 / 16 + FP32 global per row.
 * MXFP8: x and h re-quantised: E4M3 elements + E8M0 scale per 32. */
enum { MOE_A_BF16 = 1, MOE_A_NVFP4 = 2, MOE_A_MXFP8 = 3 };

/* Expert activation. */
enum { MOE_ACT_SILU_GATED = 1, MOE_ACT_RELU2 = 2 };

/* Weight packing flags (moe_weight_desc.flags).
 * MOE_WFLAG_FP4_TILES: NVFP4 only.  Also store every 128-row x 256-K block of
 * W13 and W2 as a 128-byte-swizzled tile of E2M1 codes plus its E4M3 scales
 * arranged for tensor memory, which the prefill kernel feeds straight to the
 * block-scaled FP4 tensor-core MMA when the activations are NVFP4 (W4A4; b12x
 * project page, "What's in here": NVFP4 activations).  Costs another 0.5625
 * bytes per weight element.  Without it W4A4 prefill dequantises to FP16. */
enum { MOE_WFLAG_FP4_TILES = 1 };

typedef struct moe_weight_desc {
  int32_t num_experts;   /* E, 1..512                         */
  int32_t hidden;        /* H, multiple of 128                */
  int32_t intermediate;  /* I, multiple of 64                 */
  int32_t wfmt;          /* MOE_W_*                           */
  int32_t act;           /* MOE_ACT_*                         */
  int32_t flags;         /* MOE_WFLAG_* bits, 0 for none      */
} moe_weight_desc;

typedef struct moe_weight_plan_s *moe_weight_plan;
typedef struct moe_plan_s *moe_plan_t;
typedef struct moe_binding_s *moe_binding;

typedef struct moe_caps {
  moe_weight_plan wplan; /* from moe_plan_weights                             */
  int32_t top_k;         /* K, 1..16                                          */
  int32_t max_tokens;    /* capacity T_max >= 1; scratch is sized for it      */
  int32_t afmt;          /* MOE_A_*                                           */
} moe_caps;

/* Human-readable name of a status code (static storage, never NULL). */
MOE_API const char *moe_status_str(moe_status s);

/* ----------------------------------------------------------- weights ---- */

/* Validate a weight description and report the size of the packed buffer
 * (b12x project page, "Using it": fused_moe.plan_weights(quant_modes=...,
 * source_format="modelopt_nvfp4")).  Host only.  *out is owned by the caller
 * and released with moe_destroy_weight_plan. */
MOE_API moe_status moe_plan_weights(const moe_weight_desc *desc, moe_weight_plan *out,
                            size_t *packed_bytes);

/* Repack checkpoint tensors into `packed` (b12x project page, "Using it":
 * fused_moe.prepare_weights, run once per model).  All pointers
 * are device pointers, read-only except `packed`.  Source layout (the
 * modelopt_nvfp4 reading: row-major, K contiguous, two E2M1 codes per byte,
 * element 2j in the low nibble):
 *   w13_codes  uint8 [E, N13, H/2]   N13 = 2I (gate rows [0,I) then up rows [I,2I)) or I (ReLU^2)
 *   w13_scales uint8 [E, N13, H/bs]  bs = 16 (E4M3, NVFP4) or 32 (E8M0, MXFP4)
 *   w13_global float [E, N13/I]      NVFP4 only (gate, up) or (w1); NULL for MXFP4
 *   w2_codes   uint8 [E, H, I/2]
 *   w2_scales  uint8 [E, H, I/bs]
 *   w2_global  float [E]             NVFP4 only; NULL for MXFP4
 *   packed     device buffer of packed_bytes (from moe_plan_weights)
 * Asynchronous on `stream`; the sources may be freed once the stream has
 * passed this call. */
MOE_API moe_status moe_prepare_weights(moe_weight_plan wplan, const void *w13_codes,
                               const void *w13_scales, const float *w13_global,
                               const void *w2_codes, const void *w2_scales,
                               const float *w2_global, void *packed,
                               cudaStream_t stream);

/* ------------------------------------------------------- plan / bind ---- */

/* MOE_OK if the library has kernels for these caps, else MOE_ERR_UNSUPPORTED
 * or MOE_ERR_INVALID_ARG (b12x project page, "Using it": every op exports
 * is_supported()).  Host only. */
MOE_API moe_status moe_is_supported(const moe_caps *caps);

/* Fix every launch decision for `caps` and report the scratch size and the
 * tile (m_tile) that expert groups are padded to (b12x project page, "Using
 * it": plan is host-side; plan.scratch_specs()).  Host only; the weight plan
 * may be destroyed afterwards (the plan keeps a copy). */
MOE_API moe_status moe_plan(const moe_caps *caps, moe_plan_t *out, size_t *scratch_bytes,
                    int32_t *m_tile);

/* Plan options (moe_plan_set_option).
 * MOE_OPT_SINGLE_LAUNCH: 1 runs a decode plan's
 *   whole forward as one persistent launch, the pages' unified dynamic path
 *   (b12x project page, "What's in here": a persistent-grid path for NVFP4 and
 *   MXFP8 activations): routing, the activation quantiser, GEMM1, the h
 *   re-quantiser, GEMM2 and the combine run as phases of one cooperative grid,
 *   separated by grid barriers whose waits are bounded.  Supported for plans of
 *   at most 1024 (token, slot) pairs (max_tokens x top_k) with NVFP4 weights
 *   and BF16, NVFP4 or MXFP8 activations, or MXFP4 weights and BF16 or MXFP8
 *   activations.  0 (the default) runs one launch per stage, each launched
 *   with programmatic dependent launch so that a stage's set-up and weight
 *   stream overlap the end of the one before; that overlap makes the
 *   per-stage launches faster on decode batches than the grid barriers of the
 *   single launch.  Both give bit-identical outputs; moe_run_timed always runs
 *   one launch per stage. */
/* MOE_OPT_OUT_F32: 1 makes `out` FP32 [num_tokens, H] instead of BF16: the
 *   forward's per-token sums before their rounding to BF16, for a layer split
 *   over ranks along the intermediate dimension (tensor parallelism: b12x
 *   project page, "What's in here", the fused FP4 TP MoE), where each rank's
 *   result is a partial sum that the ranks add in a fixed order before
 *   rounding.  Not combinable with MOE_OPT_SINGLE_LAUNCH (MOE_ERR_UNSUPPORTED).
 *   moe_run_host copies 4-byte elements back. */
enum { MOE_OPT_SINGLE_LAUNCH = 1, MOE_OPT_OUT_F32 = 2 };

/* Set a plan option; applies to bindings made afterwards.  Host only.
 * MOE_ERR_UNSUPPORTED if the plan cannot take the value, MOE_ERR_INVALID_ARG
 * for an unknown option. */
MOE_API moe_status moe_plan_set_option(moe_plan_t plan, int32_t option, int32_t value);

/* Record the pointers of one forward (b12x project page, "Using it":
 * fused_moe.bind(plan, scratch=..., a=x, experts=..., topk_weights=tw,
 * topk_ids=ti)).  Host only; nothing is read or written on the device.
 *   scratch       device, >= scratch_bytes from moe_plan, 256-byte aligned
 *   packed        device, the buffer written by moe_prepare_weights
 *   x             device, BF16 [num_tokens, H]
 *   topk_ids      device, int32 [num_tokens, K]; ids outside [0, E) are dropped
 *   topk_weights  device, float [num_tokens, K]
 *   num_tokens    0..max_tokens (0 makes moe_run a no-op)
 *   out           device, BF16 [num_tokens, H] (FP32 with MOE_OPT_OUT_F32)
 * The binding holds no reference to the plan; destroy it with
 * moe_destroy_binding. */
MOE_API moe_status moe_bind(moe_plan_t plan, void *scratch, size_t scratch_bytes,
                    const void *packed, const void *x, const int32_t *topk_ids,
                    const float *topk_weights, int32_t num_tokens, void *out,
                    moe_binding *out_binding);

/* ----------------------------------------------------------------- run -- */

/* Run the bound forward on `stream` (b12x project page, "Using it":
 * fused_moe.run(binding)): routing, activation quantiser (NVFP4/MXFP8),
 * GEMM1 + activation, re-quantisation of h (NVFP4/MXFP8), GEMM2 scaled by
 * topk_weights, and a deterministic per-token combine into `out`.
 * Asynchronous; no allocation, no synchronisation; capturable. */
MOE_API moe_status moe_run(moe_binding b, cudaStream_t stream);

/* End-to-end variant for callers holding host buffers: copies x, topk_ids and
 * topk_weights from host memory into the bound device buffers, runs, copies
 * `out` back to host memory and synchronises `stream`.  Host buffers have the
 * shapes given to moe_bind; pinned memory makes the copies asynchronous. */
MOE_API moe_status moe_run_host(moe_binding b, const void *x_host, const int32_t *ids_host,
                        const float *weights_host, void *out_host,
                        cudaStream_t stream);

/* Stages of moe_run, in launch order, for moe_run_timed. */
enum { MOE_STAGE_ROUTE = 0, MOE_STAGE_QUANT_X = 1, MOE_STAGE_GEMM1 = 2, MOE_STAGE_QUANT_H = 3,
       MOE_STAGE_GEMM2 = 4, MOE_STAGE_COMBINE = 5, MOE_NUM_STAGES = 6 };

/* moe_run that also records caller-created CUDA events around every stage
 * (the per-kernel timing of the pages' B12X_TIMING=1 switch, b12x project
 * page, section "PCIe DMA wire modes", last paragraph): events[i] is recorded
 * on `stream` just before stage i and events[MOE_NUM_STAGES] after the last
 * stage, so cudaEventElapsedTime(events[i], events[i+1]) is the device time of
 * stage i (zero for a stage the activation format skips).  `events` is a host
 * array of MOE_NUM_STAGES+1 cudaEvent_t created with timing enabled.  Nothing
 * is synchronised.  Under stream capture the events are recorded as external
 * event nodes (cudaEventRecordExternal), so every replay of the graph records
 * them again. */
MOE_API moe_status moe_run_timed(moe_binding b, cudaStream_t stream, cudaEvent_t *events);

/* Number of kernels the last forward on `b` (moe_run, moe_run_timed or
 * moe_run_host) enqueued, counted on the host as they were launched; 0 before
 * the first forward.  Lets a caller count device launches per forward (for
 * example to size a CUDA graph or to report launches per step).  No CUDA call. */
MOE_API moe_status moe_launch_count(moe_binding b, int32_t *n);

/* Copy the device status word of the last run to host `status[4]` and
 * synchronise `stream`:
 *   status[0] flags: bit 0 = out-of-range ids were dropped, bit 1 = a bounded
 *             device wait timed out;
 *   status[1] number of dropped (token, slot) pairs;
 *   status[2], status[3] reserved (0).
 * Returns MOE_ERR_TIMEOUT if bit 1 is set, else MOE_OK. */
MOE_API moe_status moe_device_status(moe_binding b, cudaStream_t stream, int32_t *status);

/* Copy the routing stage's outputs of the last run to host memory and
 * synchronise `stream` (for bit-exact checks of the expert sort):
 *   counts [E], offsets [E+1] (each group padded to m_tile), pair_pos [T*K]
 *   (-1 for dropped pairs), sorted_pair [offsets[E]] (pair p = t*K + k, -1 in
 *   padding).  MOE_ERR_CAPACITY if sorted_cap < offsets[E]. */
MOE_API moe_status moe_debug_routing(moe_binding b, cudaStream_t stream, int32_t *counts,
                             int32_t *offsets, int32_t *pair_pos,
                             int32_t *sorted_pair, int32_t sorted_cap);

/* Copy GEMM1's output h of the last run to host memory and synchronise
 * `stream` (for checks of the first contraction on its own): h [rows][I] FP32,
 * one row per slot of the expert-sorted pair list (moe_debug_routing's
 * sorted_pair gives each slot's pair; rows of padding slots are unspecified),
 * before any re-quantisation.  *rows = offsets[E].  MOE_ERR_CAPACITY if
 * rows_cap < offsets[E]; a run with no tokens gives *rows = 0. */
MOE_API moe_status moe_debug_hidden(moe_binding b, cudaStream_t stream, float *h, int32_t rows_cap,
                                    int32_t *rows);

/* Self-test of the failure detection (no counterpart on the pages).  Every
 * device-side wait in this library is bounded: a wait that nothing completes
 * gives up after about two seconds, sets bit 1 (timeout) of the status word
 * and lets its kernel return, so the CUDA context stays usable.  This call
 * clears the caller's device status word `status_dev` (int32_t[4]), launches
 * one CTA on `stream` whose mbarrier wait nothing completes, copies the status
 * word to host `status[4]` and synchronises `stream`.  Returns MOE_ERR_TIMEOUT
 * when the wait gave up (the expected outcome), MOE_OK if it did not,
 * MOE_ERR_INVALID_ARG for a null pointer, MOE_ERR_CUDA on a CUDA error.  Takes
 * about two seconds; allocates nothing. */
MOE_API moe_status moe_selftest_wait_timeout(cudaStream_t stream, int32_t *status_dev, int32_t *status);

/* Self-test of the single-launch forward's grid barriers (no counterpart on
 * the pages).  Runs the binding's single-launch forward once with CTA 0
 * withholding its arrival at the grid barrier after GEMM1: the other CTAs'
 * bounded waits give up after about two seconds, set bit 1 (timeout) of the
 * status word and carry on, and the kernel returns (the output of this run is
 * void).  Copies the status word to host `status[4]` and synchronises
 * `stream`.  Returns MOE_ERR_TIMEOUT when the waits gave up (the expected
 * outcome), MOE_OK if they did not, MOE_ERR_UNSUPPORTED if the binding's plan
 * does not run as a single launch.  A following moe_run on the binding is a
 * normal forward. */
MOE_API moe_status moe_selftest_grid_barrier_timeout(moe_binding b, cudaStream_t stream, int32_t *status);

/* ------------------------------------------------------ no-allocation run -- */

/* Size of the library-owned scratch array behind moe_run_no_alloc. */
#define MOE_NO_ALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/* The pages have no counterpart to this call; it exists for callers that
 * cannot allocate device memory: plugin or custom-op interfaces that hand the
 * op only its input and output buffers and no workspace, and applications
 * whose memory pool owns the whole device, where an extra cudaMalloc would
 * fail or fragment the pool.
 *
 * Runs the same forward as moe_bind + moe_run for `plan` (x, topk_ids,
 * topk_weights, out and packed as in moe_bind; all device pointers), but its
 * scratch is a file-scope device array of MOE_NO_ALLOC_SCRATCH_BYTES (32 MiB)
 * inside the library instead of a caller buffer.  Every device that loads the
 * library holds that array until the process exits.  The call allocates
 * nothing: no cudaMalloc / cudaFree, no host heap.
 *   - Plans whose scratch (moe_plan's scratch_bytes) exceeds
 *     MOE_NO_ALLOC_SCRATCH_BYTES are rejected with MOE_ERR_CAPACITY, as is
 *     num_tokens > max_tokens; bad pointers give MOE_ERR_INVALID_ARG.
 *   - The first call in a CUDA context looks up the array's device address
 *     (with that device current); make that first call before any stream
 *     capture.  A device reset gives the device a new context, and the next
 *     call looks the address up again.
 *   - All calls share the one array, which keeps the last call's contents; each
 *     call clears what must start at zero.  Calls that overlap on the GPU (other
 *     streams, other host threads) race on it: serialise them.
 *   - Dropped ids and timed-out device waits are recorded in a status word
 *     inside the array; read it with moe_no_alloc_device_status.
 * Asynchronous on `stream` like moe_run. */
MOE_API moe_status moe_run_no_alloc(moe_plan_t plan, const void *packed, const void *x,
                                    const int32_t *topk_ids, const float *topk_weights,
                                    int32_t num_tokens, void *out, cudaStream_t stream);

/* Status word of the last moe_run_no_alloc with tokens on the current device
 * (no counterpart on the pages): copies it from the library's array to host
 * `status[4]` and synchronises `stream`.  Same layout and return codes as
 * moe_device_status: MOE_ERR_TIMEOUT when a bounded device wait gave up,
 * otherwise MOE_OK (status[0] bit 0 and status[1] report dropped ids).
 * `plan` is the plan of that call.  Allocates nothing. */
MOE_API moe_status moe_no_alloc_device_status(moe_plan_t plan, cudaStream_t stream, int32_t *status);

/* ------------------------------------------------------------ quantiser -- */

enum { MOE_Q_NVFP4 = 1, MOE_Q_MXFP4 = 2, MOE_Q_MXFP8 = 3 };
enum { MOE_G_NONE = 0, MOE_G_PER_TENSOR = 1, MOE_G_PER_ROW = 2 };

/* Block-quantise `batch` row-major matrices [rows, cols] (the row quantizers
 * quantization.nvfp4 / quantization.mxfp8, b12x project page, "What's in
 * here"; also the checkpoint-style weight quantiser).  Device pointers:
 *   src     float [batch, rows, cols] (src_bf16 = 0) or BF16 (src_bf16 = 1)
 *   codes   NVFP4/MXFP4: uint8 [batch, rows, cols/2], element 2j in the low
 *           nibble; MXFP8: uint8 [batch, rows, cols] (E4M3)
 *   scales  uint8 [batch, rows, cols/bs]: E4M3 (NVFP4, bs 16) or E8M0 (MX, bs 32)
 *   global  float: [batch] (MOE_G_PER_TENSOR) or [batch, rows] (MOE_G_PER_ROW);
 *           NVFP4 only, NULL for MX formats (gmode must be MOE_G_NONE)
 * NVFP4: g = amax/(6*448); s = E4M3_rne_sat((amax_b/6)/g); q = E2M1_rne_sat(x/(s*g)).
 * MX:    X = floor(log2(amax_b)) - emax (2 for E2M1, 8 for E4M3), clamped to
 *        [-127,127]; s = X+127; q = ELEM_rne_sat(x/2^X).
 * cols must be a multiple of 16 (NVFP4) or 32 (MX).  batch or rows 0 is a no-op. */
MOE_API moe_status moe_quantize(int32_t qfmt, int32_t gmode, int32_t src_bf16,
                        const void *src, int64_t batch, int64_t rows, int64_t cols,
                        void *codes, void *scales, float *global,
                        cudaStream_t stream);

/* ------------------------------------------------------------- destroy -- */

MOE_API void moe_destroy_weight_plan(moe_weight_plan p);
MOE_API void moe_destroy_plan(moe_plan_t p);
MOE_API void moe_destroy_binding(moe_binding b);

/* ------------------------------------------------------- measurement ---- */

/* Issue rate of back-to-back tensor-core MMAs on this device, in TFLOP/s: one
 * CTA per SM issuing `iters` x 4 tcgen05.mma (M=128, N = n in {128, 256}) from
 * fixed shared-memory operands.  kind: MOE_PEAK_F16 (kind::f16, K=16),
 * MOE_PEAK_FP4 (kind::mxf4nvf4 block_scale scale_vec::4X, E2M1 x E2M1 with
 * UE4M3 scales, K=64) or MOE_PEAK_MXFP8 (kind::mxf8f6f4 block_scale
 * scale_vec::1X, E4M3 x E4M3 with UE8M0 scales, K=32).  The roofline
 * denominator of the prefill kernels (no counterpart on the pages).  Allocates
 * 16 bytes of device memory and two events, synchronises the device. */
enum { MOE_PEAK_F16 = 0, MOE_PEAK_FP4 = 1, MOE_PEAK_MXFP8 = 2 };
MOE_API moe_status moe_measure_mma_peak(int32_t kind, int32_t n, int32_t iters, float *tflops);

#ifdef __cplusplus
}
#endif
#endif /* BQMOE_MOE_H */
