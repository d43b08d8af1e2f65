/*
 * moe_lora.h -- C ABI of libmoelora, a GB300 (sm_103a) library for the
 * routed BF16 Mixture-of-Experts layer forward with per-token multi-adapter
 * LoRA.
 *
 * The forward follows the single-stream pipeline described in
 * "[WIP][LoRA] BF16 support for the experimental_sgl_trtllm MoE-LoRA path &
 * lora expert_outer_shared" (yushengsu-thu/sglang#4), "Files changed" table
 * (launcher row) and Flow 1(A):
 *   routing -> permute (bf16 gather) -> gate_up GEMM (K = hidden, N = 2*inter)
 *   -> LoRA-aware SwiGLU (gate_up LoRA delta added before the activation)
 *   -> down GEMM (K = inter, N = hidden) + down LoRA delta -> finalize
 * and the interface of ``trtllm_bf16_routed_moe_lora`` in the prhub digest
 * of sgl-project/sglang#28953 (core.py excerpt).
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers unless stated otherwise.  The
 *     caller owns every buffer; the library never allocates, frees,
 *     synchronises the stream (except moe_read_device_status) or calls back.
 *   - Tensors are dense row-major.  bf16 tensors are passed as void* (the
 *     bits of __nv_bfloat16).  Rows of bf16 tensors must start on 16-byte
 *     boundaries: base pointers 16-byte aligned and H, I multiples of 8.
 *   - Arguments are checked on the host before anything is launched; a
 *     failed check returns a negative moe_status_t and launches nothing.
 *   - Work is enqueued on ``stream`` (a cudaStream_t) in stream order, with
 *     no allocation and no host synchronisation, so a call can be captured
 *     into a CUDA graph.  The device-side status word (see
 *     moe_read_device_status) reports problems found on the device.
 *   - Calls on one stream that share a workspace are ordered by the stream;
 *     calls that overlap on the GPU must not share a workspace.
 */
#ifndef MOE_LORA_H_
#define MOE_LORA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;                          /* cudaStream_t == struct CUstream_st* */
typedef struct CUstream_st* moe_stream_t;
struct CUevent_st;                           /* cudaEvent_t  == struct CUevent_st*  */

#define MOE_LORA_ABI_VERSION 1

typedef enum {
  MOE_OK = 0,
  MOE_ERR_NULL = -1,            /* a required pointer is NULL                         */
  MOE_ERR_SHAPE = -2,           /* a size is out of range (T < 0, top_k > E, ...)     */
  MOE_ERR_ALIGN = -3,           /* a pointer, size or stride breaks the 16-byte rule  */
  MOE_ERR_UNSUPPORTED = -4,     /* outside the supported limits listed below          */
  MOE_ERR_WORKSPACE = -5,       /* workspace NULL, misaligned or too small            */
  MOE_ERR_CUDA = -6,            /* a CUDA runtime/driver call failed                   */
  MOE_ERR_DEVICE_TIMEOUT = -7,  /* device: a pipeline wait hit its time limit         */
  MOE_ERR_BAD_MAPPING = -8,     /* device: token_lora_mapping outside [-1, A)         */
  MOE_ERR_BAD_EXPERT_ID = -9    /* device: a topk id outside [-1, E)                  */
} moe_status_t;

/* Supported limits (larger values return MOE_ERR_UNSUPPORTED). */
#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_TOP_K 32
#define MOE_MAX_RANK 128
#define MOE_MAX_ADAPTERS 64

/* Human-readable name of a status code.  Never returns NULL. */
const char* moe_status_string(int status);

/* ABI version of the loaded library (MOE_LORA_ABI_VERSION at build time). */
int moe_lora_abi_version(void);

/* ---------------------------------------------------------------------------
 * moe_route_topk -- step 1, routing.
 *
 * The pages take the router's top-k ids and weights in sglang's standard
 * top-k format (prhub digest of sgl-project/sglang#28953, lora_dispatch.py
 * and moe_overlap.py excerpts: ``topk_output.topk_ids / topk_weights``) and
 * do not show the routing function.  It is read as: softmax over the logits,
 * top-k, renormalise over the selected experts.  Selection compares the raw
 * float32 logits, ties go to the lower expert id, and slots are ordered by
 * descending logit; weights are exp(l_j - m) / sum exp(l_j' - m) over the
 * selected slots, m the largest selected logit, in float32.
 *
 *   logits   [T, E] float32, device.  NaN logits give unspecified (but valid,
 *            distinct, in-range) ids.
 *   topk_ids [T, top_k] int32, device, written.
 *   topk_w   [T, top_k] float32, device, written.
 * Limits: 1 <= top_k <= min(E, 32), E <= 1024, T >= 0 (T == 0 is a no-op).
 * ------------------------------------------------------------------------- */
int moe_route_topk(const float* logits, int T, int E, int top_k,
                   int32_t* topk_ids, float* topk_w, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * moe_permute -- step 2, expert-grouped permutation and row gather.
 *
 * The "moe::dev::permute (bf16 gather)" stage of the launcher row in the
 * "Files changed" table of yushengsu-thu/sglang#4; the expanded-to-permuted
 * index is the one ``trtllm_bf16_routed_moe_lora`` returns with
 * do_finalize=False (prhub digest of sgl-project/sglang#28953, core.py).
 *
 * Expanded index x = t*top_k + j.  With n_e the number of slots routed to
 * expert e:  expert_offsets[e] = sum_{e' < e} n_e', expert_offsets[E] =
 * number of routed slots; expanded_to_permuted[x] = expert_offsets[id[x]] +
 * #{x' < x : id[x'] == id[x]} (stable); permuted_to_expanded is its inverse
 * on [0, expert_offsets[E]) and -1 beyond.  If ``hidden`` and
 * ``permuted_hidden`` are both non-NULL, permuted_hidden[p] = hidden[t(p)].
 *
 * An id of -1 means "not routed" (the slot gets permuted index -1).  Any
 * other id outside [0, E) is treated like -1 and sets MOE_ERR_BAD_EXPERT_ID
 * in the device status word, which lives at the start of ``ws``.
 *
 *   topk_ids [T, top_k] int32, device.
 *   hidden   [T, H] bf16, device, or NULL (then no gather).
 *   expert_offsets [E + 1], expanded_to_permuted [T*top_k],
 *   permuted_to_expanded [T*top_k]: int32, device, written.
 *   permuted_hidden [T*top_k, H] bf16, device, written, or NULL.
 *   ws, ws_bytes: device scratch of at least moe_permute_workspace_size(),
 *            256-byte aligned; its contents need not be initialised.
 * ------------------------------------------------------------------------- */
size_t moe_permute_workspace_size(int T, int top_k, int E);
int moe_permute(const int32_t* topk_ids, int T, int top_k, int E,
                const void* hidden, int H,
                int32_t* expert_offsets, int32_t* expanded_to_permuted,
                int32_t* permuted_to_expanded, void* permuted_hidden,
                void* ws, size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * moe_permute_noalloc -- moe_permute without a caller-provided scratch buffer.
 *
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory (for instance a plugin running inside a
 * framework that owns all device buffers and forbids cudaMalloc, or an
 * allocator's own start-up code) and so have no spare buffer to pass as
 * moe_permute's ``ws``.  The results are those of moe_permute with the same
 * arguments.
 *
 * Scratch: one fixed device array inside the library (status word plus the
 * per-chunk expert counts, about 256 KiB), held by every GPU that loads the
 * library until the process exits.  Nothing is allocated or freed by a call.
 * Limit: T * top_k <= MOE_NOALLOC_MAX_SLOTS and E <= MOE_MAX_EXPERTS; larger
 * sizes return MOE_ERR_UNSUPPORTED before anything is enqueued.
 * The first call on each device looks up the array's device address on the
 * current device and keeps it for the life of the process; make that first
 * call before any stream capture.  A cudaDeviceReset (or a new primary
 * context on the device) invalidates the kept address: do not call this
 * entry point again on a device after resetting it.
 * Every call on a device uses the same array, and the array keeps the last
 * call's contents: calls whose work overlaps on the GPU (other streams,
 * other host threads) race and give undefined results.  Order them on one
 * stream or with events.
 *
 *   status_out: device int32, or NULL.  When non-NULL it receives the device
 *     status word of this call (MOE_OK, or MOE_ERR_BAD_EXPERT_ID when an id
 *     outside [-1, E) was seen), in stream order.
 * Other arguments as for moe_permute.
 * ------------------------------------------------------------------------- */
#define MOE_NOALLOC_MAX_SLOTS 65536
int moe_permute_noalloc(const int32_t* topk_ids, int T, int top_k, int E,
                        const void* hidden, int H,
                        int32_t* expert_offsets, int32_t* expanded_to_permuted,
                        int32_t* permuted_to_expanded, void* permuted_hidden,
                        int32_t* status_out, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * LoRA factors of one projection (gate_up or down).
 *
 * One rank-r pair per (adapter, expert) (sglang#4 Flow 1(A):
 * ``merged_experts_fused_moe_lora_add`` shrink then expand into the
 * gate_up / down deltas; the shrink intermediate is [tokens, top_k,
 * lora_a.shape[2]] per the prhub report on sgl-project/sglang#28091).
 *   gate_up: A is [r, H], B is [2I, r];   down: A is [r, I], B is [H, r].
 * The factor of (adapter a, expert e) starts at
 *   A + a*a_stride_adapter + e*a_stride_expert   (elements of bf16)
 * and its rows are contiguous.  An expert stride of 0 makes that factor
 * shared by all experts: the "shared-outer (TML)" layout of sglang#4 Flow 2,
 * where gate_up A is [1, r, H] and down B is [1, H, r] per adapter.
 * Strides must be multiples of 8 elements and of r for the B factor.
 * ------------------------------------------------------------------------- */
typedef struct {
  const void* A;
  const void* B;
  int64_t a_stride_adapter, a_stride_expert;
  int64_t b_stride_adapter, b_stride_expert;
} moe_lora_factors_t;

/* Number of stage boundaries recorded when moe_lora_args_t.stage_events is set. */
#define MOE_NUM_STAGE_EVENTS 8

/* ---------------------------------------------------------------------------
 * Kernel-choice overrides (moe_lora_args_t.tuning), for measurement and
 * tests.  A zeroed struct keeps every choice of the library; the library
 * reads no environment variables, so a captured CUDA graph runs exactly the
 * kernels its arguments name.
 *   cta_pairs:      0 = auto (pairs for 256-wide token tiles), 1 = never,
 *                   2 = pairs for 128- and 256-wide tiles.
 *   shrink_kernel:  0 = auto, 1 = the 16-row-tile LoRA shrink kernel,
 *                   2 = the row-block shrink kernel (not for a shared gate_up
 *                   A factor, which always uses the 16-row kernel).
 *   shrink_in_gemm: 0 = auto (for decode-sized tiles both LoRA shrinks run
 *                   inside the expert GEMMs, after a row-gather kernel),
 *                   1 = never (separate gather/shrink kernels),
 *                   2 = the row gather inside the gate_up GEMM as well.
 *   gemm_max_ctas:  0 = auto (SM count x resident CTAs per SM); otherwise
 *                   at most this many CTAs in each expert GEMM's persistent
 *                   grid (rounded up to a pair for CTA pairs).  Any value is
 *                   correct: no CTA waits on work that a CTA which has not
 *                   started owns.
 * Values outside these sets return MOE_ERR_UNSUPPORTED.
 * ------------------------------------------------------------------------- */
typedef struct {
  int cta_pairs;
  int shrink_kernel;
  int shrink_in_gemm;
  int gemm_max_ctas;
} moe_lora_tuning_t;

/* ---------------------------------------------------------------------------
 * moe_lora_forward arguments.
 *
 *   hidden [T, H] bf16; router_logits [T, E] float32;
 *   w13 [E, 2I, H] bf16 (rows [0, I) gate, rows [I, 2I) up);
 *   w2 [E, H, I] bf16;
 *   token_lora_mapping [T] int32: adapter slot per token, -1 = no adapter;
 *     values outside [-1, num_adapters) are treated as -1 and set
 *     MOE_ERR_BAD_MAPPING in the device status word.  May be NULL when
 *     num_adapters == 0 or rank == 0.
 *   gate_up, down: LoRA factors (ignored when num_adapters == 0 or rank == 0).
 *   scaling: LoRA scale s; each delta is s * B (A x).
 *   out [T, H] bf16, written.
 *   topk_ids_out [T, top_k] int32, topk_w_out [T, top_k] float32,
 *   expanded_to_permuted_out [T*top_k] int32: optional copies of the
 *     routing, NULL to skip.
 *   workspace, workspace_bytes: device scratch of at least
 *     moe_lora_workspace_size(), 256-byte aligned.  It holds the device
 *     status word and every intermediate; see moe_lora_workspace_plan.
 *   tile_n: token-tile width of the expert GEMMs (16, 32, 64, 128 or 256;
 *     0 = chosen from T*top_k/E).
 *   wait_timeout_ms: limit of every device-side pipeline wait (0 = 2000 ms).
 *     A wait that runs out sets MOE_ERR_DEVICE_TIMEOUT and the kernel exits.
 *   debug_flags: 0, or MOE_DEBUG_* bits (failure-path tests only).
 *   adapter_scaling: NULL (every adapter uses ``scaling``) or a HOST array of
 *     num_adapters LoRA scales (e.g. alpha_a / r_a per adapter).  The values
 *     are read during the call and travel with the launches, so a captured
 *     CUDA graph keeps the values of the capture.
 *   Per-adapter ranks: pad each adapter's factors with zero rows (A) and zero
 *     columns (B) to the common ``rank``; the padding contributes exactly 0.
 *   Separate gate and up LoRAs (A_g [r,H], B_g [I,r], A_u [r,H], B_u [I,r]):
 *     pass them as the rank-2r gate_up pair A = [A_g; A_u],
 *     B = [[B_g, 0], [0, B_u]], which gives the same two deltas.
 *   stage_events: NULL, or an array of MOE_NUM_STAGE_EVENTS cudaEvent_t
 *     that are recorded on ``stream`` before the first stage, between
 *     stages and after the last one (unused slots are recorded at the end).
 *   Expert parallelism (the local_expert_offset / local_num_experts
 *   arguments of trtllm_bf16_routed_moe_lora in "[WIP][LoRA] BF16 support for
 *   the experimental_sgl_trtllm MoE-LoRA path & lora expert_outer_shared"):
 *     num_router_experts: experts the router scores (router_logits is then
 *       [T, num_router_experts]); 0 = E, no sharding.
 *     local_expert_offset: this call holds experts [offset, offset + E) of
 *       them; w13, w2 and the LoRA factors are indexed by the local expert.
 *     Routing is global (topk_ids_out holds global ids); slots routed to
 *     experts of other shards are skipped (expanded_to_permuted = -1), so
 *     ``out`` is this shard's partial sum and the sum of ``out`` over a
 *     partition of the experts is the layer output (the caller all-reduces).
 *     Requires E <= num_router_experts <= MOE_MAX_EXPERTS and
 *     0 <= offset <= num_router_experts - E, else MOE_ERR_SHAPE.  Callers
 *     built against the header without these two fields pass the smaller
 *     struct_size and get no sharding.
 *   weight_format, w13_scale, w2_scale: FP8 block-scaled expert weights (see
 *     MOE_WEIGHTS_FP8_E4M3_B128); callers passing a struct_size that ends
 *     before weight_format get bf16 weights.
 *   tuning: kernel-choice overrides (moe_lora_tuning_t); callers passing a
 *     struct_size that ends before it get the library's choices.
 *   side_stream, side_events: the two-stream schedule of the gate_up LoRA
 *     ("[WIP][LoRA] BF16 support for the experimental_sgl_trtllm MoE-LoRA
 *     path & lora expert_outer_shared", Summary "Phase 2" and Flow 1(B): the
 *     gate_up LoRA runs on a second stream and joins on an event before its
 *     result is used).  When side_stream is non-NULL, the gate_up LoRA shrink
 *     U = s A_gu x runs on side_stream while ``stream`` gathers the permuted
 *     rows; side_events[0] (recorded on ``stream`` after the permute) forks
 *     and side_events[1] (recorded on side_stream after the shrink) joins
 *     before the gate_up GEMM, which adds the expand s B_gu U.  The shrinks
 *     then never run inside the GEMMs.  Both events are created by the
 *     caller (cudaEventDisableTiming is fine) and must not be in use by
 *     another call in flight; the sequence can be captured into a CUDA graph
 *     from ``stream`` (the fork/join become graph edges).  With rank 0 or no
 *     adapters the side stream is not used.  NULL events with a non-NULL
 *     side_stream return MOE_ERR_NULL.
 *   activation_format: MOE_ACT_BF16, or MOE_ACT_FP8_E4M3_G128 for the W8A8
 *     path (requires MOE_WEIGHTS_FP8_E4M3_B128 weights, else
 *     MOE_ERR_UNSUPPORTED, and a workspace of moe_lora_workspace_size_ex()
 *     with that format).  Callers passing a struct_size that ends before it
 *     get bf16 activations.
 * ------------------------------------------------------------------------- */
typedef struct {
  uint32_t struct_size;           /* sizeof(moe_lora_args_t) */
  int T, H, I, E, top_k, num_adapters, rank;
  float scaling;
  const void* hidden;
  const void* w13;
  const void* w2;
  const float* router_logits;
  const int32_t* token_lora_mapping;
  moe_lora_factors_t gate_up;
  moe_lora_factors_t down;
  void* out;
  int32_t* topk_ids_out;
  float* topk_w_out;
  int32_t* expanded_to_permuted_out;
  void* workspace;
  size_t workspace_bytes;
  int tile_n;
  int wait_timeout_ms;
  uint32_t debug_flags;           /* 0 in normal use; see MOE_DEBUG_* */
  struct CUevent_st* const* stage_events;
  const float* adapter_scaling;   /* HOST array [num_adapters] or NULL */
  int local_expert_offset;        /* expert parallelism; 0 without sharding */
  int num_router_experts;         /* 0 = E */
  int weight_format;              /* MOE_WEIGHTS_BF16 (0) or MOE_WEIGHTS_FP8_E4M3_B128 */
  const float* w13_scale;         /* FP8: [E, ceil(2I/128), ceil(H/128)] float32 */
  const float* w2_scale;          /* FP8: [E, ceil(H/128), ceil(I/128)] float32 */
  moe_lora_tuning_t tuning;       /* zeroed = the library's choices */
  struct CUstream_st* side_stream;       /* NULL, or see below */
  struct CUevent_st* side_events[2];     /* caller-created events for side_stream */
  int activation_format;          /* MOE_ACT_BF16 (0) or MOE_ACT_FP8_E4M3_G128 */
} moe_lora_args_t;

/* Expert weight formats (moe_lora_args_t.weight_format). */
#define MOE_WEIGHTS_BF16 0
/* w13 [E, 2I, H] and w2 [E, H, I] as float8 e4m3 (finite-only variant: max
 * 448, no infinities, 0x7F/0xFF are NaN), one float32 scale per 128 x 128
 * block of (rows, K): w[e][n][k] = e4m3(q[e][n][k]) * scale[e][n/128][k/128].
 * The block-quant format of the pages' FP8 sibling path
 * (trtllm_fp8_block_scale_routed_moe_lora) as read here; activations stay
 * bf16 and the dequantized weights enter the tensor cores as bf16.
 * Requires H % 16 == 0 and I % 16 == 0 (MOE_ERR_ALIGN) and both scale
 * arrays (MOE_ERR_NULL). */
#define MOE_WEIGHTS_FP8_E4M3_B128 1

/* Activation formats (moe_lora_args_t.activation_format). */
#define MOE_ACT_BF16 0
/* The pages' FP8 path ("[WIP][LoRA] BF16 support for the
 * experimental_sgl_trtllm MoE-LoRA path & lora expert_outer_shared", Flow
 * 1(A): the bf16 path is the FP8 one without a per_token_group_quant_fp8 of
 * the hidden input and without a post-activation quant).  Read as: per row
 * and group of MOE_ACT_FP8_GROUP consecutive columns, in float32, scale =
 * max(amax, 1e-10) / 448 and code = e4m3(x / scale), nearest with ties to
 * even, saturating at +-448 (see moe_per_token_group_quant_fp8).  The
 * hidden rows are quantized before the gate_up GEMM; the activation h =
 * silu(gate) * up is quantized from its float32 value before the down GEMM.
 * Both expert GEMMs multiply e4m3 by e4m3 on the tensor cores, applying the
 * weight-block x token-group scales per 128-K block; the LoRA deltas read
 * the unquantized bf16 hidden rows and activation.  Token tiles are at most
 * 128 wide (tile_n 256 runs as 128). */
#define MOE_ACT_FP8_E4M3_G128 1
#define MOE_ACT_FP8_GROUP 128

/* ---------------------------------------------------------------------------
 * moe_per_token_group_quant_fp8 -- the activation quantizer of the FP8 path.
 *
 * The per_token_group_quant_fp8 step of Flow 1(A) in "[WIP][LoRA] BF16
 * support for the experimental_sgl_trtllm MoE-LoRA path & lora
 * expert_outer_shared".  For output row i and column group g (columns
 * [128 g, 128 g + 128) of K), in float32:
 *   scales[i, g] = max(max_k |x[src(i), k]|, 1e-10) / 448      (IEEE divide)
 *   codes[i, k]  = e4m3(x[src(i), k] / scales[i, g])           (IEEE divide,
 *                  nearest, ties to even, |.| > 448 saturates to 448)
 * with src(i) = row_map[i] / map_div when row_map is non-NULL (a negative
 * row_map[i] gives a zero row: codes 0, scale 1e-10 / 448), else src(i) = i.
 * e4m3 is the finite-only float8 variant (bias 7, max 448).
 *
 *   x        [*, K] device, bf16 (x_is_f32 = 0) or float32 (x_is_f32 = 1),
 *            16-byte aligned.
 *   rows, K  output rows and columns; K a multiple of 16 (MOE_ERR_ALIGN).
 *   row_map  [rows] int32 device, or NULL.  map_div >= 1.
 *   codes    [rows, K] uint8 device, written.
 *   scales   [rows, ceil(K / 128)] float32 device, written.
 * Returns MOE_OK once enqueued; rows == 0 is a no-op.
 * ------------------------------------------------------------------------- */
int moe_per_token_group_quant_fp8(const void* x, int x_is_f32, int rows, int K,
                                  const int32_t* row_map, int map_div, uint8_t* codes,
                                  float* scales, moe_stream_t stream);

/* Test-only flag for debug_flags: the gate_up GEMM's MMA role first waits on
 * a barrier that nothing signals, so its wait runs out after wait_timeout_ms;
 * the kernel then reports MOE_ERR_DEVICE_TIMEOUT, drains its own copies and
 * MMAs, frees its tensor memory and exits (the output is then garbage). */
#define MOE_DEBUG_STALL_GATE_UP_MMA 1u
/* Test-only flag: when the LoRA shrink runs inside the gate_up GEMM
 * (decode-sized tiles), the row flag of permuted row 0 is never raised, so
 * the wait for that row's token tile runs out after wait_timeout_ms with
 * MOE_ERR_DEVICE_TIMEOUT (the output is then garbage).  Without that mode
 * the flag has no effect. */
#define MOE_DEBUG_HOLD_SHRINK_ROW 2u

/* Byte offsets of the intermediates inside the workspace (for inspection). */
typedef struct {
  size_t total_bytes;
  size_t status;              /* int32[4]: status word, detail                 */
  size_t topk_ids;            /* int32 [T*top_k]                               */
  size_t topk_w;              /* float [T*top_k]                               */
  size_t expert_offsets;      /* int32 [E+1]                                   */
  size_t expanded_to_permuted;/* int32 [T*top_k]                               */
  size_t permuted_to_expanded;/* int32 [T*top_k]                               */
  size_t row_adapter;         /* int32 [T*top_k] adapter of each permuted row  */
  size_t permute_scratch;     /* counting-sort scratch, tile tables, adapter
                                 masks, tile flags of the in-GEMM shrink      */
  size_t permuted_hidden;     /* bf16  [T*top_k, H]                            */
  size_t lora_u;              /* bf16  [T*top_k, A*r] s*A_gu x, one-hot slot   */
  size_t act;                 /* bf16  [T*top_k, I]   h = silu(gate)*up        */
  size_t lora_v;              /* bf16  [T*top_k, A*r] s*A_dn h, one-hot slot   */
  size_t expert_out;          /* bf16  [T*top_k, H]   y = w2 h + delta         */
} moe_lora_workspace_plan_t;

/* Fills ``plan`` (host pointer).  Returns MOE_OK or MOE_ERR_SHAPE/UNSUPPORTED. */
int moe_lora_workspace_plan(int T, int H, int I, int E, int top_k, int num_adapters,
                            int rank, moe_lora_workspace_plan_t* plan);
/* Bytes of workspace moe_lora_forward needs with bf16 activations (0 on
 * invalid sizes). */
size_t moe_lora_workspace_size(int T, int H, int I, int E, int top_k, int num_adapters,
                               int rank);
/* As moe_lora_workspace_size, for the given activation_format: FP8
 * activations add, after the bf16 plan, the quantized permuted rows and
 * activation with their scales and the float32 activation (0 on invalid
 * sizes or formats). */
size_t moe_lora_workspace_size_ex(int T, int H, int I, int E, int top_k, int num_adapters,
                                  int rank, int activation_format);

/* ---------------------------------------------------------------------------
 * moe_lora_forward -- the whole layer forward (steps 1-7) on one stream.
 *
 * out[t] = sum_j w[t,j] * ( w2[e] h + s * B_dn (A_dn h) ),
 *   h = silu(g[:I]) * g[I:],  g = w13[e] x_t + s * B_gu (A_gu x_t),
 * e = topk_ids[t, j], LoRA terms present only when mapping[t] >= 0 and
 * rank > 0 (sglang#4 "Files changed" launcher and dispatch rows; Flow 1(A)
 * and Flow 2).  Intermediates are bf16 between kernels; every GEMM
 * accumulates in float32.
 * Limits: H, I multiples of 8; rank a multiple of 8 and <= 128;
 * num_adapters <= 64; E <= 1024; top_k <= 32.
 * Returns MOE_OK once everything is enqueued; device-side problems are in
 * the status word (moe_read_device_status).
 * ------------------------------------------------------------------------- */
int moe_lora_forward(const moe_lora_args_t* args, moe_stream_t stream);

/* Synchronises ``stream``, then returns the device status word that the
 * last call using ``workspace`` left (MOE_OK or a negative device code), or
 * MOE_ERR_CUDA if the synchronisation or the copy failed. */
int moe_read_device_status(const void* workspace, moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_LORA_H_ */
