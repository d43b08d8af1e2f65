// Internal declarations shared by the kernel translation units and the C-ABI
// shim.  Nothing here is part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_lora.h"

namespace moe {

// Raises a kernel's dynamic shared-memory limit once per device, so that the
// launch path itself issues only launches (and stays capturable).
cudaError_t ensure_smem_limit(const void* func, int bytes);

// Launch with programmatic stream serialization: the kernel may start while
// its predecessor drains, and must call griddepcontrol.wait (pdl_wait)
// before touching anything the predecessor writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Token-tile widths for which the permute scan writes per-expert tile
// prefixes: tile_start[bn_index][e] = sum_{e' < e} ceil(n_e' / bn).
constexpr int kNumTileWidths = 5;
__host__ __device__ constexpr int tile_width_of(int idx) { return 16 << idx; }  // 16..256
__host__ __device__ constexpr int tile_width_index(int bn) {
  return bn == 16 ? 0 : bn == 32 ? 1 : bn == 64 ? 2 : bn == 128 ? 3 : 4;
}

// ---------------------------------------------------------------- routing
cudaError_t launch_route_topk(const float* logits, int T, int E, int top_k, int32_t* ids,
                              float* w, cudaStream_t s);

// ---------------------------------------------------------------- permute
struct PermuteParams {
  const int32_t* topk_ids;      // [n] expanded ids
  int n;                        // T * top_k
  int top_k;
  int E;
  int H;
  const __nv_bfloat16* hidden;  // [T, H] or null
  __nv_bfloat16* permuted;      // [n, H] or null
  const int32_t* mapping;       // [T] or null (forward only)
  int num_adapters;
  int32_t* row_adapter;         // [n] or null (forward only)
  int32_t* expert_offsets;      // [E + 1]
  int32_t* e2p;                 // [n]
  int32_t* p2e;                 // [n]
  int32_t* chunk_counts;        // [nchunks, E]
  int32_t* tile_start;          // [kNumTileWidths, E + 1] or null
  int* status;
  // Expert parallelism: ids are global in [0, id_limit); this call holds
  // experts [id_offset, id_offset + E); other ids are dropped.  Without
  // sharding id_offset = 0, id_limit = E.
  int id_offset;
  int id_limit;
};
constexpr int kPermuteChunk = 1024;
// Counting-sort scratch: chunk counts [nchunks, E], the tile prefixes
// [kNumTileWidths, E + 1], then the 16-row-tile adapter masks (gmask_bytes).
size_t permute_scratch_bytes(int n, int E);
size_t gmask_bytes(int n, int E);
// Tile flags of the in-kernel shrink: two arrays (gate_up, down) of
// ceil(n / 16) + E + 1 words each, after the adapter masks.  A 16-wide tile
// index is below ceil(n / 16) + E - 1, so the last word of each array is
// free: it holds that GEMM's row counter (shrink_rows_in_gemm).
size_t shrink_flag_words(int n, int E);
cudaError_t launch_permute(const PermuteParams& p, cudaStream_t s);

// Routing + permute of the forward in three chained kernels (past the one-CTA
// permute; E <= kRoutePermuteMaxE, top_k dividing kPermuteChunk): routing,
// count per chunk of whole tokens, then scan + scatter per chunk.  Writes topk ids and
// weights, expert offsets, both maps, row adapters and the tile prefixes of
// tile_width_mask; chunk_counts needs ceil(T * top_k / kPermuteChunk) x E
// words.  Clears the device status words (status[0..3]).
constexpr int kRoutePermuteMaxE = 256;
struct RoutePermuteParams {
  const float* logits;          // [T, id_limit]
  int T, top_k, E;
  int id_offset, id_limit;      // as in PermuteParams
  int32_t* topk_ids;            // [T * top_k] global ids
  float* topk_w;                // [T * top_k]
  const int32_t* mapping;       // [T] or null
  int num_adapters;
  int32_t* row_adapter;         // [n] or null
  int32_t* expert_offsets;      // [E + 1]
  int32_t* e2p;                 // [n]
  int32_t* p2e;                 // [n]
  int32_t* chunk_counts;        // [nchunks, E]
  int32_t* tile_start;          // [kNumTileWidths, E + 1]
  uint32_t tile_width_mask;
  int* status;
  int tokens_per_chunk;         // set by the launcher
};
bool route_permute_fits(int T, int top_k, int E);
cudaError_t launch_route_permute(const RoutePermuteParams& p, cudaStream_t s);

// ------------------------------------------------- gather + LoRA shrink
// Per 16-row tile of one expert: copy the source rows (gathered[p] = X[src(p)])
// and/or U[p, a*r + i] = bf16(scaling * sum_k A[a, e(p)][i, k] * X[src(p), k])
// for the row's own adapter a, 0 in every other column of the row.
struct ShrinkParams {
  const __nv_bfloat16* X;       // source rows [*, K]
  const int32_t* p2e;           // src(p) = p2e[p] / top_k; null: src(p) = p
  int top_k;
  int K;
  int kc;                       // K elements staged per phase
  __nv_bfloat16* gathered;      // [n, K] row copy, or null
  const __nv_bfloat16* A;       // factor base (ignored when rank == 0 or U == null)
  int64_t a_stride_adapter;     // elements
  int64_t a_stride_expert;      // elements (0 = shared)
  const int32_t* row_adapter;   // [n]
  const int32_t* expert_offsets;// [E + 1]
  const int32_t* tile_start16;  // [E + 1] prefix of ceil(n_e / 16)
  int E;
  int num_adapters;
  int rank;                     // 0: gather only
  float scaling[MOE_MAX_ADAPTERS];  // per adapter
  __nv_bfloat16* U;             // [n, num_adapters * rank], or null
  int* status;
  uint64_t timeout_ns;
  // Per-token mode (gate_up A shared by all experts, so u depends on the
  // token only): tiles of 16 tokens; rows are hidden rows; results and
  // gathered copies go to every permuted row e2p[t*top_k + j] of the token.
  int per_token;
  int T;
  const int32_t* e2p;           // [T * top_k]
  const int32_t* mapping;       // [T]
  const int32_t* tile_start_rows;  // [E + 1] prefix of ceil(n_e / rows_shrink_tile()) (row-block kernel)
  // Or null.  gmask[t]: adapters present in the expert-GEMM token tile that
  // contains 16-row tile t.  The CTA of (t, adapter a) exits at once when a is
  // absent there (no GEMM tile reads a's columns of these rows), unless it
  // owes the row gather (adapter slot 0).
  const uint64_t* gmask;
  // 1 when the routing tables (offsets, tile prefixes, row adapters) are
  // complete at launch (the down shrink, two kernels after the permute): the
  // row-block kernel then reads them and prefetches its factor before it
  // waits for the previous kernel (griddepcontrol.wait).
  int tables_ready;
};
int shrink_chunk(int K, int rank, size_t smem_budget);
// Factor columns one CTA of launch_gather_shrink holds (the rank, or a
// 16-column slice of it in the per-token mode; 0 without U): the rank that
// sizes its K phases.
int gather_shrink_cta_rank(const ShrinkParams& p);
// Per-token mode: the shared-memory budget of one CTA with which the whole
// grid (ceil(T / 16) tiles x adapters x rank slices) is resident at once on
// sms SMs of smem_per_sm bytes each (at most 200 KB; for grids beyond four
// CTAs an SM, the budget of four).
size_t per_token_shrink_budget(const ShrinkParams& p, int sms, size_t smem_per_sm);
cudaError_t launch_gather_shrink(const ShrinkParams& p, int n_rows, cudaStream_t s);
// Many rows: rows_shrink_tile()-row tiles of one expert, K streamed through a cp.async
// pipeline.  Not for the per-token mode.  Uses p.tile_start_rows.
cudaError_t launch_rows_shrink(const ShrinkParams& p, int n_rows, cudaStream_t s);
int rows_shrink_tile();  // rows per CTA of the row-block shrink (a tile width of the tables)

// ------------------------------------------------- one-CTA permute (fused)
struct FusedPermuteParams {
  const float* logits;          // [T, E]: route first; null: read topk_ids
  int32_t* topk_ids;            // [T*k] written (routing) or read
  float* topk_w;                // [T*k] written when routing
  int T, top_k, E;
  const int32_t* mapping;       // [T] or null
  int num_adapters;
  int32_t* row_adapter;         // [n] or null
  int32_t* expert_offsets;      // [E + 1]
  int32_t* e2p;                 // [n]
  int32_t* p2e;                 // [n]
  int32_t* tile_start;          // [kNumTileWidths, E + 1] or null
  uint32_t tile_width_mask;     // bit i: write the prefix for width 16 << i
  int* status;                  // cleared by the kernel
  int id_offset;                // as in PermuteParams; logits are [T, id_limit]
  int id_limit;
  // Or null: per 16-row tile, the adapter mask of the enclosing gemm_bn-wide
  // GEMM tile (see ShrinkParams::gmask); needs row_adapter and the 16-wide
  // tile prefix (tile_width_mask bit 0).
  uint64_t* gmask;
  int gemm_bn;
  int* clear_flags;             // or null: clear_count words zeroed first
  int clear_count;
};
bool small_permute_fits(int n, int E);
cudaError_t launch_small_permute(const FusedPermuteParams& p, cudaStream_t s);

// ------------------------------------------------------- expert GEMMs
// Swap-AB grouped GEMM: D[feature, token] = W_e[feature, :] . X[token, :]
// (+ LoRA expand as extra K blocks), accumulated in TMEM.
struct GemmParams {
  const int32_t* expert_offsets;  // [E + 1]
  const int32_t* tile_start;      // [E + 1] tile prefix for this tile width
  const int32_t* row_adapter;     // [n]
  int E;
  int K;                          // main reduction length (H or I)
  int rows_per_expert;            // rows of the weight per expert (2I or H)
  int gu_single_box;              // gate_up weight map is the 5-D one-box view
  int debug_stall_mma;            // test only: MMA role first waits on a barrier nobody signals
  int debug_hold_row;             // test only: the in-kernel shrink never counts permuted row 0
  int n_feat;                     // output features (I for gate_up, H for down)
  int feat_blocks;                // feature blocks per expert
  int num_adapters;               // 0 = no LoRA
  int rank;
  int64_t lb_row_stride_adapter;  // B-factor rows between adapters
  int64_t lb_row_stride_expert;   // B-factor rows between experts (0 = shared)
  __nv_bfloat16* out;             // [n, n_feat]
  int* status;
  uint64_t timeout_ns;
  // FP8 weights (e4m3, 128 x 128 blocks): w_scale [E, scale_nb, scale_kb]
  // float32, scale_nb = ceil(rows_per_expert / 128), scale_kb = ceil(K / 128).
  const float* w_scale;
  int scale_nb;
  int scale_kb;
  // 1 when the kernel launched just before this one is the shrink, which
  // calls griddepcontrol.wait before it lets dependents launch: the routing
  // tables are then complete when this grid starts, and the weight stream
  // may begin before this grid's own wait.  0: everything waits first.
  int tables_ready;
  // LoRA shrink inside the kernel (narrow tiles, one CTA per tile, rank <=
  // 32): before their first accumulator, the epilogue warps of every CTA
  // claim permuted rows one at a time from row_counter and write each
  // claimed row of su = bf16(s_a A[a, e] x) (the row's own adapter's
  // columns; zeros in the others), then count the row on its token tile's
  // flag; the producer waits until a tile's flag equals its row count before
  // the tile's first LoRA block.  Rows go only to CTAs that are running, so
  // every wait ends whatever number of CTAs the GPU holds at once.  The
  // flags and the counter are cleared by the permute of the same forward.
  int fuse_shrink;
  const __nv_bfloat16* sx;             // [n, K]: the token rows (xp or h)
  // Or also gather them: sx row p = gather_src row gather_map[p] / gather_div
  // (hidden rows by slot), written by the same in-kernel pass; the producer
  // then waits for a tile's flag before the tile's first K block.
  const __nv_bfloat16* gather_src;
  const int32_t* gather_map;
  int gather_div;
  const __nv_bfloat16* sa;             // A factors, rows of K elements
  int64_t sa_stride_adapter;           // elements between adapters
  int64_t sa_stride_expert;            // elements between experts
  __nv_bfloat16* su;                   // [n, num_adapters * rank]
  int* tile_flags;                     // [tiles of this width]
  int* row_counter;                    // next unclaimed permuted row (zeroed by the permute)
  // FP8 activations (fp8_gemm_kernel): token-row scales [n, ceil(K / 128)]
  // of the e4m3 token operand, and (gate_up) the float32 activation output
  // [n, n_feat] for the post-activation quant.
  const float* x_scale;
  float* out_f32;
  float sscale[MOE_MAX_ADAPTERS];      // per adapter
};
enum GemmMode { kGateUp = 0, kDown = 1 };
int gemm_stage_count(int bn, bool pair);
int gemm_ctas_per_sm(int bn);
size_t gemm_smem_bytes(int bn, bool pair);
// pair: clusters of two CTAs sharing one M = 256 MMA (cta_group::2).
bool gemm_use_pair(int bn);
// w8: FP8 block-scaled weights (tm_w is then a 1-byte view, p.w_scale set);
// one CTA per tile (no pair).  grid: CTAs of the persistent grid (pairs: at
// most as many clusters of two as can be resident).  tm_xs, tm_lus: the
// token maps of tm_x and tm_lu with boxes 32 rows high, for tiles of at most
// 32 rows per CTA (wide tiles only; otherwise pass tm_x and tm_lu).
cudaError_t launch_expert_gemm(int mode, int bn, bool pair, bool w8, const CUtensorMap& tm_w,
                               const CUtensorMap& tm_x, const CUtensorMap& tm_lb,
                               const CUtensorMap& tm_lu, const CUtensorMap& tm_xs,
                               const CUtensorMap& tm_lus, const GemmParams& p, int grid,
                               cudaStream_t s);

// ------------------------------------------------ FP8 activations (W8A8)
// Per row and group of kActGroup columns, float32: scale = max(amax, kActEps)
// / kE4m3Max, code = e4m3(x / scale) (nearest even, saturating).
constexpr int kActGroup = 128;
constexpr float kActEps = 1e-10f;
constexpr float kE4m3Max = 448.0f;
struct QuantParams {
  const void* x;                // source rows [*, K]: bf16 (x_f32 = 0) or float32
  int x_f32;
  const int32_t* row_map;       // or null: output row i reads source row row_map[i] / map_div
  int map_div;                  //   (row_map[i] < 0: a zero row)
  int rows;
  int K;                        // a multiple of 16
  uint8_t* codes;               // [rows, K]
  float* scales;                // [rows, ceil(K / kActGroup)]
  __nv_bfloat16* copy;          // or null: bf16 copy of each (float32) source row
};
cudaError_t launch_quant_groups(const QuantParams& p, cudaStream_t s);
// W8A8 expert GEMM: e4m3 weights (tm_w: 1-byte views with 128-byte swizzle,
// box {128, 16, 2, 4, 1} for gate_up, {128, 128} for down) and e4m3 token
// rows (tm_x, box {128, bn}); p.w_scale, p.x_scale set; gate_up writes the
// float32 activation to p.out_f32, down writes bf16 y to p.out.  bn <= 128.
int fp8_gemm_ctas_per_sm(int bn);
cudaError_t launch_fp8_gemm(int mode, int bn, const CUtensorMap& tm_w, const CUtensorMap& tm_x,
                            const CUtensorMap& tm_lb, const CUtensorMap& tm_lu, const GemmParams& p, int grid,
                            cudaStream_t s);

// --------------------------------------------------------------- finalize
cudaError_t launch_finalize(const __nv_bfloat16* y, const int32_t* e2p, const float* w, int T,
                            int top_k, int H, __nv_bfloat16* out, cudaStream_t s);

}  // namespace moe
