// C ABI of libmoelora: argument checks, workspace plan, TMA descriptors and
// the launch sequence of the routed MoE-LoRA forward.
//
// Stage order follows the single-stream pipeline of "[WIP][LoRA] BF16
// support for the experimental_sgl_trtllm MoE-LoRA path & lora
// expert_outer_shared" (yushengsu-thu/sglang#4), Flow 1(A):
//   routing -> permute -> gate_up LoRA shrink -> gate_up GEMM (+ expand,
//   + LoRA-aware SwiGLU) -> down LoRA shrink -> down GEMM (+ expand)
//   -> finalize.
// Everything is enqueued on the caller's stream; nothing is allocated and
// the host never waits, so the sequence can be captured into a CUDA graph.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/moe_lora.h"
#include "kernels.cuh"

namespace {

using moe::GemmParams;
using moe::PermuteParams;
using moe::ShrinkParams;

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------ TMA encoding
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D bf16 tensor [outer, inner] with row pitch row_bytes, box
// [box_outer, box_inner], 128-byte swizzle, zero fill out of bounds.
bool encode_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
               uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// N-D tensor (dims innermost first, strides in bytes for dims 1..rank-1),
// zero fill out of bounds: bf16 with 128-byte swizzle, or (fp8) bytes
// without swizzle (the W8A16 converter warps read them) or, with sw128, with
// 128-byte swizzle (the FP8 tensor-core operands).
bool encode_nd(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
               const uint64_t* strides, const uint32_t* box, bool fp8 = false, bool sw128 = false) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
    if (i + 1 < rank) st[i] = strides[i];
  }
  return fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank,
            const_cast<void*>(base), d, st, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE,
            (fp8 && !sw128) ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// w13 [E, 2I, H] seen so that one K block of feature block fb lands as
// 4 groups x (16 gate rows, 16 up rows).  With I % 16 == 0 a 5-D view
// {H, 16 rows, 2 halves, I/16 groups, E} does it in one box; otherwise a 3-D
// view {H, I, 2E} in four boxes of {64, 16, 2}.  Rows past I fall outside a
// dimension of either view and are zero-filled.
bool encode_w13(CUtensorMap* m, const void* w13, int H, int I, int E, bool* single_box,
                bool fp8 = false) {
  const uint64_t row = static_cast<uint64_t>(H) * (fp8 ? 1 : 2);
  if (I % 16 == 0) {
    const uint64_t dims[5] = {static_cast<uint64_t>(H), 16, 2, static_cast<uint64_t>(I / 16),
                              static_cast<uint64_t>(E)};
    const uint64_t strides[4] = {row, row * I, row * 16, row * 2 * I};
    const uint32_t box[5] = {64, 16, 2, 4, 1};
    if (encode_nd(m, w13, 5, dims, strides, box, fp8)) {
      *single_box = true;
      return true;
    }
  }
  const uint64_t dims[3] = {static_cast<uint64_t>(H), static_cast<uint64_t>(I),
                            2ull * static_cast<uint64_t>(E)};
  const uint64_t strides[2] = {row, row * I};
  const uint32_t box[3] = {64, 16, 2};
  *single_box = false;
  return encode_nd(m, w13, 3, dims, strides, box, fp8);
}

// ------------------------------------------------------------ workspace plan
bool sizes_ok(int T, int H, int I, int E, int top_k, int num_adapters, int rank) {
  return T >= 0 && H > 0 && I > 0 && E > 0 && top_k > 0 && num_adapters >= 0 && rank >= 0;
}

int limits_status(int H, int I, int E, int top_k, int num_adapters, int rank) {
  if (E > MOE_MAX_EXPERTS || top_k > MOE_MAX_TOP_K || rank > MOE_MAX_RANK ||
      num_adapters > MOE_MAX_ADAPTERS)
    return MOE_ERR_UNSUPPORTED;
  if (top_k > E) return MOE_ERR_SHAPE;
  if (H % 8 != 0 || I % 8 != 0) return MOE_ERR_ALIGN;
  if (rank % 8 != 0) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

void fill_plan(int T, int H, int I, int E, int top_k, int num_adapters, int rank,
               moe_lora_workspace_plan_t* pl) {
  const size_t n = static_cast<size_t>(T) * top_k;
  const size_t lora_cols = (num_adapters > 0 && rank > 0) ? static_cast<size_t>(num_adapters) * rank : 0;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align_up(bytes);
    return at;
  };
  std::memset(pl, 0, sizeof(*pl));
  pl->status = take(16);
  pl->topk_ids = take(n * 4);
  pl->topk_w = take(n * 4);
  pl->expert_offsets = take((static_cast<size_t>(E) + 1) * 4);
  pl->expanded_to_permuted = take(n * 4);
  pl->permuted_to_expanded = take(n * 4);
  pl->row_adapter = take(n * 4);
  pl->permute_scratch = take(moe::permute_scratch_bytes(static_cast<int>(n), E));
  // The permuted hidden rows are dead once the gate_up GEMM has run, so the
  // down GEMM's output reuses them; likewise the two LoRA operands.
  pl->permuted_hidden = take(n * static_cast<size_t>(H) * 2);
  pl->expert_out = pl->permuted_hidden;
  pl->lora_u = take(n * lora_cols * 2);
  pl->lora_v = pl->lora_u;
  pl->act = take(n * static_cast<size_t>(I) * 2);
  pl->total_bytes = o;
}

// FP8 activations: buffers after the bf16 plan (byte offsets from the
// workspace start).
struct Fp8ActPlan {
  size_t xq;     // uint8 [n, H]   quantized permuted hidden rows
  size_t xs;     // float [n, ceil(H / 128)]
  size_t hf;     // float [n, I]   activation before its quant
  size_t hq;     // uint8 [n, I]
  size_t hs;     // float [n, ceil(I / 128)]
  size_t total_bytes;
};

void fill_fp8_plan(int T, int H, int I, int top_k, size_t base, Fp8ActPlan* f) {
  const size_t n = static_cast<size_t>(T) * top_k;
  const size_t gh = (static_cast<size_t>(H) + moe::kActGroup - 1) / moe::kActGroup;
  const size_t gi = (static_cast<size_t>(I) + moe::kActGroup - 1) / moe::kActGroup;
  size_t o = base;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align_up(bytes);
    return at;
  };
  f->xq = take(n * H);
  f->xs = take(n * gh * 4);
  f->hf = take(n * I * 4);
  f->hq = take(n * I);
  f->hs = take(n * gi * 4);
  f->total_bytes = o;
}

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

size_t smem_per_sm() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess) return 0;
  return static_cast<size_t>(n);
}

// Token-tile width from the rows per expert.  avg assumes every expert is
// routed to; skewed routing touches fewer experts with more rows each, and a
// tile narrower than an expert's rows streams that expert's weights once per
// tile.  So: the power of two >= 2 avg, raised up to 64 (still two CTAs per
// SM) when 4 avg reaches it.
int auto_tile_n(int n_rows, int E) {
  const int touched = std::max(1, std::min(E, n_rows));
  const int avg = (n_rows + touched - 1) / touched;
  int bn = 16;
  while (bn < 256 && bn < 2 * avg) bn *= 2;
  while (bn < 64 && bn < 4 * avg) bn *= 2;
  return bn;
}

}  // namespace

namespace moe {

cudaError_t ensure_smem_limit(const void* func, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, int> done;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lock(mu);
  int& have = done[std::make_pair(dev, func)];
  if (have >= bytes) return cudaSuccess;
  err = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (err == cudaSuccess) have = bytes;
  return err;
}

}  // namespace moe

extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_NULL: return "MOE_ERR_NULL: a required pointer is NULL";
    case MOE_ERR_SHAPE: return "MOE_ERR_SHAPE: a size is out of range";
    case MOE_ERR_ALIGN: return "MOE_ERR_ALIGN: pointer, size or stride breaks the 16-byte rule";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: outside the supported limits";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace NULL, misaligned or too small";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call failed";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT: a device pipeline wait timed out";
    case MOE_ERR_BAD_MAPPING: return "MOE_ERR_BAD_MAPPING: token_lora_mapping outside [-1, A)";
    case MOE_ERR_BAD_EXPERT_ID: return "MOE_ERR_BAD_EXPERT_ID: a topk id outside [-1, E)";
    default: return "unknown moe status";
  }
}

int moe_lora_abi_version(void) { return MOE_LORA_ABI_VERSION; }

int moe_route_topk(const float* logits, int T, int E, int top_k, int32_t* topk_ids, float* topk_w,
                   moe_stream_t stream) {
  if (T < 0 || E <= 0 || top_k <= 0) return MOE_ERR_SHAPE;
  if (E > MOE_MAX_EXPERTS || top_k > MOE_MAX_TOP_K) return MOE_ERR_UNSUPPORTED;
  if (top_k > E) return MOE_ERR_SHAPE;
  if (T == 0) return MOE_OK;
  if (logits == nullptr || topk_ids == nullptr || topk_w == nullptr) return MOE_ERR_NULL;
  (void)cudaGetLastError();  // launch checks below must not report an earlier, unrelated error
  return cuda_status(moe::launch_route_topk(logits, T, E, top_k, topk_ids, topk_w, stream));
}

size_t moe_permute_workspace_size(int T, int top_k, int E) {
  if (T < 0 || top_k <= 0 || E <= 0) return 0;
  return align_up(16) + moe::permute_scratch_bytes(T * top_k, E);
}

int moe_permute(const int32_t* topk_ids, int T, int top_k, int E, const void* hidden, int H,
                int32_t* expert_offsets, int32_t* expanded_to_permuted,
                int32_t* permuted_to_expanded, void* permuted_hidden, void* ws, size_t ws_bytes,
                moe_stream_t stream) {
  if (T < 0 || E <= 0 || top_k <= 0) return MOE_ERR_SHAPE;
  if (E > MOE_MAX_EXPERTS || top_k > MOE_MAX_TOP_K) return MOE_ERR_UNSUPPORTED;
  if (expert_offsets == nullptr || ws == nullptr) return MOE_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0 ||
      ws_bytes < moe_permute_workspace_size(T, top_k, E))
    return MOE_ERR_WORKSPACE;
  const bool gather = hidden != nullptr && permuted_hidden != nullptr;
  if (gather && (H <= 0 || H % 8 != 0 || !aligned16(hidden) || !aligned16(permuted_hidden)))
    return MOE_ERR_ALIGN;
  int* status = static_cast<int*>(ws);
  (void)cudaGetLastError();  // launch checks below must not report an earlier, unrelated error
  if (cudaMemsetAsync(status, 0, 16, stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (T == 0) return cuda_status(cudaMemsetAsync(expert_offsets, 0, (E + 1) * sizeof(int32_t), stream));
  if (topk_ids == nullptr || expanded_to_permuted == nullptr || permuted_to_expanded == nullptr)
    return MOE_ERR_NULL;
  const int n = T * top_k;
  uint8_t* scratch = static_cast<uint8_t*>(ws) + align_up(16);
  PermuteParams p{};
  p.topk_ids = topk_ids;
  p.n = n;
  p.top_k = top_k;
  p.E = E;
  p.H = H;
  p.hidden = gather ? static_cast<const __nv_bfloat16*>(hidden) : nullptr;
  p.permuted = gather ? static_cast<__nv_bfloat16*>(permuted_hidden) : nullptr;
  p.expert_offsets = expert_offsets;
  p.e2p = expanded_to_permuted;
  p.p2e = permuted_to_expanded;
  p.chunk_counts = reinterpret_cast<int32_t*>(scratch);
  p.tile_start = nullptr;
  p.status = status;
  return cuda_status(moe::launch_permute(p, stream));
}

int moe_lora_workspace_plan(int T, int H, int I, int E, int top_k, int num_adapters, int rank,
                            moe_lora_workspace_plan_t* plan) {
  if (plan == nullptr) return MOE_ERR_NULL;
  if (!sizes_ok(T, H, I, E, top_k, num_adapters, rank)) return MOE_ERR_SHAPE;
  const int st = limits_status(H, I, E, top_k, num_adapters, rank);
  if (st != MOE_OK) return st;
  fill_plan(T, H, I, E, top_k, num_adapters, rank, plan);
  return MOE_OK;
}

size_t moe_lora_workspace_size(int T, int H, int I, int E, int top_k, int num_adapters, int rank) {
  moe_lora_workspace_plan_t pl;
  if (moe_lora_workspace_plan(T, H, I, E, top_k, num_adapters, rank, &pl) != MOE_OK) return 0;
  return pl.total_bytes;
}

size_t moe_lora_workspace_size_ex(int T, int H, int I, int E, int top_k, int num_adapters, int rank,
                                  int activation_format) {
  const size_t base = moe_lora_workspace_size(T, H, I, E, top_k, num_adapters, rank);
  if (base == 0 || activation_format == MOE_ACT_BF16) return base;
  if (activation_format != MOE_ACT_FP8_E4M3_G128) return 0;
  Fp8ActPlan f;
  fill_fp8_plan(T, H, I, top_k, base, &f);
  return f.total_bytes;
}

int moe_per_token_group_quant_fp8(const void* x, int x_is_f32, int rows, int K, const int32_t* row_map,
                                  int map_div, uint8_t* codes, float* scales, moe_stream_t stream) {
  if (rows < 0 || K <= 0 || map_div < 1 || (x_is_f32 != 0 && x_is_f32 != 1)) return MOE_ERR_SHAPE;
  if (K % 16 != 0) return MOE_ERR_ALIGN;
  if (rows == 0) return MOE_OK;
  if (x == nullptr || codes == nullptr || scales == nullptr) return MOE_ERR_NULL;
  if (!aligned16(x) || !aligned16(codes) || (reinterpret_cast<uintptr_t>(scales) & 3) != 0)
    return MOE_ERR_ALIGN;
  (void)cudaGetLastError();  // launch checks below must not report an earlier, unrelated error
  moe::QuantParams q{};
  q.x = x;
  q.x_f32 = x_is_f32;
  q.row_map = row_map;
  q.map_div = map_div;
  q.rows = rows;
  q.K = K;
  q.codes = codes;
  q.scales = scales;
  q.copy = nullptr;
  return cuda_status(moe::launch_quant_groups(q, stream));
}

int moe_read_device_status(const void* workspace, moe_stream_t stream) {
  if (workspace == nullptr) return MOE_ERR_NULL;
  int host[4] = {0, 0, 0, 0};
  if (cudaMemcpyAsync(host, workspace, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  return host[0];
}

int moe_lora_forward(const moe_lora_args_t* a, moe_stream_t stream) {
  if (a == nullptr) return MOE_ERR_NULL;
  // Structures from before the expert-parallel fields end at adapter_scaling,
  // those from before the weight-format fields at num_router_experts, those
  // from before the tuning and side-stream fields at w2_scale.
  constexpr size_t kSizeNoShard = offsetof(moe_lora_args_t, local_expert_offset);
  constexpr size_t kSizeNoFormat = offsetof(moe_lora_args_t, weight_format);
  constexpr size_t kSizeNoTuning = offsetof(moe_lora_args_t, tuning);
  constexpr size_t kSizeNoActFormat = offsetof(moe_lora_args_t, activation_format);
  if (a->struct_size < kSizeNoShard) return MOE_ERR_UNSUPPORTED;
  const bool has_shard = a->struct_size >= kSizeNoFormat;
  const bool has_format = a->struct_size >= kSizeNoTuning;
  const bool has_tuning = a->struct_size >= kSizeNoActFormat;
  const bool has_act = a->struct_size >= sizeof(moe_lora_args_t);
  moe_lora_tuning_t tune;
  std::memset(&tune, 0, sizeof(tune));
  if (has_tuning) tune = a->tuning;
  if (tune.cta_pairs < 0 || tune.cta_pairs > 2 || tune.shrink_kernel < 0 || tune.shrink_kernel > 2 ||
      tune.shrink_in_gemm < 0 || tune.shrink_in_gemm > 2 || tune.gemm_max_ctas < 0)
    return MOE_ERR_UNSUPPORTED;
  cudaStream_t side = has_tuning ? reinterpret_cast<cudaStream_t>(a->side_stream) : nullptr;
  if (side != nullptr && (a->side_events[0] == nullptr || a->side_events[1] == nullptr))
    return MOE_ERR_NULL;
  const int wfmt = has_format ? a->weight_format : MOE_WEIGHTS_BF16;
  const bool w8 = wfmt == MOE_WEIGHTS_FP8_E4M3_B128;
  const int T = a->T, H = a->H, I = a->I, E = a->E, K = a->top_k;
  const int shard_off = has_shard ? a->local_expert_offset : 0;
  const int R = (has_shard && a->num_router_experts != 0) ? a->num_router_experts : E;
  if (!sizes_ok(T, H, I, E, K, a->num_adapters, a->rank)) return MOE_ERR_SHAPE;
  int st = limits_status(H, I, E, K, a->num_adapters, a->rank);
  if (st != MOE_OK) return st;
  if (R < E || R > MOE_MAX_EXPERTS || K > R || shard_off < 0 || shard_off > R - E) return MOE_ERR_SHAPE;
  if (wfmt != MOE_WEIGHTS_BF16 && wfmt != MOE_WEIGHTS_FP8_E4M3_B128) return MOE_ERR_UNSUPPORTED;
  const int afmt = has_act ? a->activation_format : MOE_ACT_BF16;
  if (afmt != MOE_ACT_BF16 && afmt != MOE_ACT_FP8_E4M3_G128) return MOE_ERR_UNSUPPORTED;
  const bool a8 = afmt == MOE_ACT_FP8_E4M3_G128;  // W8A8: FP8 activations need FP8 weights
  if (a8 && !w8) return MOE_ERR_UNSUPPORTED;
  // FP8 weight rows are 1 byte per element: TMA wants 16-byte row pitches.
  if (w8 && (H % 16 != 0 || I % 16 != 0)) return MOE_ERR_ALIGN;
  const bool lora = a->num_adapters > 0 && a->rank > 0;
  const int A = lora ? a->num_adapters : 0;
  const int r = lora ? a->rank : 0;
  if (a->tile_n != 0 && a->tile_n != 16 && a->tile_n != 32 && a->tile_n != 64 && a->tile_n != 128 &&
      a->tile_n != 256)
    return MOE_ERR_UNSUPPORTED;
  if (a->wait_timeout_ms < 0) return MOE_ERR_SHAPE;
  (void)cudaGetLastError();  // launch checks below must not report an earlier, unrelated error

  struct CUevent_st* const* ev = a->stage_events;
  int ev_next = 0;
  auto mark = [&]() -> bool {
    if (ev == nullptr || ev_next >= MOE_NUM_STAGE_EVENTS) return true;
    return cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev[ev_next++]), stream) == cudaSuccess;
  };
  auto finish_marks = [&]() -> bool {
    while (ev != nullptr && ev_next < MOE_NUM_STAGE_EVENTS)
      if (!mark()) return false;
    return true;
  };
  if (T == 0) {  // nothing to compute; tensor pointers may be NULL
    if (a->workspace != nullptr) {
      if ((reinterpret_cast<uintptr_t>(a->workspace) & (kAlign - 1)) != 0) return MOE_ERR_WORKSPACE;
      if (cudaMemsetAsync(a->workspace, 0, 16, stream) != cudaSuccess) return MOE_ERR_CUDA;
    }
    return finish_marks() ? MOE_OK : MOE_ERR_CUDA;
  }

  if (a->hidden == nullptr || a->w13 == nullptr || a->w2 == nullptr ||
      a->router_logits == nullptr || a->out == nullptr || a->workspace == nullptr)
    return MOE_ERR_NULL;
  if (!aligned16(a->hidden) || !aligned16(a->w13) || !aligned16(a->w2) || !aligned16(a->out))
    return MOE_ERR_ALIGN;
  if (w8 && (a->w13_scale == nullptr || a->w2_scale == nullptr)) return MOE_ERR_NULL;
  if (w8 && ((reinterpret_cast<uintptr_t>(a->w13_scale) | reinterpret_cast<uintptr_t>(a->w2_scale)) & 3))
    return MOE_ERR_ALIGN;
  if (lora) {
    if (a->token_lora_mapping == nullptr || a->gate_up.A == nullptr || a->gate_up.B == nullptr ||
        a->down.A == nullptr || a->down.B == nullptr)
      return MOE_ERR_NULL;
    const moe_lora_factors_t* fs[2] = {&a->gate_up, &a->down};
    for (const moe_lora_factors_t* f : fs) {
      if (!aligned16(f->A) || !aligned16(f->B)) return MOE_ERR_ALIGN;
      if (f->a_stride_adapter < 0 || f->a_stride_expert < 0 || f->b_stride_adapter < 0 ||
          f->b_stride_expert < 0)
        return MOE_ERR_SHAPE;
      if (f->a_stride_adapter % 8 || f->a_stride_expert % 8 || f->b_stride_adapter % 8 ||
          f->b_stride_expert % 8)
        return MOE_ERR_ALIGN;
      if (f->b_stride_adapter % r || f->b_stride_expert % r) return MOE_ERR_ALIGN;
    }
  }
  if ((reinterpret_cast<uintptr_t>(a->workspace) & (kAlign - 1)) != 0) return MOE_ERR_WORKSPACE;
  moe_lora_workspace_plan_t pl;
  fill_plan(T, H, I, E, K, A, r, &pl);
  Fp8ActPlan f8{};
  if (a8) fill_fp8_plan(T, H, I, K, pl.total_bytes, &f8);
  if (a->workspace_bytes < (a8 ? f8.total_bytes : pl.total_bytes)) return MOE_ERR_WORKSPACE;
  const int64_t n = static_cast<int64_t>(T) * K;
  if (n >= (int64_t(1) << 31) || static_cast<int64_t>(E) * 2 * I >= (int64_t(1) << 31) ||
      static_cast<int64_t>(E) * H >= (int64_t(1) << 31))
    return MOE_ERR_UNSUPPORTED;

  uint8_t* ws = static_cast<uint8_t*>(a->workspace);
  int* status = reinterpret_cast<int*>(ws + pl.status);
  // The one-CTA permute clears the status word itself; otherwise clear it here.
  const bool small_permute = moe::small_permute_fits(static_cast<int>(n), E);
  const bool fuse_route = small_permute && T <= 128;
  // Past the one-CTA permute: routing and the permutation in two kernels
  // (they clear the status word themselves), else routing + three kernels.
  const bool route_permute = !small_permute && moe::route_permute_fits(T, K, E);
  if (!small_permute && !route_permute && cudaMemsetAsync(status, 0, 16, stream) != cudaSuccess)
    return MOE_ERR_CUDA;

  int32_t* topk_ids = a->topk_ids_out ? a->topk_ids_out : reinterpret_cast<int32_t*>(ws + pl.topk_ids);
  float* topk_w = a->topk_w_out ? a->topk_w_out : reinterpret_cast<float*>(ws + pl.topk_w);
  int32_t* e2p = a->expanded_to_permuted_out ? a->expanded_to_permuted_out
                                             : reinterpret_cast<int32_t*>(ws + pl.expanded_to_permuted);
  int32_t* offsets = reinterpret_cast<int32_t*>(ws + pl.expert_offsets);
  int32_t* p2e = reinterpret_cast<int32_t*>(ws + pl.permuted_to_expanded);
  int32_t* row_adapter = reinterpret_cast<int32_t*>(ws + pl.row_adapter);
  int32_t* chunk_counts = reinterpret_cast<int32_t*>(ws + pl.permute_scratch);
  const size_t nchunks = (static_cast<size_t>(n) + moe::kPermuteChunk - 1) / moe::kPermuteChunk;
  int32_t* tile_start = reinterpret_cast<int32_t*>(
      ws + pl.permute_scratch + align_up(nchunks * E * sizeof(int32_t)));
  uint64_t* gmask = reinterpret_cast<uint64_t*>(
      reinterpret_cast<uint8_t*>(tile_start) + align_up(moe::kNumTileWidths * (E + 1) * sizeof(int32_t)));
  int* flags_gu = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(gmask) + moe::gmask_bytes(static_cast<int>(n), E));
  int* flags_dn = flags_gu + moe::shrink_flag_words(static_cast<int>(n), E);
  __nv_bfloat16* xp = reinterpret_cast<__nv_bfloat16*>(ws + pl.permuted_hidden);
  __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(ws + pl.expert_out);
  __nv_bfloat16* U = reinterpret_cast<__nv_bfloat16*>(ws + pl.lora_u);
  __nv_bfloat16* V = reinterpret_cast<__nv_bfloat16*>(ws + pl.lora_v);
  __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(ws + pl.act);

  // Rows this shard expects (all of them without sharding): the tile width
  // and the shrink variant follow the rows per local expert.
  const int64_t n_local = n * E / R;
  int bn = a->tile_n ? a->tile_n : auto_tile_n(static_cast<int>(n_local), E);
  if (a8 && bn > 128) bn = 128;  // the W8A8 epilogue holds a tile row in registers
  // CTA pairs sharing one M = 256 MMA (cta_group::2) for wide tiles; each CTA
  // of a pair loads bn / 2 token rows.  FP8 weights run one CTA per tile.
  bool pair = moe::gemm_use_pair(bn);
  if (tune.cta_pairs == 1) pair = false;
  if (tune.cta_pairs == 2) pair = bn >= 128;
  if (w8) pair = false;
  const int sms = num_sms();
  if (sms <= 0) return MOE_ERR_CUDA;
  // Many rows, or a large rank with several rows per expert (the factor is
  // then read once per row tile instead of once per 16 rows): row tiles
  // streamed through a cp.async pipeline.  The per-token mode keeps the
  // 16-row kernel.
  bool row_blocks = n_local > 16 * static_cast<int64_t>(sms) ||
                    (r >= 64 && n_local >= 8 * std::min<int64_t>(E, n_local));
  if (tune.shrink_kernel != 0) row_blocks = tune.shrink_kernel == 2;
  // Decode-sized tiles: the LoRA shrinks run inside the expert GEMMs (their
  // epilogue warps are idle until the first accumulator is ready), so no
  // shrink kernel sits between the permute and the gate_up GEMM or between
  // the GEMMs.  Needs the one-CTA permute (it clears the tile flags and the
  // row counters), one CTA per 16-wide tile, rank <= 32 and per-expert
  // gate_up A factors.  The two-stream schedule keeps the shrinks in kernels
  // of their own.
  const bool fuse_shrink = lora && small_permute && bn == 16 && !pair && r <= 32 && !row_blocks &&
                           a->gate_up.a_stride_expert != 0 && tune.shrink_in_gemm != 1 &&
                           side == nullptr;
  // With bf16 activations the row gather runs first as a small kernel of its
  // own, which lets the gate_up GEMM launch as soon as the permute is done and
  // stream weights before the rows are in; only its LoRA blocks then wait for
  // the in-kernel shrink.  (Tuning 2: the gather inside the gate_up GEMM too,
  // whose first loads then wait for the tile's rows.)  W8A8 gathers in its
  // row quantizer.
  const bool gather_kernel = fuse_shrink && !a8 && tune.shrink_in_gemm != 2;
  const bool two_streams = lora && side != nullptr;
  // Persistent grid of the expert GEMMs.
  int gemm_grid = sms * (a8 ? moe::fp8_gemm_ctas_per_sm(bn) : moe::gemm_ctas_per_sm(bn));
  if (tune.gemm_max_ctas > 0) gemm_grid = std::min(gemm_grid, std::max(tune.gemm_max_ctas, pair ? 2 : 1));
  const uint64_t timeout_ns =
      static_cast<uint64_t>(a->wait_timeout_ms ? a->wait_timeout_ms : 2000) * 1000000ull;

  // TMA descriptors (host-encoded, passed by value as kernel parameters).
  CUtensorMap tm_w13, tm_w2, tm_xp, tm_h, tm_bgu, tm_bdn, tm_u, tm_v;
  bool gu_single_box = false;
  const uint64_t w2_dims[2] = {static_cast<uint64_t>(I), static_cast<uint64_t>(E) * H};
  const uint64_t w2_row[1] = {static_cast<uint64_t>(I) * (w8 ? 1 : 2)};
  const uint32_t w2_box[2] = {64, 128};
  const int tok_box = pair ? bn / 2 : bn;  // token rows per CTA and stage
  bool enc = encode_w13(&tm_w13, a->w13, H, I, E, &gu_single_box, w8) &&
             encode_nd(&tm_w2, a->w2, 2, w2_dims, w2_row, w2_box, w8) &&
             encode_2d(&tm_xp, xp, H, n, H * 2ull, 64, tok_box) &&
             encode_2d(&tm_h, h, I, n, I * 2ull, 64, tok_box);
  int64_t gu_rs_a = 0, gu_rs_e = 0, dn_rs_a = 0, dn_rs_e = 0;
  if (enc && lora) {
    gu_rs_a = a->gate_up.b_stride_adapter / r;
    gu_rs_e = a->gate_up.b_stride_expert / r;
    dn_rs_a = a->down.b_stride_adapter / r;
    dn_rs_e = a->down.b_stride_expert / r;
    const uint64_t gu_rows = (A - 1) * gu_rs_a + (E - 1) * gu_rs_e + 2ull * I;
    const uint64_t dn_rows = (A - 1) * dn_rs_a + (E - 1) * dn_rs_e + static_cast<uint64_t>(H);
    if (gu_rows >= (1ull << 31) || dn_rows >= (1ull << 31)) return MOE_ERR_UNSUPPORTED;
    enc = encode_2d(&tm_bgu, a->gate_up.B, r, gu_rows, r * 2ull, 64, 16) &&
          encode_2d(&tm_bdn, a->down.B, r, dn_rows, r * 2ull, 64, 128) &&
          encode_2d(&tm_u, U, static_cast<uint64_t>(A) * r, n, A * r * 2ull, 64, tok_box) &&
          encode_2d(&tm_v, V, static_cast<uint64_t>(A) * r, n, A * r * 2ull, 64, tok_box);
  } else {
    tm_bgu = tm_w13;
    tm_bdn = tm_w2;
    tm_u = tm_xp;
    tm_v = tm_h;
  }
  // W8A8: e4m3 weights and token rows, 128-byte rows with 128-byte swizzle
  uint8_t* xq = a8 ? ws + f8.xq : nullptr;
  float* xs = a8 ? reinterpret_cast<float*>(ws + f8.xs) : nullptr;
  float* hf = a8 ? reinterpret_cast<float*>(ws + f8.hf) : nullptr;
  uint8_t* hq = a8 ? ws + f8.hq : nullptr;
  float* hs = a8 ? reinterpret_cast<float*>(ws + f8.hs) : nullptr;
  if (enc && a8) {
    const uint64_t row = static_cast<uint64_t>(H);
    const uint64_t d13[5] = {static_cast<uint64_t>(H), 16, 2, static_cast<uint64_t>(I / 16),
                             static_cast<uint64_t>(E)};
    const uint64_t s13[4] = {row, row * I, row * 16, row * 2 * I};
    const uint32_t b13[5] = {128, 16, 2, 4, 1};
    const uint64_t d2[2] = {static_cast<uint64_t>(I), static_cast<uint64_t>(E) * H};
    const uint64_t s2[1] = {static_cast<uint64_t>(I)};
    const uint32_t b2[2] = {128, 128};
    const uint64_t dxq[2] = {static_cast<uint64_t>(H), static_cast<uint64_t>(n)};
    const uint64_t sxq[1] = {static_cast<uint64_t>(H)};
    const uint64_t dhq[2] = {static_cast<uint64_t>(I), static_cast<uint64_t>(n)};
    const uint64_t shq[1] = {static_cast<uint64_t>(I)};
    const uint32_t btok[2] = {128, static_cast<uint32_t>(bn)};
    enc = encode_nd(&tm_w13, a->w13, 5, d13, s13, b13, true, true) &&
          encode_nd(&tm_w2, a->w2, 2, d2, s2, b2, true, true) &&
          encode_nd(&tm_xp, xq, 2, dxq, sxq, btok, true, true) &&
          encode_nd(&tm_h, hq, 2, dhq, shq, btok, true, true);
  }
  // Wide bf16 tiles: token maps with 32-row boxes for tiles of few rows
  CUtensorMap tm_xp_s = tm_xp, tm_h_s = tm_h, tm_u_s = tm_u, tm_v_s = tm_v;
  if (enc && tok_box > 32 && !w8) {
    enc = encode_2d(&tm_xp_s, xp, H, n, H * 2ull, 64, 32) && encode_2d(&tm_h_s, h, I, n, I * 2ull, 64, 32);
    if (enc && lora)
      enc = encode_2d(&tm_u_s, U, static_cast<uint64_t>(A) * r, n, A * r * 2ull, 64, 32) &&
            encode_2d(&tm_v_s, V, static_cast<uint64_t>(A) * r, n, A * r * 2ull, 64, 32);
  }
  if (!enc) return MOE_ERR_CUDA;

  if (!mark()) return MOE_ERR_CUDA;
  // 1-2. routing and permutation (one CTA when it fits)
  moe::FusedPermuteParams fp{};
  fp.logits = fuse_route ? a->router_logits : nullptr;
  fp.topk_ids = topk_ids;
  fp.topk_w = topk_w;
  fp.T = T;
  fp.top_k = K;
  fp.E = E;
  fp.mapping = lora ? a->token_lora_mapping : nullptr;
  fp.num_adapters = A;
  fp.row_adapter = row_adapter;
  fp.expert_offsets = offsets;
  fp.e2p = e2p;
  fp.p2e = p2e;
  fp.tile_start = tile_start;
  // widths read later: the 16-row shrink, the row-block shrink, the GEMM
  fp.tile_width_mask = (1u << moe::tile_width_index(16)) |
                       (1u << moe::tile_width_index(moe::rows_shrink_tile())) |
                       (1u << moe::tile_width_index(bn));
  fp.status = status;
  // Per 16-row tile, the adapters of its GEMM tile: lets the 16-row shrink
  // skip (tile, adapter) pairs without work.
  fp.gmask = (lora && small_permute && !fuse_shrink) ? gmask : nullptr;
  fp.gemm_bn = bn;
  fp.clear_flags = fuse_shrink ? flags_gu : nullptr;
  fp.clear_count = fuse_shrink ? static_cast<int>(2 * moe::shrink_flag_words(static_cast<int>(n), E)) : 0;
  fp.id_offset = shard_off;
  fp.id_limit = R;
  if (!fuse_route && !route_permute &&
      moe::launch_route_topk(a->router_logits, T, R, K, topk_ids, topk_w, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (!mark()) return MOE_ERR_CUDA;
  if (small_permute) {
    if (moe::launch_small_permute(fp, stream) != cudaSuccess) return MOE_ERR_CUDA;
  } else if (route_permute) {
    moe::RoutePermuteParams rp{};
    rp.logits = a->router_logits;
    rp.T = T;
    rp.top_k = K;
    rp.E = E;
    rp.id_offset = shard_off;
    rp.id_limit = R;
    rp.topk_ids = topk_ids;
    rp.topk_w = topk_w;
    rp.mapping = fp.mapping;
    rp.num_adapters = A;
    rp.row_adapter = row_adapter;
    rp.expert_offsets = offsets;
    rp.e2p = e2p;
    rp.p2e = p2e;
    rp.chunk_counts = chunk_counts;
    rp.tile_start = tile_start;
    rp.tile_width_mask = fp.tile_width_mask;
    rp.status = status;
    if (moe::launch_route_permute(rp, stream) != cudaSuccess) return MOE_ERR_CUDA;
  } else {
    PermuteParams pp{};
    pp.topk_ids = topk_ids;
    pp.n = static_cast<int>(n);
    pp.top_k = K;
    pp.E = E;
    pp.H = H;
    pp.hidden = nullptr;  // rows are gathered by the next kernel
    pp.permuted = nullptr;
    pp.mapping = fp.mapping;
    pp.num_adapters = A;
    pp.row_adapter = row_adapter;
    pp.expert_offsets = offsets;
    pp.e2p = e2p;
    pp.p2e = p2e;
    pp.chunk_counts = chunk_counts;
    pp.tile_start = tile_start;
    pp.status = status;
    pp.id_offset = shard_off;
    pp.id_limit = R;
    if (moe::launch_permute(pp, stream) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (!mark()) return MOE_ERR_CUDA;
  // 3. row gather + gate_up LoRA shrink: xp = hidden[t(p)], U = s * A_gu x
  //    (one-hot per adapter).  Few tiles (decode): one phase per CTA; many
  //    tiles: smaller phases so that several CTAs share an SM.
  const size_t shrink_budget = n_local <= 16 * static_cast<int64_t>(sms) ? 200 * 1024 : 72 * 1024;
  ShrinkParams sp{};
  sp.X = static_cast<const __nv_bfloat16*>(a->hidden);
  sp.p2e = p2e;
  sp.top_k = K;
  sp.K = H;
  sp.gathered = xp;
  sp.A = lora ? static_cast<const __nv_bfloat16*>(a->gate_up.A) : nullptr;
  sp.a_stride_adapter = lora ? a->gate_up.a_stride_adapter : 0;
  sp.a_stride_expert = lora ? a->gate_up.a_stride_expert : 0;
  sp.row_adapter = row_adapter;
  sp.expert_offsets = offsets;
  sp.tile_start16 = tile_start + moe::tile_width_index(16) * (E + 1);
  sp.E = E;
  sp.num_adapters = A;
  sp.rank = r;
  for (int i = 0; i < MOE_MAX_ADAPTERS; ++i)
    sp.scaling[i] = (a->adapter_scaling != nullptr && i < A) ? a->adapter_scaling[i] : a->scaling;
  sp.U = (lora && !fuse_shrink) ? U : nullptr;  // fused: the gather alone
  sp.status = status;
  sp.timeout_ns = timeout_ns;
  // A shared gate_up A factor makes u a function of the token alone.
  sp.per_token = (lora && a->gate_up.a_stride_expert == 0) ? 1 : 0;
  sp.T = T;
  // Per token: phases sized so that the whole grid is resident in one wave
  // (more phases cost less than a second wave of CTAs).
  sp.kc = moe::shrink_chunk(H, moe::gather_shrink_cta_rank(sp),
                            sp.per_token ? moe::per_token_shrink_budget(sp, sms, smem_per_sm()) : shrink_budget);
  sp.e2p = e2p;
  sp.mapping = lora ? a->token_lora_mapping : nullptr;
  sp.tile_start_rows = tile_start + moe::tile_width_index(moe::rows_shrink_tile()) * (E + 1);
  sp.gmask = fp.gmask;
  if (a8) {
    // W8A8: the permuted rows go out quantized (no bf16 copy); the gate_up
    // shrink reads the bf16 hidden rows through the permutation.
    moe::QuantParams qp{};
    qp.x = a->hidden;
    qp.x_f32 = 0;
    qp.row_map = p2e;
    qp.map_div = K;
    qp.rows = static_cast<int>(n);
    qp.K = H;
    qp.codes = xq;
    qp.scales = xs;
    if (moe::launch_quant_groups(qp, stream) != cudaSuccess) return MOE_ERR_CUDA;
    sp.gathered = nullptr;
  }
  auto launch_shrink = [&](const ShrinkParams& q, cudaStream_t s) {
    return row_blocks && !q.per_token ? moe::launch_rows_shrink(q, static_cast<int>(n), s)
                                      : moe::launch_gather_shrink(q, static_cast<int>(n), s);
  };
  if (two_streams) {
    // Fork after the permute: the shrink (U only) on the side stream, the
    // row gather (xp only) here; join before the gate_up GEMM.
    cudaEvent_t fork = reinterpret_cast<cudaEvent_t>(a->side_events[0]);
    cudaEvent_t join = reinterpret_cast<cudaEvent_t>(a->side_events[1]);
    ShrinkParams sq = sp;
    sq.gathered = nullptr;
    sp.U = nullptr;
    if (cudaEventRecord(fork, stream) != cudaSuccess || cudaStreamWaitEvent(side, fork, 0) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (launch_shrink(sq, side) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaEventRecord(join, side) != cudaSuccess) return MOE_ERR_CUDA;
    if (launch_shrink(sp, stream) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamWaitEvent(stream, join, 0) != cudaSuccess) return MOE_ERR_CUDA;
  } else if (!fuse_shrink && (!a8 || lora) &&  // fused: the shrink runs inside the gate_up GEMM
             launch_shrink(sp, stream) != cudaSuccess) {
    return MOE_ERR_CUDA;
  } else if (gather_kernel &&  // fused: the row gather alone (sp.U is null)
             moe::launch_gather_shrink(sp, static_cast<int>(n), stream) != cudaSuccess) {
    return MOE_ERR_CUDA;
  }
  if (!mark()) return MOE_ERR_CUDA;
  // 4. gate_up GEMM + LoRA expand + SwiGLU -> h
  GemmParams gp{};
  gp.expert_offsets = offsets;
  gp.tile_start = tile_start + moe::tile_width_index(bn) * (E + 1);
  gp.row_adapter = row_adapter;
  gp.E = E;
  gp.K = H;
  gp.rows_per_expert = 2 * I;
  gp.gu_single_box = gu_single_box ? 1 : 0;
  gp.debug_stall_mma = (a->debug_flags & MOE_DEBUG_STALL_GATE_UP_MMA) ? 1 : 0;
  gp.debug_hold_row = (a->debug_flags & MOE_DEBUG_HOLD_SHRINK_ROW) ? 1 : 0;
  gp.n_feat = I;
  gp.feat_blocks = (I + 63) / 64;
  gp.num_adapters = A;
  gp.rank = r;
  gp.lb_row_stride_adapter = gu_rs_a;
  gp.lb_row_stride_expert = gu_rs_e;
  gp.out = h;
  gp.status = status;
  gp.timeout_ns = timeout_ns;
  // Launched right after the gate_up shrink or the row gather (n > 0 here),
  // which wait for the permute before they let this grid launch, or (gather
  // inside the GEMM) right after the permute, whose tables may still be in
  // flight.  W8A8 with the in-kernel shrink also waits first (fp8_gemm reads
  // no tables_ready): weights streamed before its row quantizer completes
  // slowed the in-kernel shrink that its first LoRA blocks wait for.
  gp.tables_ready = (fuse_shrink && !gather_kernel) ? 0 : 1;
  gp.w_scale = w8 ? a->w13_scale : nullptr;
  gp.scale_nb = (2 * I + 127) / 128;
  gp.scale_kb = (H + 127) / 128;
  gp.fuse_shrink = fuse_shrink ? 1 : 0;
  gp.x_scale = xs;
  gp.out_f32 = hf;
  if (fuse_shrink) {
    gp.sx = a8 ? nullptr : xp;  // W8A8: the GEMM reads the quantized rows; no bf16 copy
    gp.gather_src = gather_kernel ? nullptr : static_cast<const __nv_bfloat16*>(a->hidden);
    gp.gather_map = p2e;
    gp.gather_div = K;
    gp.sa = static_cast<const __nv_bfloat16*>(a->gate_up.A);
    gp.sa_stride_adapter = a->gate_up.a_stride_adapter;
    gp.sa_stride_expert = a->gate_up.a_stride_expert;
    gp.su = U;
    gp.tile_flags = flags_gu;
    gp.row_counter = flags_gu + moe::shrink_flag_words(static_cast<int>(n), E) - 1;
    for (int i = 0; i < MOE_MAX_ADAPTERS; ++i) gp.sscale[i] = sp.scaling[i];
  }
  if ((a8 ? moe::launch_fp8_gemm(moe::kGateUp, bn, tm_w13, tm_xp, tm_bgu, tm_u, gp, gemm_grid, stream)
          : moe::launch_expert_gemm(moe::kGateUp, bn, pair, w8, tm_w13, tm_xp, tm_bgu, tm_u, tm_xp_s, tm_u_s, gp,
                                    gemm_grid, stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (!mark()) return MOE_ERR_CUDA;
  if (a8) {
    // post-activation quant from the float32 activation, plus the bf16 copy
    // the down LoRA shrink reads
    moe::QuantParams qp{};
    qp.x = hf;
    qp.x_f32 = 1;
    qp.row_map = nullptr;
    qp.map_div = 1;
    qp.rows = static_cast<int>(n);
    qp.K = I;
    qp.codes = hq;
    qp.scales = hs;
    qp.copy = h;
    if (moe::launch_quant_groups(qp, stream) != cudaSuccess) return MOE_ERR_CUDA;
  }
  // 5. down LoRA shrink: V = s * A_dn h (fused: inside the down GEMM)
  if (lora && !fuse_shrink) {
    sp.X = h;
    sp.p2e = nullptr;
    sp.K = I;
    sp.gathered = nullptr;
    sp.A = static_cast<const __nv_bfloat16*>(a->down.A);
    sp.a_stride_adapter = a->down.a_stride_adapter;
    sp.a_stride_expert = a->down.a_stride_expert;
    sp.U = V;
    sp.kc = moe::shrink_chunk(I, r, shrink_budget);
    sp.per_token = 0;
    sp.tables_ready = 1;  // the permute completed before the gate_up GEMM let this grid launch
    if ((row_blocks ? moe::launch_rows_shrink(sp, static_cast<int>(n), stream)
                    : moe::launch_gather_shrink(sp, static_cast<int>(n), stream)) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if (!mark()) return MOE_ERR_CUDA;
  // 6. down GEMM + LoRA expand -> y
  gp.K = I;
  gp.rows_per_expert = H;
  gp.n_feat = H;
  gp.feat_blocks = (H + 127) / 128;
  gp.debug_stall_mma = 0;
  gp.debug_hold_row = 0;
  gp.lb_row_stride_adapter = dn_rs_a;
  gp.lb_row_stride_expert = dn_rs_e;
  gp.out = y;
  // After the shrink, or (fused) after the gate_up GEMM, which runs no
  // earlier than the gate_up shrink's own wait: the tables are complete.
  gp.tables_ready = lora ? 1 : 0;
  if (fuse_shrink) {
    gp.sx = h;
    gp.gather_src = nullptr;
    gp.sa = static_cast<const __nv_bfloat16*>(a->down.A);
    gp.sa_stride_adapter = a->down.a_stride_adapter;
    gp.sa_stride_expert = a->down.a_stride_expert;
    gp.su = V;
    gp.tile_flags = flags_dn;
    gp.row_counter = flags_dn + moe::shrink_flag_words(static_cast<int>(n), E) - 1;
  }
  gp.w_scale = w8 ? a->w2_scale : nullptr;
  gp.scale_nb = (H + 127) / 128;
  gp.scale_kb = (I + 127) / 128;
  gp.x_scale = hs;
  gp.out_f32 = nullptr;
  if ((a8 ? moe::launch_fp8_gemm(moe::kDown, bn, tm_w2, tm_h, tm_bdn, tm_v, gp, gemm_grid, stream)
          : moe::launch_expert_gemm(moe::kDown, bn, pair, w8, tm_w2, tm_h, tm_bdn, tm_v, tm_h_s, tm_v_s, gp,
                                    gemm_grid, stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (!mark()) return MOE_ERR_CUDA;
  // 7. finalize
  if (moe::launch_finalize(y, e2p, topk_w, T, K, H, static_cast<__nv_bfloat16*>(a->out), stream) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  if (!finish_marks()) return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // extern "C"
