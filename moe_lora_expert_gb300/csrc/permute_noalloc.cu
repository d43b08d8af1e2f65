// moe_permute_noalloc: the expert-grouped permutation of moe_permute for
// callers that cannot allocate device memory.
//
// Who needs it: code that runs where no allocator may be called, such as a
// plugin inside a host framework that owns every device buffer and forbids
// cudaMalloc on its streams, or a custom allocator's own bootstrap path.
// Such a caller has its inputs and outputs but no spare device buffer to
// hand over as the counting-sort scratch that moe_permute takes.
//
// The scratch (the device status word and the per-chunk expert counts) lives
// in one file-scope device array of fixed size instead.  Every GPU that loads
// the library keeps that array until the process exits.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/moe_lora.h"
#include "kernels.cuh"

namespace {

// Status word (16 bytes, padded to 256) followed by the per-chunk counts:
// ceil(n / 1024) chunks x E experts of int32.
constexpr int kStatusInts = 64;
constexpr int kCountInts =
    ((MOE_NOALLOC_MAX_SLOTS + moe::kPermuteChunk - 1) / moe::kPermuteChunk) * MOE_MAX_EXPERTS;

static __device__ __align__(256) int32_t g_noalloc_scratch[kStatusInts + kCountInts];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
int32_t* g_scratch_ptr[kMaxDevices] = {};

// Device address of the array on the current device.  The first call per
// device looks it up (the name itself is only a host-side stand-in) and the
// address is kept for the process: a device reset invalidates it, which the
// header states.
int32_t* scratch_on_current_device(int* status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *status = MOE_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      *status = MOE_ERR_CUDA;
      return nullptr;
    }
    g_scratch_ptr[dev] = static_cast<int32_t*>(p);
  }
  return g_scratch_ptr[dev];
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int moe_permute_noalloc(const int32_t* topk_ids, int T, int top_k, int E,
                                   const void* hidden, int H, int32_t* expert_offsets,
                                   int32_t* expanded_to_permuted, int32_t* permuted_to_expanded,
                                   void* permuted_hidden, int32_t* status_out,
                                   moe_stream_t stream) {
  if (T < 0 || E <= 0 || top_k <= 0) return MOE_ERR_SHAPE;
  if (E > MOE_MAX_EXPERTS || top_k > MOE_MAX_TOP_K) return MOE_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(T) * top_k > MOE_NOALLOC_MAX_SLOTS) return MOE_ERR_UNSUPPORTED;
  if (expert_offsets == nullptr) return MOE_ERR_NULL;
  const bool gather = hidden != nullptr && permuted_hidden != nullptr;
  if (gather && (H <= 0 || H % 8 != 0 || !aligned16(hidden) || !aligned16(permuted_hidden)))
    return MOE_ERR_ALIGN;
  if (T > 0 && (topk_ids == nullptr || expanded_to_permuted == nullptr ||
                permuted_to_expanded == nullptr))
    return MOE_ERR_NULL;

  int st = MOE_OK;
  int32_t* scratch = scratch_on_current_device(&st);
  if (scratch == nullptr) return st;
  (void)cudaGetLastError();  // launch checks below must not report an earlier, unrelated error

  // The status word must start at zero; the counts are fully rewritten.
  if (cudaMemsetAsync(scratch, 0, kStatusInts * sizeof(int32_t), stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (T == 0) {
    if (cudaMemsetAsync(expert_offsets, 0, (E + 1) * sizeof(int32_t), stream) != cudaSuccess)
      return MOE_ERR_CUDA;
  } else {
    moe::PermuteParams p{};
    p.topk_ids = topk_ids;
    p.n = T * top_k;
    p.top_k = top_k;
    p.E = E;
    p.H = H;
    p.hidden = gather ? static_cast<const __nv_bfloat16*>(hidden) : nullptr;
    p.permuted = gather ? static_cast<__nv_bfloat16*>(permuted_hidden) : nullptr;
    p.expert_offsets = expert_offsets;
    p.e2p = expanded_to_permuted;
    p.p2e = permuted_to_expanded;
    p.chunk_counts = scratch + kStatusInts;
    p.tile_start = nullptr;
    p.status = scratch;
    if (moe::launch_permute(p, stream) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (status_out != nullptr &&
      cudaMemcpyAsync(status_out, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice, stream) !=
          cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
