// Routing (top-k softmax, renormalised), the expert-grouped permutation with
// its row gather, and the weighted finalize.
//
// Pipeline stages "routing -> moe::dev::permute (bf16 gather)" and
// "finalize" of the launcher row in the "Files changed" table of
// "[WIP][LoRA] BF16 support for the experimental_sgl_trtllm MoE-LoRA path &
// lora expert_outer_shared" (yushengsu-thu/sglang#4).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/moe_lora.h"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

constexpr unsigned kFull = 0xFFFFFFFFu;

// ------------------------------------------------------------------ router
// One warp per token.  Expert i lives in lane i % 32, register slot i / 32.
// A selection key orders by the float32 logit (as a sortable integer, -0
// folded onto +0) and, among equal logits, by the lower expert id; 0 marks
// "already taken / no expert".  Every real key is > 0.
__device__ __forceinline__ uint32_t float_order_bits(float l) {
  uint32_t b = __float_as_uint(l);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float float_from_order_bits(uint32_t o) {
  const uint32_t b = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
  return __uint_as_float(b);
}

template <int EPL>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T,
                                                         int E, int k, int32_t* __restrict__ ids,
                                                         float* __restrict__ w) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* row = logits + static_cast<size_t>(t) * E;

  uint64_t key[EPL];
#pragma unroll
  for (int s = 0; s < EPL; ++s) {
    const int i = s * 32 + lane;
    key[s] = (i < E) ? ((static_cast<uint64_t>(float_order_bits(row[i])) << 32) |
                        static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(i)))
                     : 0ull;
  }

  float my_logit = 0.f;  // lane j keeps slot j
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    uint64_t best = 0;
#pragma unroll
    for (int s = 0; s < EPL; ++s) best = key[s] > best ? key[s] : best;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const uint64_t o = __shfl_xor_sync(kFull, best, off);
      best = o > best ? o : best;
    }
    const uint32_t idx = 0xFFFFFFFFu - static_cast<uint32_t>(best & 0xFFFFFFFFull);
#pragma unroll
    for (int s = 0; s < EPL; ++s)
      if (static_cast<uint32_t>(s * 32 + lane) == idx) key[s] = 0ull;
    if (lane == j) {
      my_logit = float_from_order_bits(static_cast<uint32_t>(best >> 32));
      my_id = static_cast<int>(idx);
    }
  }

  // Renormalised softmax over the selected slots: exp(l_j - m) / sum.
  const float m = __shfl_sync(kFull, my_logit, 0);
  const float ex = (lane < k) ? expf(my_logit - m) : 0.f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
  if (lane < k) {
    ids[static_cast<size_t>(t) * k + lane] = my_id;
    w[static_cast<size_t>(t) * k + lane] = ex / sum;
  }
}

cudaError_t launch_route_topk(const float* logits, int T, int E, int top_k, int32_t* ids, float* w,
                              cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const dim3 grid((T + 7) / 8), block(256);
  const int epl = (E + 31) / 32;
  if (epl <= 1) route_topk_kernel<1><<<grid, block, 0, s>>>(logits, T, E, top_k, ids, w);
  else if (epl <= 2) route_topk_kernel<2><<<grid, block, 0, s>>>(logits, T, E, top_k, ids, w);
  else if (epl <= 4) route_topk_kernel<4><<<grid, block, 0, s>>>(logits, T, E, top_k, ids, w);
  else if (epl <= 8) route_topk_kernel<8><<<grid, block, 0, s>>>(logits, T, E, top_k, ids, w);
  else if (epl <= 16) route_topk_kernel<16><<<grid, block, 0, s>>>(logits, T, E, top_k, ids, w);
  else route_topk_kernel<32><<<grid, block, 0, s>>>(logits, T, E, top_k, ids, w);
  return cudaGetLastError();
}

// ----------------------------------------------------------------- permute
// Three kernels: (1) per 1024-slot chunk, the stable rank of every slot among
// the earlier slots of the same expert in the chunk, and the chunk's
// per-expert counts; (2) one block turns the counts into expert offsets,
// per-chunk bases and tile prefixes; (3) one warp per slot writes the final
// permuted index, the inverse map, the row's adapter, and copies the row.

__device__ __forceinline__ int checked_id(int id, int E, int* status, bool report) {
  if (id == -1) return -1;
  if (id < -1 || id >= E) {
    if (report) set_status(status, MOE_ERR_BAD_EXPERT_ID);
    return -1;
  }
  return id;
}

__global__ void __launch_bounds__(32) permute_count_kernel(PermuteParams p) {
  extern __shared__ int cnt[];
  const int lane = threadIdx.x;
  for (int e = lane; e < p.E; e += 32) cnt[e] = 0;
  __syncwarp();
  const int base = blockIdx.x * kPermuteChunk;
  const int end = min(base + kPermuteChunk, p.n);
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int x0 = base; x0 < end; x0 += 32) {
    const int x = x0 + lane;
    const bool valid = x < end;
    const int id = valid ? checked_id(p.topk_ids[x], p.E, p.status, true) : -1;
    const bool routed = id >= 0;
    const unsigned group = __match_any_sync(kFull, routed ? id : -2);
    const int rank = __popc(group & lt_mask);
    const int prev = routed ? cnt[id] : 0;
    __syncwarp();
    if (routed && rank == 0) cnt[id] = prev + __popc(group);
    __syncwarp();
    if (valid) p.e2p[x] = routed ? prev + rank : -1;  // rank inside the chunk for now
  }
  __syncwarp();
  for (int e = lane; e < p.E; e += 32) p.chunk_counts[blockIdx.x * p.E + e] = cnt[e];
}

// Exclusive scan over the block (blockDim.x == 1024).  Returns the exclusive
// prefix of ``v`` and writes the block total to *total.
__device__ int block_exclusive_scan_1024(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(kFull, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int s = warp_sums[lane];
    int si = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(kFull, si, off);
      if (lane >= off) si += o;
    }
    warp_sums[lane] = si - s;  // exclusive prefix of the warp totals
    if (lane == 31) *total = si;
  }
  __syncthreads();
  const int res = warp_sums[warp] + incl - v;
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(1024) permute_scan_kernel(PermuteParams p, int nchunks) {
  __shared__ int warp_sums[32];
  __shared__ int s_total;
  const int e = threadIdx.x;
  int total = 0;
  if (e < p.E) {
    for (int c = 0; c < nchunks; ++c) {
      const int v = p.chunk_counts[c * p.E + e];
      p.chunk_counts[c * p.E + e] = total;
      total += v;
    }
  }
  const int off = block_exclusive_scan_1024(e < p.E ? total : 0, warp_sums, &s_total);
  if (e < p.E) p.expert_offsets[e] = off;
  if (e == 0) p.expert_offsets[p.E] = s_total;
  if (p.tile_start != nullptr) {
    for (int wi = 0; wi < kNumTileWidths; ++wi) {
      const int bn = tile_width_of(wi);
      const int tiles = e < p.E ? (total + bn - 1) / bn : 0;
      const int ts = block_exclusive_scan_1024(tiles, warp_sums, &s_total);
      if (e < p.E) p.tile_start[wi * (p.E + 1) + e] = ts;
      if (e == 0) p.tile_start[wi * (p.E + 1) + p.E] = s_total;
    }
  }
}

__global__ void __launch_bounds__(256) permute_scatter_kernel(PermuteParams p) {
  const int lane = threadIdx.x & 31;
  const int x = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (x >= p.n) return;
  int pidx = -1;
  if (lane == 0) {
    const int id = checked_id(p.topk_ids[x], p.E, p.status, false);
    if (id >= 0) {
      pidx = p.expert_offsets[id] + p.chunk_counts[(x / kPermuteChunk) * p.E + id] + p.e2p[x];
      p.p2e[pidx] = x;
      if (p.row_adapter != nullptr) {
        int a = -1;
        if (p.num_adapters > 0 && p.mapping != nullptr) {
          a = p.mapping[x / p.top_k];
          if (a < -1 || a >= p.num_adapters) {
            set_status(p.status, MOE_ERR_BAD_MAPPING);
            a = -1;
          }
        }
        p.row_adapter[pidx] = a;
      }
    }
    p.e2p[x] = pidx;
  }
  pidx = __shfl_sync(kFull, pidx, 0);
  if (pidx < 0 || p.hidden == nullptr || p.permuted == nullptr) return;
  const uint4* src = reinterpret_cast<const uint4*>(p.hidden + static_cast<size_t>(x / p.top_k) * p.H);
  uint4* dst = reinterpret_cast<uint4*>(p.permuted + static_cast<size_t>(pidx) * p.H);
  const int nvec = p.H / 8;
  for (int v = lane; v < nvec; v += 32) dst[v] = __ldg(src + v);
}

__global__ void permute_fill_tail_kernel(int32_t* p2e, const int32_t* offsets, int E, int n) {
  const int x = blockIdx.x * blockDim.x + threadIdx.x;
  if (x < n && x >= offsets[E]) p2e[x] = -1;
}

size_t permute_scratch_bytes(int n, int E) {
  const size_t nchunks = (static_cast<size_t>(n) + kPermuteChunk - 1) / kPermuteChunk;
  const size_t a = (nchunks * E * sizeof(int32_t) + 255) & ~static_cast<size_t>(255);
  const size_t b = (static_cast<size_t>(kNumTileWidths) * (E + 1) * sizeof(int32_t) + 255) &
                   ~static_cast<size_t>(255);
  return a + b;
}

cudaError_t launch_permute(const PermuteParams& p, cudaStream_t s) {
  if (p.n == 0) return cudaSuccess;
  const int nchunks = (p.n + kPermuteChunk - 1) / kPermuteChunk;
  permute_count_kernel<<<nchunks, 32, p.E * sizeof(int), s>>>(p);
  permute_scan_kernel<<<1, 1024, 0, s>>>(p, nchunks);
  permute_scatter_kernel<<<(p.n + 7) / 8, 256, 0, s>>>(p);
  permute_fill_tail_kernel<<<(p.n + 255) / 256, 256, 0, s>>>(p.p2e, p.expert_offsets, p.E, p.n);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- finalize
// out[t, :] = sum_j w[t, j] * y[e2p[t*k + j], :], summed in slot order in
// float32, rounded to bf16 (nearest even).  One thread per 8 columns.
__global__ void __launch_bounds__(256) finalize_kernel(const __nv_bfloat16* __restrict__ y,
                                                       const int32_t* __restrict__ e2p,
                                                       const float* __restrict__ w, int k, int H,
                                                       __nv_bfloat16* __restrict__ out) {
  const int t = blockIdx.x;
  const int c8 = blockIdx.y * blockDim.x + threadIdx.x;
  if (c8 * 8 >= H) return;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  for (int j = 0; j < k; ++j) {
    const int p = e2p[static_cast<size_t>(t) * k + j];
    if (p < 0) continue;
    const float wj = w[static_cast<size_t>(t) * k + j];
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(y + static_cast<size_t>(p) * H) + c8);
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h2[i]);
      acc[2 * i] = fmaf(wj, f.x, acc[2 * i]);
      acc[2 * i + 1] = fmaf(wj, f.y, acc[2 * i + 1]);
    }
  }
  uint4 o;
  __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
  for (int i = 0; i < 4; ++i) o2[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
  reinterpret_cast<uint4*>(out + static_cast<size_t>(t) * H)[c8] = o;
}

cudaError_t launch_finalize(const __nv_bfloat16* y, const int32_t* e2p, const float* w, int T,
                            int top_k, int H, __nv_bfloat16* out, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const dim3 grid(T, (H / 8 + 255) / 256);
  finalize_kernel<<<grid, 256, 0, s>>>(y, e2p, w, top_k, H, out);
  return cudaGetLastError();
}

}  // namespace moe
