// Routing (top-k softmax, renormalised), the expert-grouped permutation with
// its row gather, and the weighted finalize.
//
// Pipeline stages "routing -> moe::dev::permute (bf16 gather)" and
// "finalize" of the launcher row in the "Files changed" table of
// "[WIP][LoRA] BF16 support for the experimental_sgl_trtllm MoE-LoRA path &
// lora expert_outer_shared" (yushengsu-thu/sglang#4).
#include <algorithm>
#include <atomic>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/moe_lora.h"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

constexpr unsigned kFull = 0xFFFFFFFFu;

// ------------------------------------------------------------------ router
// One warp per token.  Expert i lives in lane i % 32, register slot i / 32.
// The selection key is the float32 logit as a sortable unsigned integer
// (-0 folded onto +0); 0 marks "already taken / no expert" (every finite
// logit has a key > 0).  Each round takes the largest key with two warp
// reductions (redux.sync): the maximum key, then the lowest expert id among
// the lanes holding it, so equal logits go to the lower id.
__device__ __forceinline__ uint32_t float_order_bits(float l) {
  uint32_t b = __float_as_uint(l);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float float_from_order_bits(uint32_t o) {
  const uint32_t b = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
  return __uint_as_float(b);
}

// Routes one token with a whole warp; lane j < k ends with slot j's expert
// id and renormalised weight.
template <int EPL>
__device__ __forceinline__ void route_token(const float* __restrict__ row, int E, int k, int lane,
                                            int* out_id, float* out_w) {
  uint32_t key[EPL];
#pragma unroll
  for (int s = 0; s < EPL; ++s) {
    const int i = s * 32 + lane;
    key[s] = (i < E) ? float_order_bits(row[i]) : 0u;
  }

  float my_logit = 0.f;  // lane j keeps slot j
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    // this lane's best: the largest key, the lowest slot (= id) among equals
    // (selects only, no conditional stores: the keys stay in registers)
    uint32_t best = 0u;
    int bs = 0;
#pragma unroll
    for (int s = 0; s < EPL; ++s) {
      const bool gt = key[s] > best;
      bs = gt ? s : bs;
      best = gt ? key[s] : best;
    }
    const uint32_t m = __reduce_max_sync(kFull, best);
    const uint32_t cand = (best == m) ? static_cast<uint32_t>(bs * 32 + lane) : 0xFFFFFFFFu;
    const uint32_t idx = __reduce_min_sync(kFull, cand);
    const bool mine = static_cast<int>(idx & 31u) == lane;
#pragma unroll
    for (int s = 0; s < EPL; ++s) key[s] = (mine && static_cast<uint32_t>(s) == (idx >> 5)) ? 0u : key[s];
    if (lane == j) {
      my_logit = float_from_order_bits(m);
      my_id = static_cast<int>(idx);
    }
  }

  // Renormalised softmax over the selected slots: exp(l_j - m) / sum.
  const float m = __shfl_sync(kFull, my_logit, 0);
  const float ex = (lane < k) ? expf(my_logit - m) : 0.f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
  *out_id = my_id;
  *out_w = ex / sum;
}

template <int EPL>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T,
                                                         int E, int k, int32_t* __restrict__ ids,
                                                         float* __restrict__ w) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  pdl_wait();  // no-ops unless launched as a programmatic dependent launch
  pdl_launch_dependents();
  if (t >= T) return;
  int id;
  float wt;
  route_token<EPL>(logits + static_cast<size_t>(t) * E, E, k, lane, &id, &wt);
  if (lane < k) {
    ids[static_cast<size_t>(t) * k + lane] = id;
    w[static_cast<size_t>(t) * k + lane] = wt;
  }
}

cudaError_t launch_route_topk_pdl(const float* logits, int T, int E, int top_k, int32_t* ids, float* w,
                                  cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const dim3 grid((T + 7) / 8), block(256);
  const int epl = (E + 31) / 32;
  if (epl <= 1) return launch_pdl(route_topk_kernel<1>, grid, block, 0, s, logits, T, E, top_k, ids, w);
  if (epl <= 2) return launch_pdl(route_topk_kernel<2>, grid, block, 0, s, logits, T, E, top_k, ids, w);
  if (epl <= 4) return launch_pdl(route_topk_kernel<4>, grid, block, 0, s, logits, T, E, top_k, ids, w);
  if (epl <= 8) return launch_pdl(route_topk_kernel<8>, grid, block, 0, s, logits, T, E, top_k, ids, w);
  if (epl <= 16) return launch_pdl(route_topk_kernel<16>, grid, block, 0, s, logits, T, E, top_k, ids, w);
  return launch_pdl(route_topk_kernel<32>, grid, block, 0, s, logits, T, E, top_k, ids, w);
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

// Expert parallelism: a routed id is global in [0, id_limit); this call holds
// experts [id_offset, id_offset + E).  Returns the local expert, or -1 for a
// slot that is not routed, or routed to another shard's expert (dropped
// without error).  Ids outside [-1, id_limit) are reported as bad.
__device__ __forceinline__ int local_id(int id, int id_offset, int E, int id_limit, int* status,
                                        bool report) {
  const int g = checked_id(id, id_limit, status, report);
  if (g < 0) return -1;
  const int e = g - id_offset;
  return (e >= 0 && e < E) ? e : -1;
}

// 8 warps per 1024-slot chunk; warp w ranks slots [128w, 128w + 128) of the
// chunk with its own counters, then the counters are merged by a prefix over
// the warps, so ranks follow the slot order of the whole chunk.
constexpr int kCountWarps = 8;
__global__ void __launch_bounds__(32 * kCountWarps) permute_count_kernel(PermuteParams p) {
  extern __shared__ int cnt[];  // [kCountWarps][E]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kCountWarps * p.E; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  const int seg = kPermuteChunk / kCountWarps;
  const int base = blockIdx.x * kPermuteChunk + warp * seg;
  const int end = min(base + seg, p.n);
  int* my = cnt + warp * p.E;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int x0 = base; x0 < end; x0 += 32) {
    const int x = x0 + lane;
    const bool valid = x < end;
    const int id = valid ? local_id(p.topk_ids[x], p.id_offset, p.E, p.id_limit, p.status, true) : -1;
    const bool routed = id >= 0;
    const unsigned group = __match_any_sync(kFull, routed ? id : -2);
    const int rank = __popc(group & lt_mask);
    const int prev = routed ? my[id] : 0;
    __syncwarp();
    if (routed && rank == 0) my[id] = prev + __popc(group);
    __syncwarp();
    if (valid) p.e2p[x] = routed ? prev + rank : -1;  // rank inside the warp segment for now
  }
  __syncthreads();
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < kCountWarps; ++w) {
      const int v = cnt[w * p.E + e];
      cnt[w * p.E + e] = run;
      run += v;
    }
    p.chunk_counts[blockIdx.x * p.E + e] = run;
  }
  __syncthreads();
  if (base < end) {
    for (int x = base + lane; x < end; x += 32) {
      const int r = p.e2p[x];
      if (r >= 0) p.e2p[x] = r + my[local_id(p.topk_ids[x], p.id_offset, p.E, p.id_limit, p.status, false)];
    }
  }
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
    // Loads in batches, so that the chain of chunks costs one memory round
    // trip per 16 chunks instead of one per chunk.
    constexpr int kBatch = 16;
    for (int c0 = 0; c0 < nchunks; c0 += kBatch) {
      int v[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) v[i] = c0 + i < nchunks ? p.chunk_counts[(c0 + i) * p.E + e] : 0;
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        if (c0 + i < nchunks) p.chunk_counts[(c0 + i) * p.E + e] = total;
        total += v[i];
      }
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

// One thread per slot: final permuted index, inverse map, row adapter.
__global__ void __launch_bounds__(256) permute_scatter_kernel(PermuteParams p) {
  const int x = blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= p.n) return;
  const int id = local_id(p.topk_ids[x], p.id_offset, p.E, p.id_limit, p.status, false);
  // Slots past the routed rows (dropped ids) have no source row.
  if (x >= p.expert_offsets[p.E]) p.p2e[x] = -1;
  int pidx = -1;
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

// permuted[p] = hidden[x / top_k] for every routed slot x (one warp per slot).
__global__ void __launch_bounds__(256) permute_gather_kernel(PermuteParams p) {
  const int lane = threadIdx.x & 31;
  const int x = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (x >= p.n) return;
  const int pidx = p.e2p[x];
  if (pidx < 0) return;
  const uint4* src = reinterpret_cast<const uint4*>(p.hidden + static_cast<size_t>(x / p.top_k) * p.H);
  uint4* dst = reinterpret_cast<uint4*>(p.permuted + static_cast<size_t>(pidx) * p.H);
  for (int v = lane; v < p.H / 8; v += 32) dst[v] = __ldg(src + v);
}

size_t permute_scratch_bytes(int n, int E) {
  const size_t nchunks = (static_cast<size_t>(n) + kPermuteChunk - 1) / kPermuteChunk;
  const size_t a = (nchunks * E * sizeof(int32_t) + 255) & ~static_cast<size_t>(255);
  const size_t b = (static_cast<size_t>(kNumTileWidths) * (E + 1) * sizeof(int32_t) + 255) &
                   ~static_cast<size_t>(255);
  return a + b + gmask_bytes(n, E) + ((2 * shrink_flag_words(n, E) * sizeof(int) + 255) & ~static_cast<size_t>(255));
}

size_t shrink_flag_words(int n, int E) { return (static_cast<size_t>(n) + 15) / 16 + E + 1; }

size_t gmask_bytes(int n, int E) {
  const size_t tiles16 = (static_cast<size_t>(n) + 15) / 16 + E + 1;
  return (tiles16 * sizeof(uint64_t) + 255) & ~static_cast<size_t>(255);
}

cudaError_t launch_permute(const PermuteParams& pin, cudaStream_t s) {
  PermuteParams p = pin;
  if (p.id_limit <= 0) p.id_limit = p.E;  // no sharding
  if (p.n == 0) return cudaSuccess;
  const int nchunks = (p.n + kPermuteChunk - 1) / kPermuteChunk;
  permute_count_kernel<<<nchunks, 32 * kCountWarps, kCountWarps * p.E * sizeof(int), s>>>(p);
  permute_scan_kernel<<<1, 1024, 0, s>>>(p, nchunks);
  permute_scatter_kernel<<<(p.n + 255) / 256, 256, 0, s>>>(p);
  if (p.hidden != nullptr && p.permuted != nullptr)
    permute_gather_kernel<<<(p.n + 7) / 8, 256, 0, s>>>(p);
  return cudaGetLastError();
}

// ------------------------------ routing + permute in three chained kernels
// The forward's path past the one-CTA permute.  The slots are cut into
// chunks of whole tokens (tokens_per_chunk * top_k <= kPermuteChunk slots).
//   route_topk_kernel, one warp per token, over the whole GPU;
//   route_count_kernel, one CTA of 32 warps per chunk: warp w ranks the
//     slots of its segment [w seg, (w + 1) seg) among the earlier slots of
//     the same expert (match_any, per-warp counters); a prefix over the
//     warps' counters turns the ranks into ranks within the chunk, and the
//     chunk's per-expert totals go out.
//   scan_scatter_kernel, one CTA per chunk: every CTA reads all chunk totals,
//     forms its chunk's per-expert base (the expert offset from a block scan
//     of the expert totals, plus the counts of earlier chunks), and writes
//     the final permuted index, the inverse map and the row adapter of its
//     slots; CTA 0 also writes the expert offsets and the tile prefixes.
// All three are programmatic dependent launches.  Stable order: slots in
// expanded order within each expert, as in the other permutes.
__global__ void __launch_bounds__(1024) route_count_kernel(const RoutePermuteParams p) {
  extern __shared__ int rc_smem[];
  const int E = p.E, k = p.top_k;
  int* cnt = rc_smem;                                        // [32][E]
  int16_t* s_ids = reinterpret_cast<int16_t*>(cnt + 32 * E);  // [kPermuteChunk]
  int16_t* s_rank = s_ids + kPermuteChunk;                    // [kPermuteChunk]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * p.tokens_per_chunk;
  const int nt = min(p.tokens_per_chunk, p.T - t0);
  const int ns = nt * k, x0 = t0 * k;
  pdl_wait();
  if (blockIdx.x == 0 && tid < 4) p.status[tid] = 0;
  for (int i = tid; i < 32 * E; i += blockDim.x) cnt[i] = 0;
  for (int x = tid; x < ns; x += blockDim.x) {  // the router's ids (global, always in range)
    const int e = __ldcg(p.topk_ids + x0 + x) - p.id_offset;
    s_ids[x] = static_cast<int16_t>(e >= 0 && e < E ? e : -1);
  }
  __syncthreads();
  const int seg = (ns + 31) / 32;
  const int xb = warp * seg, xe = min(xb + seg, ns);
  int* my = cnt + warp * E;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int xs = xb; xs < xe; xs += 32) {
    const int x = xs + lane;
    const bool valid = x < xe;
    const int id = valid ? s_ids[x] : -1;
    const bool routed = id >= 0;
    const unsigned grp = __match_any_sync(kFull, routed ? id : -2);
    const int rank = __popc(grp & lt_mask);
    const int prev = routed ? my[id] : 0;
    __syncwarp();
    if (routed && rank == 0) my[id] = prev + __popc(grp);
    __syncwarp();
    if (valid) s_rank[x] = static_cast<int16_t>(routed ? prev + rank : -1);
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < 32; ++w) {
      const int v = cnt[w * E + e];
      cnt[w * E + e] = run;
      run += v;
    }
    p.chunk_counts[static_cast<size_t>(blockIdx.x) * E + e] = run;
  }
  __syncthreads();
  pdl_launch_dependents();
  for (int x = tid; x < ns; x += blockDim.x) {
    const int id = s_ids[x];
    p.e2p[x0 + x] = id >= 0 ? s_rank[x] + cnt[(x / seg) * E + id] : -1;  // rank within the chunk
  }
}

__global__ void __launch_bounds__(1024) scan_scatter_kernel(const RoutePermuteParams p, int nchunks) {
  __shared__ int warp_sums[32];
  __shared__ int s_total;
  extern __shared__ int ss_smem[];  // [E]: the chunk's base per expert
  const int E = p.E, k = p.top_k, tid = threadIdx.x, c = blockIdx.x;
  pdl_wait();
  int pre = 0, total = 0;
  if (tid < E) {
    // loads in batches: one memory round trip per 16 chunks
    constexpr int kBatch = 16;
    for (int c0 = 0; c0 < nchunks; c0 += kBatch) {
      int v[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i)
        v[i] = c0 + i < nchunks ? __ldcg(p.chunk_counts + static_cast<size_t>(c0 + i) * E + tid) : 0;
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        if (c0 + i < c) pre += v[i];
        total += v[i];
      }
    }
  }
  const int off = block_exclusive_scan_1024(tid < E ? total : 0, warp_sums, &s_total);
  const int routed_total = s_total;
  if (tid < E) ss_smem[tid] = off + pre;
  if (c == 0) {
    if (tid < E) p.expert_offsets[tid] = off;
    if (tid == 0) p.expert_offsets[E] = routed_total;
    for (int wi = 0; wi < kNumTileWidths; ++wi) {
      if (!((p.tile_width_mask >> wi) & 1u)) continue;
      const int bn = tile_width_of(wi);
      const int tiles = tid < E ? (total + bn - 1) / bn : 0;
      const int ts = block_exclusive_scan_1024(tiles, warp_sums, &s_total);
      if (tid < E) p.tile_start[wi * (E + 1) + tid] = ts;
      if (tid == 0) p.tile_start[wi * (E + 1) + E] = s_total;
    }
  }
  __syncthreads();
  pdl_launch_dependents();
  const int t0 = c * p.tokens_per_chunk;
  const int nt = min(p.tokens_per_chunk, p.T - t0);
  const int x0 = t0 * k;
  for (int x = x0 + tid; x < x0 + nt * k; x += blockDim.x) {
    const int r = __ldcg(p.e2p + x);
    int pidx = -1;
    if (r >= 0) {
      const int e = __ldcg(p.topk_ids + x) - p.id_offset;  // routed here: a local expert
      pidx = ss_smem[e] + r;
      p.p2e[pidx] = x;
      if (p.row_adapter != nullptr) {
        int a = -1;
        if (p.num_adapters > 0 && p.mapping != nullptr) {
          a = __ldg(p.mapping + x / k);
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
  // rows past the routed ones (slots dropped by expert parallelism) have no source
  const int n = p.T * k;
  for (int x = routed_total + c * blockDim.x + tid; x < n; x += gridDim.x * blockDim.x) p.p2e[x] = -1;
}

bool route_permute_fits(int T, int top_k, int E) {
  return T > 0 && E <= kRoutePermuteMaxE && top_k <= 32 && kPermuteChunk % top_k == 0;
}

cudaError_t launch_route_permute(const RoutePermuteParams& pin, cudaStream_t s) {
  RoutePermuteParams p = pin;
  p.tokens_per_chunk = kPermuteChunk / p.top_k;
  const int nchunks = (p.T + p.tokens_per_chunk - 1) / p.tokens_per_chunk;
  const size_t smem1 = static_cast<size_t>(32) * p.E * 4 + 2 * kPermuteChunk * sizeof(int16_t);
  const size_t smem2 = static_cast<size_t>(p.E) * 4;
  cudaError_t err = launch_route_topk_pdl(p.logits, p.T, p.id_limit, p.top_k, p.topk_ids, p.topk_w, s);
  if (err != cudaSuccess) return err;
  err = ensure_smem_limit(reinterpret_cast<const void*>(route_count_kernel), (int)smem1);
  if (err != cudaSuccess) return err;
  err = launch_pdl(route_count_kernel, dim3(nchunks), dim3(1024), smem1, s, p);
  if (err != cudaSuccess) return err;
  return launch_pdl(scan_scatter_kernel, dim3(nchunks), dim3(1024), smem2, s, p, nchunks);
}

// ------------------------------------------------- one-CTA permute (fused)
// For n = T*k slots small enough that the whole counting sort fits in one
// CTA's shared memory.  Optionally routes the tokens first (one warp per
// token).  Clears the device status word, then:
//   pass 1: warp w takes slots [w*seg, (w+1)*seg) in order and gives each
//           slot its stable rank among earlier slots of the same expert in
//           the segment (match_any per 32 slots, per-warp expert counters);
//   pass 2: per expert, an exclusive scan of the 32 warp counters; a block
//           scan of the expert totals gives the expert offsets and the tile
//           prefixes;
//   pass 3: permuted index = offset[e] + warp base + rank; inverse map and
//           the row's adapter.
template <int EPL>
__global__ void __launch_bounds__(1024) small_permute_kernel(const FusedPermuteParams p) {
  extern __shared__ int4 small_smem[];
  const int n = p.T * p.top_k, E = p.E, k = p.top_k;
  const int n2 = (n + 1) & ~1;
  // 8-byte words first (the dynamic shared memory base is 16-byte aligned):
  // the adapters of each 16-row tile (p.gmask only)
  const int ntiles16 = (n + 15) / 16 + E + 1;
  unsigned long long* s_m16 = reinterpret_cast<unsigned long long*>(small_smem);
  int16_t* s_ids = reinterpret_cast<int16_t*>(s_m16 + ntiles16);
  int16_t* s_local = s_ids + n2;
  int* s_cnt = reinterpret_cast<int*>(s_local + n2);
  int* s_off = s_cnt + 32 * E;
  int* s_t16 = s_off + (E + 1);  // 16-wide tile prefix
  __shared__ int warp_sums[32];
  __shared__ int s_total;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  pdl_wait();
  if (tid == 0) p.status[0] = 0;
  for (int i = tid; i < p.clear_count; i += blockDim.x) p.clear_flags[i] = 0;
  for (int i = tid; i < 32 * E; i += blockDim.x) s_cnt[i] = 0;
  __syncthreads();
  // The next kernel may start now (after the status word and the flags are
  // cleared): every consumer of the tables below waits for this grid to
  // complete (griddepcontrol.wait) before it reads them, and the per-token
  // shrink does its factor product meanwhile.
  pdl_launch_dependents();
  if (p.logits != nullptr) {
    for (int t = warp; t < p.T; t += 32) {
      int id;
      float wt;
      route_token<EPL>(p.logits + static_cast<size_t>(t) * p.id_limit, p.id_limit, k, lane, &id, &wt);
      if (lane < k) {
        p.topk_ids[t * k + lane] = id;  // global id
        p.topk_w[t * k + lane] = wt;
        const int e = id - p.id_offset;
        s_ids[t * k + lane] = static_cast<int16_t>(e >= 0 && e < E ? e : -1);
      }
    }
  } else {
    for (int x = tid; x < n; x += blockDim.x)
      s_ids[x] = static_cast<int16_t>(local_id(p.topk_ids[x], p.id_offset, E, p.id_limit, p.status, true));
  }
  __syncthreads();

  const int seg = (n + 31) / 32;
  const int x_begin = warp * seg, x_end = min(x_begin + seg, n);
  int* cnt = s_cnt + warp * E;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int x0 = x_begin; x0 < x_end; x0 += 32) {
    const int x = x0 + lane;
    const bool valid = x < x_end;
    const int id = valid ? s_ids[x] : -1;
    const bool routed = id >= 0;
    const unsigned grp = __match_any_sync(kFull, routed ? id : -2);
    const int rank = __popc(grp & lt_mask);
    const int prev = routed ? cnt[id] : 0;
    __syncwarp();
    if (routed && rank == 0) cnt[id] = prev + __popc(grp);
    __syncwarp();
    if (valid) s_local[x] = static_cast<int16_t>(routed ? prev + rank : -1);
  }
  __syncthreads();

  int total = 0;
  if (tid < E) {
    for (int w = 0; w < 32; ++w) {
      const int v = s_cnt[w * E + tid];
      s_cnt[w * E + tid] = total;
      total += v;
    }
  }
  const int off = block_exclusive_scan_1024(tid < E ? total : 0, warp_sums, &s_total);
  if (tid < E) {
    s_off[tid] = off;
    p.expert_offsets[tid] = off;
  }
  if (tid == 0) {
    s_off[E] = s_total;
    p.expert_offsets[E] = s_total;
  }
  if (p.tile_start != nullptr) {
    for (int wi = 0; wi < kNumTileWidths; ++wi) {
      if (!((p.tile_width_mask >> wi) & 1u)) continue;
      const int bn = tile_width_of(wi);
      const int tiles = tid < E ? (total + bn - 1) / bn : 0;
      const int ts = block_exclusive_scan_1024(tiles, warp_sums, &s_total);
      if (tid < E) p.tile_start[wi * (E + 1) + tid] = ts;
      if (tid == 0) p.tile_start[wi * (E + 1) + E] = s_total;
      if (bn == 16) {
        if (tid < E) s_t16[tid] = ts;
        if (tid == 0) s_t16[E] = s_total;
      }
    }
  }
  if (p.gmask != nullptr)
    for (int i = tid; i < ntiles16; i += blockDim.x) s_m16[i] = 0ull;
  __syncthreads();

  for (int x = tid; x < n; x += blockDim.x) {
    const int id = s_ids[x];
    int pidx = -1;
    if (id >= 0) {
      pidx = s_off[id] + s_cnt[(x / seg) * E + id] + s_local[x];
      p.p2e[pidx] = x;
      if (p.row_adapter != nullptr) {
        int a = -1;
        if (p.num_adapters > 0 && p.mapping != nullptr) {
          a = p.mapping[x / k];
          if (a < -1 || a >= p.num_adapters) {
            set_status(p.status, MOE_ERR_BAD_MAPPING);
            a = -1;
          }
        }
        p.row_adapter[pidx] = a;
        if (p.gmask != nullptr && a >= 0)
          atomicOr(&s_m16[s_t16[id] + (pidx - s_off[id]) / 16], 1ull << a);
      }
    }
    p.e2p[x] = pidx;
  }
  for (int x = s_off[E] + tid; x < n; x += blockDim.x) p.p2e[x] = -1;
  if (p.gmask != nullptr) {
    __syncthreads();  // every 16-row tile's adapters are in s_m16
    const int ntiles = s_t16[E];
    const int per = p.gemm_bn / 16;  // 16-row tiles per GEMM tile
    for (int t = tid; t < ntiles; t += blockDim.x) {
      int lo = 0, hi = E - 1;  // expert of 16-row tile t
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_t16[mid] <= t) lo = mid;
        else hi = mid - 1;
      }
      // the GEMM tile starts at a multiple of gemm_bn rows within the expert
      const int first = s_t16[lo] + ((t - s_t16[lo]) / per) * per;
      const int last = min(first + per, s_t16[lo + 1]);
      unsigned long long m = 0;
      for (int u = first; u < last; ++u) m |= s_m16[u];
      p.gmask[t] = m;
    }
  }
}

size_t small_permute_smem(int n, int E) {
  const size_t n2 = (static_cast<size_t>(n) + 1) & ~static_cast<size_t>(1);
  const size_t tiles16 = (static_cast<size_t>(n) + 15) / 16 + E + 1;
  return tiles16 * 8 + n2 * 2 * 2 + static_cast<size_t>(32) * E * 4 +
         2 * (static_cast<size_t>(E) + 1) * 4;
}

bool small_permute_fits(int n, int E) {
  return n <= 8192 && small_permute_smem(n, E) <= 200 * 1024;
}

cudaError_t launch_small_permute(const FusedPermuteParams& pin, cudaStream_t s) {
  FusedPermuteParams p = pin;
  if (p.id_limit <= 0) p.id_limit = p.E;  // no sharding
  const int n = p.T * p.top_k;
  const size_t smem = small_permute_smem(n, p.E);
  const int epl = (p.id_limit + 31) / 32;  // routing scores all id_limit experts
#define MOE_SMALL_CASE(V)                                                                         \
  {                                                                                               \
    cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(small_permute_kernel<V>), (int)smem); \
    if (err != cudaSuccess) return err;                                                           \
    return launch_pdl(small_permute_kernel<V>, dim3(1), dim3(1024), smem, s, p);                  \
  }
  if (p.logits == nullptr || epl <= 1) MOE_SMALL_CASE(1)
  if (epl <= 2) MOE_SMALL_CASE(2)
  if (epl <= 4) MOE_SMALL_CASE(4)
  if (epl <= 8) MOE_SMALL_CASE(8)
  if (epl <= 16) MOE_SMALL_CASE(16)
  MOE_SMALL_CASE(32)
#undef MOE_SMALL_CASE
}

// ---------------------------------------------------------------- finalize
// out[t] = sum_j w[t, j] y[e2p[t k + j]], slots in order j = 0..k-1, fp32
// accumulation.  Persistent: CTA b takes tokens b, b + gridDim.x, ...; each
// thread owns 8 consecutive columns of one token and loads the next token's
// slot indices and weights while this token's rows are in flight.  KMAX
// (>= k) bounds the unrolled slot loops so the indices stay in registers.
template <int KMAX>
__global__ void __launch_bounds__(256) finalize_kernel(const __nv_bfloat16* __restrict__ y,
                                                       const int32_t* __restrict__ e2p,
                                                       const float* __restrict__ w, int T, int k,
                                                       int H, __nv_bfloat16* __restrict__ out) {
  const int c8 = blockIdx.y * blockDim.x + threadIdx.x;
  int p_cur[KMAX], p_nxt[KMAX];
  float w_cur[KMAX], w_nxt[KMAX];
  auto load_idx = [&](int tok, int (&pp)[KMAX], float (&ww)[KMAX]) {
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      pp[j] = j < k ? __ldcg(e2p + static_cast<size_t>(tok) * k + j) : -1;
      ww[j] = j < k ? __ldcg(w + static_cast<size_t>(tok) * k + j) : 0.f;
    }
  };
  // The slot indices and weights come from the permute, which completed
  // before the down GEMM let this grid launch: the first token's are read
  // while that GEMM drains; y only after the wait.
  int t = blockIdx.x;
  if (t < T && c8 * 8 < H) load_idx(t, p_cur, w_cur);
  pdl_wait();
  pdl_launch_dependents();
  if (c8 * 8 >= H) return;
  for (; t < T; t += gridDim.x) {
    uint4 v[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      v[j] = p_cur[j] >= 0 ? __ldg(reinterpret_cast<const uint4*>(y + static_cast<size_t>(p_cur[j]) * H) + c8)
                           : make_uint4(0, 0, 0, 0);
    // the next token's indices while the rows are in flight
    const int tn = t + static_cast<int>(gridDim.x);
    if (tn < T) load_idx(tn, p_nxt, w_nxt);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (p_cur[j] < 0) continue;
      const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&v[j]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h2[i]);
        acc[2 * i] = fmaf(w_cur[j], f.x, acc[2 * i]);
        acc[2 * i + 1] = fmaf(w_cur[j], f.y, acc[2 * i + 1]);
      }
    }
    uint4 o;
    __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
    for (int i = 0; i < 4; ++i) o2[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    reinterpret_cast<uint4*>(out + static_cast<size_t>(t) * H)[c8] = o;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      p_cur[j] = p_nxt[j];
      w_cur[j] = w_nxt[j];
    }
  }
}

template <int KMAX>
static cudaError_t launch_finalize_k(const __nv_bfloat16* y, const int32_t* e2p, const float* w,
                                     int T, int top_k, int H, __nv_bfloat16* out, cudaStream_t s) {
  constexpr int kMaxDevices = 64;
  // resident CTAs of the persistent grid, per device (computed once; host
  // threads may race to fill it with the same value)
  static std::atomic<int> ctas[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int resident = ctas[dev].load(std::memory_order_relaxed);
  if (resident == 0) {
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, finalize_kernel<KMAX>, 256, 0) !=
            cudaSuccess)
      return cudaErrorUnknown;
    resident = std::max(1, sms * per_sm);
    ctas[dev].store(resident, std::memory_order_relaxed);
  }
  const int ycols = (H / 8 + 255) / 256;
  // as few CTAs as give every CTA the same number of tokens (the last
  // round of a persistent grid is otherwise partly idle)
  const int cap = std::max(1, std::min(T, resident / ycols));
  const int rounds = (T + cap - 1) / cap;
  const int tok_ctas = (T + rounds - 1) / rounds;
  return launch_pdl(finalize_kernel<KMAX>, dim3(tok_ctas, ycols), dim3(256), 0, s, y, e2p, w, T,
                    top_k, H, out);
}

cudaError_t launch_finalize(const __nv_bfloat16* y, const int32_t* e2p, const float* w, int T,
                            int top_k, int H, __nv_bfloat16* out, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (top_k <= 8) return launch_finalize_k<8>(y, e2p, w, T, top_k, H, out, s);
  if (top_k <= 16) return launch_finalize_k<16>(y, e2p, w, T, top_k, H, out, s);
  return launch_finalize_k<MOE_MAX_TOP_K>(y, e2p, w, T, top_k, H, out, s);
}

}  // namespace moe
