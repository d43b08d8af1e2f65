// Row gather and LoRA shrink: u = s * A[a, e] x for every permuted row, written
// as the one-hot operand of the expand.
//
// The shrink half of ``merged_experts_fused_moe_lora_add`` in Flow 1(A) and
// Flow 2 of "[WIP][LoRA] BF16 support for the experimental_sgl_trtllm
// MoE-LoRA path & lora expert_outer_shared" (yushengsu-thu/sglang#4): the
// gate_up call reads the hidden rows, the down call reads the activation
// output; in the shared-outer sub-mode the gate_up A factor is addressed by
// the adapter only (expert stride 0 here).  For the gate_up call the same
// kernel also performs the "moe::dev::permute (bf16 gather)" row copy of the
// launcher row in that PR's "Files changed" table, since it reads those rows
// anyway.
//
// Output layout: U[p, a*r + i] = bf16(s * (A[a, e(p)] X[p])_i) for the row's
// own adapter a, and 0 in every other column of the row (all zero for rows
// without an adapter).  The expert GEMM multiplies B[a, e] against the
// columns of adapter a only, so rows of other adapters contribute exactly 0.
//
// One CTA per 16-row tile of one expert (tile list from the permute).  The
// tile's source rows and the factor are brought into shared memory with bulk
// copies, all in flight at once on one mbarrier (K split into phases when
// they do not fit).  8 warps split K; each lane reads 8 consecutive K
// elements of rows g and g+8 and of factor row g of each 8-wide N tile and
// feeds two m16n8k16 mma.sync steps with them (same K positions on both
// operands); partial sums meet in shared memory.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/moe_lora.h"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kShrinkThreads = 256;

__host__ __device__ inline size_t shrink_smem_bytes(int kc, int rank) {
  const size_t pitch = (static_cast<size_t>(kc) + 8) * 2;
  return 16 + (16 + static_cast<size_t>(rank)) * pitch + static_cast<size_t>(8 * 16) * rank * 4 +
         static_cast<size_t>(16) * rank * 2;
}

// NT = 0: gather only.  Otherwise the CTA computes R = 8 NT columns of the
// adapter's rank: slice blockIdx.z, columns [R z, R z + R) of p.rank (the
// per-token mode splits a large rank over several CTAs).
template <int NT>
__global__ void __launch_bounds__(kShrinkThreads) gather_shrink_kernel(const ShrinkParams p) {
  constexpr int R = 8 * NT;
  const int rs = static_cast<int>(blockIdx.z);  // rank slice
  extern __shared__ int4 shrink_smem[];
  const int KC = p.kc;
  const int pitch = KC + 8;  // elements; 16-byte pad keeps the mma loads conflict-free
  uint64_t* bar = reinterpret_cast<uint64_t*>(shrink_smem);
  __nv_bfloat16* Xs = reinterpret_cast<__nv_bfloat16*>(reinterpret_cast<uint8_t*>(shrink_smem) + 16);
  __nv_bfloat16* Fs = Xs + 16 * pitch;
  float* s_red = reinterpret_cast<float*>(Fs + R * pitch);   // [8][16][R]
  __nv_bfloat16* s_u = reinterpret_cast<__nv_bfloat16*>(s_red + 8 * 16 * R);  // [16][R]
  __shared__ int s_adapter[16];
  __shared__ int s_src[16];
  __shared__ int s_dst[16 * MOE_MAX_TOP_K];  // per-token mode: e2p of the tile's tokens
  __shared__ int s_info[3];
  __shared__ int s_ok;
  __shared__ int s_ts[MOE_MAX_EXPERTS + 1];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;

  // Per-token mode: the tile (16 tokens), the rows and the factor are the
  // layer's own inputs, so the loads and the product run while the permute
  // is still going; only the scatter to permuted rows waits for it (below).
  if (!p.per_token) pdl_wait();
  // The gather alone: the next kernel reads the gathered rows only after its
  // own griddepcontrol.wait, and the tables are complete now.
  if (!p.per_token && p.U == nullptr) pdl_launch_dependents();
  if (p.gmask != nullptr && !p.per_token) {
    // One round trip decides whether this (tile, adapter slot) has work.
    if (tid == 0) {
      const int tile = blockIdx.x;
      const int count = p.tile_start16[p.E];
      const uint64_t m = p.gmask[tile];
      const int ad = static_cast<int>(blockIdx.y);
      const bool needed = ((m >> ad) & 1ull) != 0 || (p.gathered != nullptr && ad == 0);
      s_ok = (tile < count && needed) ? 1 : 0;
    }
    __syncthreads();
    if (!s_ok) return;
  }
  // The tile prefix comes to shared memory in one coalesced pass, so that
  // the search below costs no chain of global round trips.
  if (!p.per_token)
    for (int i = tid; i <= p.E; i += kShrinkThreads) s_ts[i] = p.tile_start16[i];
  __syncthreads();
  if (tid == 0) {
    const int tile = blockIdx.x;
    const int total = p.per_token ? (p.T + 15) / 16 : s_ts[p.E];
    int e = -1, row0 = 0, nrows = 0;
    if (p.per_token && tile < total) {
      e = 0;  // the factor does not depend on the expert
      row0 = tile * 16;
      nrows = min(16, p.T - row0);
    } else if (tile < total) {
      int lo = 0, hi = p.E - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_ts[mid] <= tile) lo = mid;
        else hi = mid - 1;
      }
      e = lo;
      row0 = p.expert_offsets[lo] + (tile - s_ts[lo]) * 16;
      nrows = min(16, p.expert_offsets[lo + 1] - row0);
    }
    s_info[0] = e;
    s_info[1] = row0;
    s_info[2] = nrows;
    mbar_init(bar, 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  const int e = s_info[0], row0 = s_info[1], nrows = s_info[2];
  if (e < 0) return;
  if (tid < 16) {
    const bool in = tid < nrows;
    int a = -1;
    if (in && R > 0) {
      if (p.per_token) {  // same rule as the permute: out-of-range mappings mean "none"
        a = p.mapping[row0 + tid];
        if (a < -1 || a >= p.num_adapters) a = -1;
      } else {
        a = p.row_adapter[row0 + tid];
      }
    }
    s_adapter[tid] = a;
    s_src[tid] = in ? ((p.p2e != nullptr && !p.per_token) ? p.p2e[row0 + tid] / p.top_k : row0 + tid) : 0;
  }
  for (int i = tid; i < 16 * R; i += kShrinkThreads) s_u[i] = __float2bfloat16_rn(0.f);
  __syncthreads();

  // This CTA handles adapter slot ``ad`` of the tile: it computes u for the
  // tile's rows of that adapter and writes U columns [ad*r, ad*r + r) of
  // every row of the tile (zero for rows of other adapters).  Slot 0 also
  // copies the gathered rows.
  const int ad = static_cast<int>(blockIdx.y);
  bool present = false;
  if (R > 0 && p.U != nullptr) {
#pragma unroll
    for (int i = 0; i < 16; ++i) present |= (s_adapter[i] == ad);
  }
  // Row gather: slot 0's CTA copies each row from the staged tile.  (The
  // per-token mode copies after the permute, from global memory, below.)
  const bool do_gather = p.gathered != nullptr && !p.per_token && ad == 0;
  const int passes = (present || do_gather) ? 1 : 0;
  const int K = p.K;
  uint32_t parity = 0;
  const uint4 zero = make_uint4(0, 0, 0, 0);

  for (int pass = 0; pass < passes; ++pass) {
    const int a = present ? ad : -1;
    const __nv_bfloat16* Af =
        a >= 0 ? p.A + a * p.a_stride_adapter + static_cast<int64_t>(e) * p.a_stride_expert +
                     static_cast<int64_t>(rs) * R * K
               : nullptr;
    float acc[NT > 0 ? NT : 1][4];
#pragma unroll
    for (int nt = 0; nt < (NT > 0 ? NT : 1); ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;

    for (int kc0 = 0; kc0 < K; kc0 += KC) {
      const int cur = min(KC, K - kc0);
      if (warp == 0) {
        if (lane == 0) {
          const uint32_t bytes = static_cast<uint32_t>(nrows + (a >= 0 ? R : 0)) * cur * 2;
          mbar_arrive_expect_tx(bar, bytes);
        }
        __syncwarp();
        if (lane < nrows)
          bulk_load(Xs + lane * pitch, p.X + static_cast<size_t>(s_src[lane]) * K + kc0, cur * 2, bar);
        if (a >= 0)
          for (int i = lane; i < R; i += 32)
            bulk_load(Fs + i * pitch, Af + static_cast<size_t>(i) * K + kc0, cur * 2, bar);
      }
      // One thread waits with a time limit so that the decision is uniform;
      // then every thread observes the completed phase (data visibility).
      if (tid == 0) s_ok = mbar_wait(bar, parity, p.timeout_ns) ? 1 : 0;
      __syncthreads();
      if (!s_ok) {
        if (tid == 0) set_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
        return;
      }
      mbar_wait(bar, parity, p.timeout_ns);
      parity ^= 1;
      if (do_gather) {
        const int vpr = cur / 8;
        for (int v = tid; v < nrows * vpr; v += kShrinkThreads) {
          const int row = v / vpr, c = (v - row * vpr) * 8;
          const int dst = row0 + row;
          *reinterpret_cast<uint4*>(p.gathered + static_cast<size_t>(dst) * K + kc0 + c) =
              *reinterpret_cast<const uint4*>(Xs + row * pitch + c);
        }
      }
      if constexpr (NT > 0) {
       if (a >= 0) {
        const int nchunks = (cur + 31) / 32;
        for (int c = warp; c < nchunks; c += 8) {
          const int kk = c * 32 + t4 * 8;
          const bool kin = kk < cur;
          const uint4 xa = kin ? *reinterpret_cast<const uint4*>(Xs + g * pitch + kk) : zero;
          const uint4 xb = kin ? *reinterpret_cast<const uint4*>(Xs + (g + 8) * pitch + kk) : zero;
#pragma unroll
          for (int nt = 0; nt < (NT > 0 ? NT : 1); ++nt) {
            const uint4 f = kin ? *reinterpret_cast<const uint4*>(Fs + (nt * 8 + g) * pitch + kk) : zero;
            mma_m16n8k16_bf16(acc[nt], xa.x, xb.x, xa.y, xb.y, f.x, f.y);
            mma_m16n8k16_bf16(acc[nt], xa.z, xb.z, xa.w, xb.w, f.z, f.w);
          }
        }
       }
      }
      __syncthreads();  // shared tiles are reused by the next phase
    }
    if constexpr (NT > 0) {
     if (a >= 0) {
      float* red = s_red + warp * 16 * R;
#pragma unroll
      for (int nt = 0; nt < (NT > 0 ? NT : 1); ++nt) {
        const int col = nt * 8 + 2 * t4;
        red[g * R + col] = acc[nt][0];
        red[g * R + col + 1] = acc[nt][1];
        red[(g + 8) * R + col] = acc[nt][2];
        red[(g + 8) * R + col + 1] = acc[nt][3];
      }
      __syncthreads();
      for (int i = tid; i < 16 * R; i += kShrinkThreads) {
        if (s_adapter[i / R] != a) continue;
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) sum += s_red[w * 16 * R + i];
        s_u[i] = __float2bfloat16_rn(p.scaling[a] * sum);
      }
      __syncthreads();
     }
    }
  }
  if (p.per_token) {
    // From here on the permute's tables: wait for it, then read the
    // permuted rows of the tile's tokens once.
    pdl_wait();
    for (int i = tid; i < nrows * p.top_k; i += kShrinkThreads) s_dst[i] = p.e2p[row0 * p.top_k + i];
    __syncthreads();
    if (p.gathered != nullptr) {
      // The tile's (token, copy j) pairs q = token * top_k + j are shared out
      // over the C = gridDim.y * gridDim.z CTAs of the tile: CTA c copies
      // pairs c, c + C, ... from the source rows (just read, so in L2).
      const int C = static_cast<int>(gridDim.y * gridDim.z);
      const int c0 = ad + static_cast<int>(gridDim.y) * rs;
      const int npairs = nrows * p.top_k;
      const int mine = npairs > c0 ? (npairs - c0 + C - 1) / C : 0;
      const int vpr = K / 8;
      for (int v = tid; v < mine * vpr; v += kShrinkThreads) {
        const int i = v / vpr, c = (v - i * vpr) * 8;
        const int q = c0 + i * C;
        const int dst = s_dst[q];
        if (dst < 0) continue;  // slot not routed here (dropped id, another shard's expert)
        *reinterpret_cast<uint4*>(p.gathered + static_cast<size_t>(dst) * K + c) =
            __ldg(reinterpret_cast<const uint4*>(p.X + static_cast<size_t>(row0 + q / p.top_k) * K + c));
      }
    }
  }
  pdl_launch_dependents();

  if constexpr (NT > 0) {
   if (p.U != nullptr) {  // this adapter's columns (this slice) of every row of the tile
    const int ld = p.num_adapters * p.rank;
    constexpr int vec_per_row = R / 8;
    const int copies = p.per_token ? p.top_k : 1;  // every permuted row of the token
    for (int v = tid; v < nrows * copies * vec_per_row; v += kShrinkThreads) {
      const int rc = v / vec_per_row;
      const int c = (v - rc * vec_per_row) * 8;
      const int row = rc / copies;
      const int dst = p.per_token ? s_dst[rc] : row0 + row;
      if (dst < 0) continue;  // slot not routed here
      uint4 val = zero;
      if (s_adapter[row] == ad) val = *reinterpret_cast<const uint4*>(s_u + row * R + c);
      *reinterpret_cast<uint4*>(p.U + static_cast<size_t>(dst) * ld + ad * p.rank + rs * R + c) = val;
    }
   }
  }
}

// The largest phase (a multiple of 64) that fits the budget fixes the number
// of phases; the phases are then made equal, so that the shared memory of a
// CTA is no larger than that number of phases needs.
int shrink_chunk(int K, int rank, size_t budget) {
  if (shrink_smem_bytes(K, rank) <= budget) return K;
  int kc = 64;
  while (kc + 64 < K && shrink_smem_bytes(kc + 64, rank) <= budget) kc += 64;
  const int phases = (K + kc - 1) / kc;
  return ((K + phases - 1) / phases + 63) / 64 * 64;
}

// The per-token mode has few tiles (16 tokens each): a rank of 32 or more
// is split into 16-column slices, one CTA each, so that more CTAs share the
// factor reads.
static int gather_shrink_slices(const ShrinkParams& p) {
  return (p.per_token && p.U != nullptr && p.rank >= 32 && p.rank % 16 == 0) ? p.rank / 16 : 1;
}

int gather_shrink_cta_rank(const ShrinkParams& p) { return p.U != nullptr ? p.rank / gather_shrink_slices(p) : 0; }

size_t per_token_shrink_budget(const ShrinkParams& p, int sms, size_t smem_per_sm) {
  const int64_t ctas = static_cast<int64_t>((p.T + 15) / 16) * (p.U != nullptr ? p.num_adapters : 1) *
                       gather_shrink_slices(p);
  // Beyond four CTAs an SM the grid runs in waves whatever the phase size;
  // four then stay resident with phases of about 700 elements.
  const int64_t per_sm = std::min<int64_t>(4, std::max<int64_t>(1, (ctas + sms - 1) / sms));
  // 4 KB a CTA for its static shared memory and the per-block reservation.
  const int64_t fit = static_cast<int64_t>(smem_per_sm) / per_sm - 4096;
  return static_cast<size_t>(std::max<int64_t>(std::min<int64_t>(fit, 200 * 1024), 16 * 1024));
}

cudaError_t launch_gather_shrink(const ShrinkParams& p, int n_rows, cudaStream_t s) {
  if (n_rows == 0) return cudaSuccess;
  const int slices = gather_shrink_slices(p);
  const int NT = p.rank / 8 / slices;
  const int tiles = p.per_token ? (p.T + 15) / 16 : (n_rows + 15) / 16 + (p.E < n_rows ? p.E : n_rows);
  const dim3 grid(tiles, (NT > 0 && p.U != nullptr) ? p.num_adapters : 1, slices);
  const size_t smem = shrink_smem_bytes(p.kc, gather_shrink_cta_rank(p));
#define MOE_SHRINK_CASE(N)                                                                        \
  case N: {                                                                                       \
    cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(gather_shrink_kernel<N>), (int)smem); \
    if (err != cudaSuccess) return err;                                                           \
    return launch_pdl(gather_shrink_kernel<N>, grid, dim3(kShrinkThreads), smem, s, p);           \
  }
  switch (p.U != nullptr ? NT : 0) {  // no U: the gather alone
    MOE_SHRINK_CASE(0) MOE_SHRINK_CASE(1) MOE_SHRINK_CASE(2) MOE_SHRINK_CASE(3)
    MOE_SHRINK_CASE(4) MOE_SHRINK_CASE(5) MOE_SHRINK_CASE(6) MOE_SHRINK_CASE(7)
    MOE_SHRINK_CASE(8) MOE_SHRINK_CASE(9) MOE_SHRINK_CASE(10) MOE_SHRINK_CASE(11)
    MOE_SHRINK_CASE(12) MOE_SHRINK_CASE(13) MOE_SHRINK_CASE(14) MOE_SHRINK_CASE(15)
    MOE_SHRINK_CASE(16)
    default: return cudaErrorInvalidValue;
  }
#undef MOE_SHRINK_CASE
}

// ------------------------------------------------------ row-block variant
// For many rows (prefill).  One CTA per (kRowTile-row tile of one expert,
// adapter slot a), two threads per tile row.  The CTA takes the tile's rows of adapter a (slot 0 with a gather
// to do: all rows, for the copy) and streams K in 64-element chunks through
// a kRowStages-deep cp.async pipeline; warp w owns compacted rows
// [16w, 16w + 16) and keeps their u in registers for the whole K, so no
// cross-warp reduction is needed.  Every thread copies the same 16-byte
// column of the same four rows in every chunk, so its addresses are worked
// out once.  Shared tiles store each 128-byte row as
// eight 16-byte chunks, chunk j at position j ^ 4 (row & 1): the 8 lanes of
// a quarter-warp read rows g, g' of both parities and four chunks each, and
// land in 8 distinct bank groups.
// 64-row tiles and four stages: at prefill sizes (tens of thousands of rows)
// this gives every SM four resident CTAs with three chunks in flight each;
// 128-row tiles with three stages left the SMs latency-bound.
constexpr int kRowStages = 4;
constexpr int kRowTile = 64;
constexpr int kRowThreads = 2 * kRowTile;  // warp w owns compacted rows [16w, 16w + 16)
constexpr int kRowStride = kRowThreads / 8;  // rows between one thread's copy rows

int rows_shrink_tile() { return kRowTile; }

// At least 48 KB of shared memory per CTA, so that no more than four CTAs
// share an SM: at prefill sizes four per SM measured faster than five
// (gate_up shrink 40 against 47 us), the fifth adding L2 pressure rather
// than latency hiding.  The part above the tiles is unused.
constexpr size_t kRowMinSmem = 48 * 1024;

__host__ __device__ inline size_t rows_shrink_smem_bytes(int rank, int E) {
  const size_t need = static_cast<size_t>(kRowStages) * (kRowTile + rank) * 128 +
                      static_cast<size_t>(kRowTile) * rank * 2 + static_cast<size_t>(E + 1) * 4;
  return need > kRowMinSmem ? need : kRowMinSmem;
}

__device__ __forceinline__ int swz16(int row, int j) { return (j ^ ((row & 1) << 2)) * 16; }

template <int NT>
__global__ void __launch_bounds__(kRowThreads) rows_shrink_kernel(const ShrinkParams p) {
  constexpr int R = 8 * NT;
  constexpr int kXStage = kRowTile * 128;
  constexpr int kStage = kXStage + R * 128;
  extern __shared__ int4 rows_smem[];
  uint8_t* stages = reinterpret_cast<uint8_t*>(rows_smem);
  __nv_bfloat16* s_u = reinterpret_cast<__nv_bfloat16*>(stages + kRowStages * kStage);  // [kRowTile][R]
  int* s_ts = reinterpret_cast<int*>(s_u + kRowTile * R);                                // [E + 1]
  __shared__ int s_rows[kRowTile];  // tile row of compacted row i
  __shared__ int s_adp[kRowTile];   // adapter of tile row i
  __shared__ int s_warp_cnt[kRowThreads / 32];
  __shared__ int s_info[4];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int a = static_cast<int>(blockIdx.y);

  // tables_ready: the routing tables are complete at launch, so the tile,
  // its rows and the factor are worked out (L2 loads: no stale L1 line) and
  // the factor prefetched while the previous kernel, which writes X, drains.
  if (!p.tables_ready) pdl_wait();
  for (int i = tid; i <= p.E; i += kRowThreads) s_ts[i] = __ldcg(p.tile_start_rows + i);
  __syncthreads();
  if (tid == 0) {
    const int tile = blockIdx.x;
    int e = -1, row0 = 0, nrows = 0;
    if (tile < s_ts[p.E]) {
      int lo = 0, hi = p.E - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_ts[mid] <= tile) lo = mid;
        else hi = mid - 1;
      }
      e = lo;
      row0 = __ldcg(p.expert_offsets + lo) + (tile - s_ts[lo]) * kRowTile;
      nrows = min(kRowTile, __ldcg(p.expert_offsets + lo + 1) - row0);
    }
    s_info[0] = e;
    s_info[1] = row0;
    s_info[2] = nrows;
  }
  __syncthreads();
  const int e = s_info[0], row0 = s_info[1], nrows = s_info[2];
  if (e < 0) return;
  const bool lora = NT > 0 && p.U != nullptr;
  const bool do_gather = p.gathered != nullptr && a == 0;

  // Compact the rows this CTA loads, in tile order (block-wide ballot scan).
  bool take = false;
  if (tid < kRowTile) {
    const int ad = (tid < nrows && lora) ? __ldcg(p.row_adapter + row0 + tid) : -1;
    s_adp[tid] = ad;
    take = tid < nrows && (do_gather || ad == a);
  }
  const unsigned bal = __ballot_sync(0xFFFFFFFFu, take);
  if (lane == 0) s_warp_cnt[warp] = __popc(bal);
  __syncthreads();
  int before = 0, m = 0;
  for (int w = 0; w < kRowThreads / 32; ++w) {
    const int c = s_warp_cnt[w];
    if (w < warp) before += c;
    m += c;
  }
  if (take) s_rows[before + __popc(bal & ((1u << lane) - 1u))] = tid;
  __syncthreads();

  const int K = p.K;
  const int nchunks = (K + 63) / 64;
  const __nv_bfloat16* Af =
      lora ? p.A + a * p.a_stride_adapter + static_cast<int64_t>(e) * p.a_stride_expert : nullptr;
  const bool compute = lora && m > 0;
  if (p.tables_ready) {
    if (compute && warp == 0) {  // R rows of K: one contiguous block, in 16 KB pieces
      const uint32_t bytes = static_cast<uint32_t>(R) * K * 2;
      for (uint32_t off = lane * 16384u; off < bytes; off += 32u * 16384u)
        bulk_prefetch_l2(reinterpret_cast<const uint8_t*>(Af) + off, min(16384u, bytes - off));
    }
    pdl_wait();
  }

  // This thread's share of every chunk: column jc of compacted rows
  // (tid >> 3) + kRowStride q, and column jc of factor rows (tid >> 3) + kRowStride q.
  const int jc = tid & 7;
  const __nv_bfloat16* xsrc[4];
  __nv_bfloat16* gdst[4];
  uint32_t xoff[4];
  bool xval[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int i = (tid >> 3) + kRowStride * q;
    xval[q] = i < m;
    const int tr = xval[q] ? s_rows[i] : 0;
    const int src = p.p2e != nullptr ? p.p2e[row0 + tr] / p.top_k : row0 + tr;
    xsrc[q] = p.X + static_cast<size_t>(src) * K + jc * 8;
    gdst[q] = do_gather ? p.gathered + static_cast<size_t>(row0 + tr) * K + jc * 8 : nullptr;
    xoff[q] = static_cast<uint32_t>(i * 128 + swz16(i, jc));
  }
  constexpr int kFQ = (R + kRowStride - 1) / kRowStride;  // factor rows per thread
  const __nv_bfloat16* fsrc[kFQ > 0 ? kFQ : 1];
  uint32_t foff[kFQ > 0 ? kFQ : 1];
  bool fval[kFQ > 0 ? kFQ : 1];
#pragma unroll
  for (int q = 0; q < kFQ; ++q) {
    const int fr = (tid >> 3) + kRowStride * q;
    fval[q] = compute && fr < R;
    fsrc[q] = fval[q] ? Af + static_cast<size_t>(fr) * K + jc * 8 : p.X;
    foff[q] = static_cast<uint32_t>(kXStage + fr * 128 + swz16(fr, jc));
  }

  auto load_chunk = [&](int c, int st) {
    uint8_t* sx = stages + st * kStage;
    const int k0 = c * 64;
    const bool kval = k0 + jc * 8 < K;
#pragma unroll
    for (int q = 0; q < 4; ++q) cp_async_16(sx + xoff[q], xsrc[q] + (kval ? k0 : 0), xval[q] && kval);
#pragma unroll
    for (int q = 0; q < kFQ; ++q)
      if (fval[q]) cp_async_16(sx + foff[q], fsrc[q] + (kval ? k0 : 0), kval);
  };

  float acc[NT > 0 ? NT : 1][4];
#pragma unroll
  for (int nt = 0; nt < (NT > 0 ? NT : 1); ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;

  if (m > 0 && (compute || do_gather)) {
#pragma unroll
    for (int st = 0; st < kRowStages - 1; ++st) {
      if (st < nchunks) load_chunk(st, st);
      cp_async_commit();
    }
    for (int c = 0; c < nchunks; ++c) {
      cp_async_wait<kRowStages - 2>();
      __syncthreads();  // chunk c visible to all; stage (c - 1) % S free again
      {
        const int cn = c + kRowStages - 1;
        if (cn < nchunks) load_chunk(cn, cn % kRowStages);
        cp_async_commit();
      }
      const uint8_t* sx = stages + (c % kRowStages) * kStage;
      const int k0 = c * 64;
      if (do_gather && k0 + jc * 8 < K) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (xval[q]) *reinterpret_cast<uint4*>(gdst[q] + k0) = *reinterpret_cast<const uint4*>(sx + xoff[q]);
      }
      if constexpr (NT > 0) {
        if (compute && warp * 16 < m) {
          const uint8_t* sf = sx + kXStage;
          const int ra = warp * 16 + g, rb = ra + 8;
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
            const int j = c2 * 4 + t4;
            const uint4 xa = *reinterpret_cast<const uint4*>(sx + ra * 128 + swz16(ra, j));
            const uint4 xb = *reinterpret_cast<const uint4*>(sx + rb * 128 + swz16(rb, j));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const int f = nt * 8 + g;
              const uint4 fv = *reinterpret_cast<const uint4*>(sf + f * 128 + swz16(f, j));
              mma_m16n8k16_bf16(acc[nt], xa.x, xb.x, xa.y, xb.y, fv.x, fv.y);
              mma_m16n8k16_bf16(acc[nt], xa.z, xb.z, xa.w, xb.w, fv.z, fv.w);
            }
          }
        }
      }
    }
    cp_async_wait<0>();
  }
  pdl_launch_dependents();

  if constexpr (NT > 0) {
    if (p.U != nullptr) {
      // u of the compacted rows into s_u[tile row] (rows of adapter a only);
      // then columns [a r, a r + r) of every row of the tile: u or 0.
      for (int i = tid; i < kRowTile * R; i += kRowThreads) s_u[i] = __float2bfloat16_rn(0.f);
      __syncthreads();
      if (compute && warp * 16 < m) {
        const float sc = p.scaling[a];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int col = nt * 8 + 2 * t4;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int ci = warp * 16 + g + 8 * h;
            if (ci < m) {
              const int tr = s_rows[ci];
              if (s_adp[tr] == a) {
                s_u[tr * R + col] = __float2bfloat16_rn(sc * acc[nt][2 * h]);
                s_u[tr * R + col + 1] = __float2bfloat16_rn(sc * acc[nt][2 * h + 1]);
              }
            }
          }
        }
      }
      __syncthreads();
      const int ld = p.num_adapters * R;
      constexpr int vpr = R / 8;
      for (int v = tid; v < nrows * vpr; v += kRowThreads) {
        const int row = v / vpr, c = (v - row * vpr) * 8;
        *reinterpret_cast<uint4*>(p.U + static_cast<size_t>(row0 + row) * ld + a * R + c) =
            *reinterpret_cast<const uint4*>(s_u + row * R + c);
      }
    }
  }
}

cudaError_t launch_rows_shrink(const ShrinkParams& p, int n_rows, cudaStream_t s) {
  if (n_rows == 0) return cudaSuccess;
  const int NT = p.rank / 8;
  const int tiles = (n_rows + kRowTile - 1) / kRowTile + (p.E < n_rows ? p.E : n_rows);
  const dim3 grid(tiles, (NT > 0 && p.U != nullptr) ? p.num_adapters : 1);
  const size_t smem = rows_shrink_smem_bytes(p.U != nullptr ? p.rank : 0, p.E);
#define MOE_ROWS_CASE(N)                                                                          \
  case N: {                                                                                       \
    cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(rows_shrink_kernel<N>), (int)smem); \
    if (err != cudaSuccess) return err;                                                           \
    return launch_pdl(rows_shrink_kernel<N>, grid, dim3(kRowThreads), smem, s, p);             \
  }
  switch (p.U != nullptr ? NT : 0) {
    MOE_ROWS_CASE(0) MOE_ROWS_CASE(1) MOE_ROWS_CASE(2) MOE_ROWS_CASE(3)
    MOE_ROWS_CASE(4) MOE_ROWS_CASE(5) MOE_ROWS_CASE(6) MOE_ROWS_CASE(7)
    MOE_ROWS_CASE(8) MOE_ROWS_CASE(9) MOE_ROWS_CASE(10) MOE_ROWS_CASE(11)
    MOE_ROWS_CASE(12) MOE_ROWS_CASE(13) MOE_ROWS_CASE(14) MOE_ROWS_CASE(15)
    MOE_ROWS_CASE(16)
    default: return cudaErrorInvalidValue;
  }
#undef MOE_ROWS_CASE
}

}  // namespace moe
