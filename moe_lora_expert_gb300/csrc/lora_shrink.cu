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

template <int NT>  // rank = 8 * NT (NT = 0: gather only)
__global__ void __launch_bounds__(kShrinkThreads) gather_shrink_kernel(const ShrinkParams p) {
  constexpr int R = 8 * NT;
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
  __shared__ int s_info[3];
  __shared__ int s_ok;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;

  pdl_wait();
  if (tid == 0) {
    const int tile = blockIdx.x;
    const int total = p.per_token ? (p.T + 15) / 16 : p.tile_start16[p.E];
    int e = -1, row0 = 0, nrows = 0;
    if (p.per_token && tile < total) {
      e = 0;  // the factor does not depend on the expert
      row0 = tile * 16;
      nrows = min(16, p.T - row0);
    } else if (tile < total) {
      int lo = 0, hi = p.E - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.tile_start16[mid] <= tile) lo = mid;
        else hi = mid - 1;
      }
      e = lo;
      row0 = p.expert_offsets[lo] + (tile - p.tile_start16[lo]) * 16;
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
  const bool do_gather = p.gathered != nullptr && ad == 0;
  const int passes = (present || do_gather) ? 1 : 0;
  const int K = p.K;
  uint32_t parity = 0;
  const uint4 zero = make_uint4(0, 0, 0, 0);

  for (int pass = 0; pass < passes; ++pass) {
    const int a = present ? ad : -1;
    const __nv_bfloat16* Af =
        a >= 0 ? p.A + a * p.a_stride_adapter + static_cast<int64_t>(e) * p.a_stride_expert : nullptr;
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
        const int copies = p.per_token ? p.top_k : 1;  // every permuted row of the token
        for (int v = tid; v < nrows * copies * vpr; v += kShrinkThreads) {
          const int rc = v / vpr, c = (v - rc * vpr) * 8;
          const int row = rc / copies, j = rc - row * copies;
          const int dst = p.per_token ? p.e2p[(row0 + row) * p.top_k + j] : row0 + row;
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
  pdl_launch_dependents();

  if constexpr (NT > 0) {
   if (p.U != nullptr) {  // this adapter's r columns of every row of the tile
    const int ld = p.num_adapters * R;
    constexpr int vec_per_row = R / 8;
    const int copies = p.per_token ? p.top_k : 1;  // every permuted row of the token
    for (int v = tid; v < nrows * copies * vec_per_row; v += kShrinkThreads) {
      const int rc = v / vec_per_row;
      const int c = (v - rc * vec_per_row) * 8;
      const int row = rc / copies, j = rc - row * copies;
      const int dst = p.per_token ? p.e2p[(row0 + row) * p.top_k + j] : row0 + row;
      uint4 val = zero;
      if (s_adapter[row] == ad) val = *reinterpret_cast<const uint4*>(s_u + row * R + c);
      *reinterpret_cast<uint4*>(p.U + static_cast<size_t>(dst) * ld + ad * R + c) = val;
    }
   }
  }
}

int shrink_chunk(int K, int rank, size_t budget) {
  if (shrink_smem_bytes(K, rank) <= budget) return K;
  int kc = 64;
  while (kc + 64 < K && shrink_smem_bytes(kc + 64, rank) <= budget) kc += 64;
  return kc;
}

size_t shrink_launch_smem(const ShrinkParams& p) { return shrink_smem_bytes(p.kc, p.rank); }

cudaError_t launch_gather_shrink(const ShrinkParams& p, int n_rows, cudaStream_t s) {
  if (n_rows == 0) return cudaSuccess;
  const int NT = p.rank / 8;
  const int tiles = p.per_token ? (p.T + 15) / 16 : (n_rows + 15) / 16 + (p.E < n_rows ? p.E : n_rows);
  const dim3 grid(tiles, (NT > 0 && p.U != nullptr) ? p.num_adapters : 1);
  const size_t smem = shrink_smem_bytes(p.kc, p.rank);
#define MOE_SHRINK_CASE(N)                                                                        \
  case N: {                                                                                       \
    cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(gather_shrink_kernel<N>), (int)smem); \
    if (err != cudaSuccess) return err;                                                           \
    return launch_pdl(gather_shrink_kernel<N>, grid, dim3(kShrinkThreads), smem, s, p);           \
  }
  switch (NT) {
    MOE_SHRINK_CASE(0) MOE_SHRINK_CASE(1) MOE_SHRINK_CASE(2) MOE_SHRINK_CASE(3)
    MOE_SHRINK_CASE(4) MOE_SHRINK_CASE(5) MOE_SHRINK_CASE(6) MOE_SHRINK_CASE(7)
    MOE_SHRINK_CASE(8) MOE_SHRINK_CASE(9) MOE_SHRINK_CASE(10) MOE_SHRINK_CASE(11)
    MOE_SHRINK_CASE(12) MOE_SHRINK_CASE(13) MOE_SHRINK_CASE(14) MOE_SHRINK_CASE(15)
    MOE_SHRINK_CASE(16)
    default: return cudaErrorInvalidValue;
  }
#undef MOE_SHRINK_CASE
}

}  // namespace moe
