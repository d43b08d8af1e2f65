// LoRA shrink: u = s * A[a, e] x for every permuted row, written as the
// one-hot operand of the expand.
//
// The shrink half of ``merged_experts_fused_moe_lora_add`` in Flow 1(A) and
// Flow 2 of "[WIP][LoRA] BF16 support for the experimental_sgl_trtllm
// MoE-LoRA path & lora expert_outer_shared" (yushengsu-thu/sglang#4): the
// gate_up call reads the hidden rows, the down call reads the activation
// output; in the shared-outer sub-mode the gate_up A factor is addressed by
// the adapter only (expert stride 0 here).
//
// Output layout: U[p, a*r + i] = bf16(s * (A[a, e(p)] X[p])_i) for the row's
// own adapter a, and 0 in every other column of the row (all zero for rows
// without an adapter).  The expert GEMM multiplies B[a, e] against the
// columns of adapter a only, so rows of other adapters contribute exactly 0.
//
// One CTA per 16-row tile of one expert (tile list from the permute scan);
// 8 warps split K, each with m16n8k16 mma.sync; partial sums meet in shared
// memory.  Loads use 16-byte vectors: lane (g, t) reads 8 consecutive K
// elements of rows g and g+8 and of factor row g of each 8-wide N tile, and
// uses them for two k16 steps, the same K positions on both operands.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

template <int NT>  // rank = 8 * NT
__global__ void __launch_bounds__(256) lora_shrink_kernel(const ShrinkParams p) {
  constexpr int R = 8 * NT;
  extern __shared__ float4 shrink_smem[];
  float* s_red = reinterpret_cast<float*>(shrink_smem);                  // [8][16][R]
  __nv_bfloat16* s_u = reinterpret_cast<__nv_bfloat16*>(s_red + 8 * 16 * R);  // [16][R]
  __shared__ int s_adapter[16];
  __shared__ int s_info[3];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;

  if (tid == 0) {
    const int tile = blockIdx.x;
    const int total = p.tile_start16[p.E];
    int e = -1, row0 = 0, nrows = 0;
    if (tile < total) {
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
  }
  __syncthreads();
  const int e = s_info[0], row0 = s_info[1], nrows = s_info[2];
  if (e < 0) return;
  if (tid < 16) s_adapter[tid] = tid < nrows ? p.row_adapter[row0 + tid] : -1;
  for (int i = tid; i < 16 * R; i += 256) s_u[i] = __float2bfloat16_rn(0.f);
  __syncthreads();

  uint64_t amask = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i)
    if (s_adapter[i] >= 0) amask |= 1ull << s_adapter[i];

  const int K = p.K;
  const int nchunks = (K + 31) / 32;
  const __nv_bfloat16* xa_row = p.X + static_cast<size_t>(row0 + g) * K;
  const __nv_bfloat16* xb_row = p.X + static_cast<size_t>(row0 + g + 8) * K;
  const bool va = g < nrows, vb = g + 8 < nrows;
  const uint4 zero = make_uint4(0, 0, 0, 0);

  while (amask) {
    const int a = __ffsll(static_cast<long long>(amask)) - 1;
    amask &= amask - 1;
    const __nv_bfloat16* Af = p.A + a * p.a_stride_adapter + static_cast<int64_t>(e) * p.a_stride_expert;
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;

    for (int c = warp; c < nchunks; c += 8) {
      const int kk = c * 32 + t4 * 8;
      const bool kin = kk < K;
      const uint4 xa = (kin && va) ? __ldg(reinterpret_cast<const uint4*>(xa_row + kk)) : zero;
      const uint4 xb = (kin && vb) ? __ldg(reinterpret_cast<const uint4*>(xb_row + kk)) : zero;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint4 f =
            kin ? __ldg(reinterpret_cast<const uint4*>(Af + static_cast<size_t>(nt * 8 + g) * K + kk))
                : zero;
        mma_m16n8k16_bf16(acc[nt], xa.x, xb.x, xa.y, xb.y, f.x, f.y);
        mma_m16n8k16_bf16(acc[nt], xa.z, xb.z, xa.w, xb.w, f.z, f.w);
      }
    }
    // fragment (row g / g+8, columns 8nt + 2t4 + {0,1}) -> shared partials
    float* red = s_red + warp * 16 * R;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int col = nt * 8 + 2 * t4;
      red[g * R + col] = acc[nt][0];
      red[g * R + col + 1] = acc[nt][1];
      red[(g + 8) * R + col] = acc[nt][2];
      red[(g + 8) * R + col + 1] = acc[nt][3];
    }
    __syncthreads();
    for (int i = tid; i < 16 * R; i += 256) {
      const int row = i / R;
      if (s_adapter[row] != a) continue;
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) sum += s_red[w * 16 * R + i];
      s_u[i] = __float2bfloat16_rn(p.scaling * sum);
    }
    __syncthreads();
  }

  // Whole rows of U: the own adapter's r values, zeros elsewhere.
  const int ld = p.num_adapters * R;
  const int vec_per_row = ld / 8;
  for (int v = tid; v < nrows * vec_per_row; v += 256) {
    const int row = v / vec_per_row;
    const int col = (v - row * vec_per_row) * 8;
    const int a = s_adapter[row];
    uint4 val = zero;
    if (a >= 0 && col >= a * R && col < (a + 1) * R)
      val = *reinterpret_cast<const uint4*>(s_u + row * R + (col - a * R));
    *reinterpret_cast<uint4*>(p.U + static_cast<size_t>(row0 + row) * ld + col) = val;
  }
}

cudaError_t launch_lora_shrink(const ShrinkParams& p, int n_rows, cudaStream_t s) {
  if (n_rows == 0) return cudaSuccess;
  const int NT = p.rank / 8;
  const int grid = (n_rows + 15) / 16 + (p.E < n_rows ? p.E : n_rows);
  const size_t smem = static_cast<size_t>(8 * 16 * p.rank) * 4 + static_cast<size_t>(16 * p.rank) * 2;
#define MOE_SHRINK_CASE(N)                                                                        \
  case N: {                                                                                       \
    cudaError_t err = cudaFuncSetAttribute(lora_shrink_kernel<N>,                                 \
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
    if (err != cudaSuccess) return err;                                                           \
    lora_shrink_kernel<N><<<grid, 256, smem, s>>>(p);                                             \
    return cudaGetLastError();                                                                    \
  }
  switch (NT) {
    MOE_SHRINK_CASE(1) MOE_SHRINK_CASE(2) MOE_SHRINK_CASE(3) MOE_SHRINK_CASE(4)
    MOE_SHRINK_CASE(5) MOE_SHRINK_CASE(6) MOE_SHRINK_CASE(7) MOE_SHRINK_CASE(8)
    MOE_SHRINK_CASE(9) MOE_SHRINK_CASE(10) MOE_SHRINK_CASE(11) MOE_SHRINK_CASE(12)
    MOE_SHRINK_CASE(13) MOE_SHRINK_CASE(14) MOE_SHRINK_CASE(15) MOE_SHRINK_CASE(16)
    default: return cudaErrorInvalidValue;
  }
#undef MOE_SHRINK_CASE
}

}  // namespace moe
