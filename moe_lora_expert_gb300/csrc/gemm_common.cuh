// Device helpers shared by the expert GEMM kernels (bf16 and FP8): work-unit
// decoding, the per-tile adapter mask, bounded barrier waits with their
// error reporting, and the TMA loads of weight and LoRA-factor blocks.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/moe_lora.h"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

constexpr unsigned kFullMask = 0xFFFFFFFFu;

struct Work {
  int e, fb, row0, nrows;
};

// Work unit u = (token tile, feature-block group).  Each CTA of a cluster of
// CL (a CTA pair: CL = 2) takes feature block group * CL + its rank, so the
// two CTAs of a pair work on the same token tile at the same time.
template <int BN>
__device__ __forceinline__ Work decode_work(int u, int crank, int CL, const int* s_off,
                                            const int* s_ts, int E, int FBg) {
  Work wk;
  const int tile = u / FBg;
  wk.fb = (u - tile * FBg) * CL + crank;
  int lo = 0, hi = E - 1;
  while (lo < hi) {  // largest e with s_ts[e] <= tile
    const int mid = (lo + hi + 1) >> 1;
    if (s_ts[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  wk.e = lo;
  wk.row0 = s_off[lo] + (tile - s_ts[lo]) * BN;
  wk.nrows = min(BN, s_off[lo + 1] - wk.row0);
  return wk;
}

// How many of the persistent grid's pmax CTAs (or clusters) take work units,
// given u units dealt round robin.  Every full round streams one unit per
// working CTA; the last round holds the u mod P leftover units, and a few
// CTAs alone cannot pull the memory bandwidth that all of them share (each
// is limited by the bytes its ring keeps in flight; about 70% of the grid
// saturates it).  In units of one unit's bytes at full bandwidth the time
// is (rounds - 1) P + max(fill, 0.7 pmax); the smallest over P in
// [3/4 pmax, pmax] is taken (the largest P on ties).  The CTAs beyond it
// take no units; they still join the in-kernel row passes.  The candidates
// are scored one per thread and meet in *s_key, which thread 0 set to ~0
// before the CTA's last barrier; every thread of the CTA calls this (it
// holds a barrier when u > pmax).
__device__ __forceinline__ int balanced_grid(int u, int pmax, unsigned long long* s_key) {
  if (u <= pmax) return pmax;  // one round
  const int psat = (pmax * 7) / 10;
  const int ncand = pmax - (3 * pmax + 3) / 4 + 1;
  for (int c = threadIdx.x; c < ncand; c += blockDim.x) {
    const int P = pmax - c;
    const int rounds = (u + P - 1) / P;
    const int fill = u - (rounds - 1) * P;
    const unsigned long long t =
        static_cast<unsigned long long>(rounds - 1) * P + static_cast<unsigned long long>(fill > psat ? fill : psat);
    atomicMin(s_key, (t << 20) | static_cast<unsigned long long>(c));
  }
  __syncthreads();
  return pmax - static_cast<int>(*s_key & 0xFFFFFull);
}

// The adapter mask of a token tile: OR of (1 << adapter) over its rows,
// computed by a whole warp.  The loads of a tile's (at most BN) row adapters
// are issued together, BN / 32 per lane, so the mask costs one round trip to
// L2; load_tile_adapters and reduce_tile_adapters split it so that the loads
// can be in flight while the warp does other work.
template <int BN>
struct TileAdapters {
  int v[(BN + 31) / 32];
};

template <int BN>
__device__ __forceinline__ void load_tile_adapters(const int32_t* row_adapter, int row0, int nrows, int lane,
                                                   TileAdapters<BN>& t) {
#pragma unroll
  for (int i = 0; i < (BN + 31) / 32; ++i) {
    const int r = lane + 32 * i;
    t.v[i] = r < nrows ? __ldcg(row_adapter + row0 + r) : -1;
  }
}

template <int BN>
__device__ __forceinline__ uint64_t reduce_tile_adapters(const TileAdapters<BN>& t) {
  uint64_t m = 0;
#pragma unroll
  for (int i = 0; i < (BN + 31) / 32; ++i)
    if (t.v[i] >= 0) m |= 1ull << t.v[i];
  const uint32_t lo = __reduce_or_sync(kFullMask, static_cast<uint32_t>(m));
  const uint32_t hi = __reduce_or_sync(kFullMask, static_cast<uint32_t>(m >> 32));
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

template <int BN>
__device__ __forceinline__ uint64_t tile_adapter_mask(const int32_t* row_adapter, int row0, int nrows,
                                                      int lane) {
  TileAdapters<BN> t;
  load_tile_adapters<BN>(row_adapter, row0, nrows, lane, t);
  return reduce_tile_adapters<BN>(t);
}

// Bounded wait that also gives up as soon as another role raised the abort flag.
// CLUSTER: acquire at cluster scope (arrivals come from the peer CTA too).
template <bool CLUSTER = false>
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                              volatile int* abort_flag) {
  const uint32_t a = smem_u32(bar);
  auto probe = [&]() { return CLUSTER ? mbar_try_wait_cluster(a, parity) : mbar_try_wait(a, parity); };
  if (probe()) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (probe()) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ void raise_timeout(int* status, volatile int* abort_flag) {
  set_status(status, MOE_ERR_DEVICE_TIMEOUT);
  *abort_flag = 1;
}

// As raise_timeout; the first error also records where in the status detail
// words: [1] = the wait (kWait*), [2] = (CTA << 8) | warp, [3] = (unit << 16)
// | (K block << 4) | ring stage.
enum WaitSite {
  kWaitProducerW8 = 1, kWaitProducer = 2, kWaitMmaAccEmpty = 4, kWaitMmaFull = 5,
  kWaitMmaFull8 = 6, kWaitEpilogue = 7, kWaitConvEmpty = 8, kWaitConvFull8 = 9,
  kWaitDrainProducer = 10, kWaitDrainProducerW8 = 11, kWaitDrainConv = 12, kWaitDrainMma = 13,
  kWaitShrinkFlag = 14
};

// A teardown wait that ran out: the status and its place, no abort (the
// roles have left their loops already).
__device__ __forceinline__ void note_drain_timeout(int* status, int site, int stage) {
  if (status != nullptr && atomicCAS(status, 0, MOE_ERR_DEVICE_TIMEOUT) == 0) {
    status[1] = site;
    status[2] = static_cast<int>((blockIdx.x << 8) | (threadIdx.x >> 5));
    status[3] = stage & 15;
  }
}
__device__ __forceinline__ void raise_timeout_at(int* status, volatile int* abort_flag, int site, int unit,
                                                 int blk, int stage) {
  if (status != nullptr && atomicCAS(status, 0, MOE_ERR_DEVICE_TIMEOUT) == 0) {
    status[1] = site;
    status[2] = static_cast<int>((blockIdx.x << 8) | (threadIdx.x >> 5));
    status[3] = (unit << 16) | ((blk & 0xFFF) << 4) | (stage & 15);
  }
  *abort_flag = 1;
}

// Weight-side (A operand) loads of one K block: 128 rows of the feature block.
// gate_up: the map views w13 so that one box (or four, see the host code)
// brings gate rows 64 fb + 16q + (0..15) to smem rows 32q + (0..15) and the
// matching up rows to smem rows 32q + 16 + (0..15), q = 0..3.
// PAIR: the bytes complete on the pair leader's barrier, ``cbar`` (a
// shared::cluster address); otherwise on this CTA's ``bar``.
template <bool PAIR>
__device__ __forceinline__ void load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, uint32_t cbar,
                                        int c0, int c1, uint64_t pol) {
  if constexpr (PAIR) tma_load_2d_pair(dst, map, cbar, c0, c1, pol);
  else tma_load_2d(dst, map, bar, c0, c1, pol);
}

// ESZ: bytes per weight element (2 bf16, 1 fp8): the smem offset between
// the four 16-row boxes of the 3-D gate_up view.
template <int MODE, bool PAIR, int ESZ = 2>
__device__ __forceinline__ void load_weight_block(uint8_t* sA, const CUtensorMap* map,
                                                  uint64_t* bar, uint32_t cbar, int kc, int e, int fb,
                                                  int rows_per_expert, int gu_single_box,
                                                  uint64_t pol) {
  if (MODE == kGateUp) {
    if (gu_single_box) {
      // map dims {H, 16 rows, 2 halves, I/16 groups, E}
      if constexpr (PAIR) tma_load_5d_pair(sA, map, cbar, kc, 0, 0, fb * 4, e, pol);
      else tma_load_5d(sA, map, bar, kc, 0, 0, fb * 4, e, pol);
    } else {
      // map dims {H, I, 2E}, box {64, 16, 2}
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if constexpr (PAIR) tma_load_3d_pair(sA + q * 2048 * ESZ, map, cbar, kc, fb * 64 + q * 16, 2 * e, pol);
        else tma_load_3d(sA + q * 2048 * ESZ, map, bar, kc, fb * 64 + q * 16, 2 * e, pol);
      }
    }
  } else {
    load_2d<PAIR>(sA, map, bar, cbar, kc, e * rows_per_expert + fb * 128, pol);
  }
}

// LoRA B-factor (A operand of the expand) loads: same row arrangement, from
// the 2-D map over all factor rows (box {64, 16} for gate_up, {64, 128} down).
template <int MODE, bool PAIR>
__device__ __forceinline__ void load_lora_b_block(uint8_t* sA, const CUtensorMap* map,
                                                  uint64_t* bar, uint32_t cbar, int kc, int64_t row_base,
                                                  int fb, int n_feat, uint64_t pol) {
  if (MODE == kGateUp) {
#pragma unroll
    for (int bx = 0; bx < 8; ++bx) {
      const int q = bx >> 1, up = bx & 1;
      const int64_t row = row_base + static_cast<int64_t>(up) * n_feat + fb * 64 + q * 16;
      load_2d<PAIR>(sA + bx * 2048, map, bar, cbar, kc, static_cast<int>(row), pol);
    }
  } else {
    load_2d<PAIR>(sA, map, bar, cbar, kc, static_cast<int>(row_base + fb * 128), pol);
  }
}

// The LoRA shrink of the permuted rows, by the four epilogue warps (ew =
// 0..3) before their first accumulator (GemmParams::fuse_shrink).  Rows are
// claimed one at a time from p.row_counter (thread 0 claims the next row
// while the current one is computed), so only CTAs that are running take
// rows: a producer that waits for a tile waits on rows that running CTAs,
// its own included, finish without waiting on anything.  For row p with adapter
// a = row_adapter[p] >= 0, su[p, a r + i] = bf16(s_a sum_k A[a, e][i][k]
// sx[p][k]) for i < r; every other column of the row is zero.  The 128
// threads split K in 8-element pieces (thread j takes k = 8 j + 1024 m), sum
// their pieces for 8 outputs at a time, reduce across each warp by shuffles
// and across the four warps in shared memory (s_red, 4 x 32 floats).  Each
// finished row adds one to the flag of its token tile (release, after a
// proxy fence that makes the row visible to other CTAs' TMA reads); a tile
// is complete when its flag equals its row count.  With p.gather_src the
// pass first copies the row's token vector from gather_src (the hidden row
// of its slot) into sx, so the gather needs no kernel of its own; with sx
// null it reads the row from gather_src and copies nothing.
template <int BN>
__device__ void shrink_rows_in_gemm(const GemmParams& p, const int* s_off, const int* s_ts, int ew,
                                    int lane, float* s_red) {
  const int R = p.rank, ld = p.num_adapters * p.rank, K = p.K;
  const int tid = ew * 32 + lane;
  const int nrows_all = s_off[p.E];
  volatile int* s_row = reinterpret_cast<volatile int*>(s_red + 128);  // the claimed row
  int next = tid == 0 ? atomicAdd(p.row_counter, 1) : 0;
  while (true) {
    if (tid == 0) *s_row = next;
    named_barrier_sync(1, 128);  // the claimed row is visible to the four warps
    const int prow = *s_row;
    if (prow >= nrows_all) break;
    if (tid == 0) next = atomicAdd(p.row_counter, 1);  // in flight while this row is computed
    int lo = 0, hi = p.E - 1;  // expert of the row: largest e with s_off[e] <= prow
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_off[mid] <= prow) lo = mid;
      else hi = mid - 1;
    }
    const int e = lo;
    const int tile = s_ts[e] + (prow - s_off[e]) / BN;
    const int a = __ldcg(p.row_adapter + prow);
    __nv_bfloat16* urow = p.su + static_cast<size_t>(prow) * ld;
    const __nv_bfloat16* x = p.sx + static_cast<size_t>(prow) * K;
    if (p.gather_src != nullptr) {
      x = p.gather_src + static_cast<size_t>(__ldcg(p.gather_map + prow) / p.gather_div) * K;
      if (p.sx != nullptr) {  // the row copy (null: the rows are only read)
        __nv_bfloat16* dst = const_cast<__nv_bfloat16*>(p.sx) + static_cast<size_t>(prow) * K;
        for (int k = tid * 8; k < K; k += 128 * 8)
          *reinterpret_cast<uint4*>(dst + k) = __ldg(reinterpret_cast<const uint4*>(x + k));
      }
    }
    // the other adapters' columns: zero (8 columns per store)
    for (int c = tid * 8; c < ld; c += 128 * 8)
      if (a < 0 || c / R != a) *reinterpret_cast<uint4*>(urow + c) = make_uint4(0, 0, 0, 0);
    if (a >= 0) {  // uniform over the CTA
      const __nv_bfloat16* A = p.sa + a * p.sa_stride_adapter + static_cast<int64_t>(e) * p.sa_stride_expert;
      for (int i0 = 0; i0 < R; i0 += 8) {
        float acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = 0.f;
        for (int k = tid * 8; k < K; k += 128 * 8) {
          const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x + k));
          const __nv_bfloat162* x2 = reinterpret_cast<const __nv_bfloat162*>(&xv);
          float xf[8];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const float2 f = __bfloat1622float2(x2[h]);
            xf[2 * h] = f.x;
            xf[2 * h + 1] = f.y;
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint4 av = __ldg(reinterpret_cast<const uint4*>(A + static_cast<size_t>(i0 + q) * K + k));
            const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&av);
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const float2 f = __bfloat1622float2(a2[h]);
              acc[q] = fmaf(f.x, xf[2 * h], acc[q]);
              acc[q] = fmaf(f.y, xf[2 * h + 1], acc[q]);
            }
          }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) acc[q] += __shfl_xor_sync(kFullMask, acc[q], off);
        }
        if (lane == 0) {
#pragma unroll
          for (int q = 0; q < 8; ++q) s_red[ew * 32 + i0 + q] = acc[q];
        }
      }
      named_barrier_sync(1, 128);  // every warp's partial sums of this row
      if (ew == 0 && lane < R)
        urow[a * R + lane] = __float2bfloat16_rn(
            p.sscale[a] * (s_red[lane] + s_red[32 + lane] + s_red[64 + lane] + s_red[96 + lane]));
    }
    fence_proxy_async_global();
    named_barrier_sync(1, 128);  // the row is written; s_red is free again
    if (tid == 0 && !(p.debug_hold_row && prow == 0)) {
      __threadfence();
      red_release_gpu_add(p.tile_flags + tile, 1);
    }
  }
  named_barrier_sync(1, 128);  // every warp has read *s_row: the staging tiles are free
}

// Bounded wait until ``count`` rows of a token tile are published by the
// in-kernel pass; then a proxy fence orders the TMA reads of them after it.
__device__ __forceinline__ bool wait_tile_rows(const int* flag, int count, uint64_t limit_ns,
                                               volatile int* abort_flag) {
  const uint64_t t0 = global_timer_ns();
  while (ld_acquire_gpu(flag) < count)
    if (*abort_flag || global_timer_ns() - t0 > limit_ns) return false;
  fence_proxy_async_global();
  return true;
}

}  // namespace moe
