// The FP8 (W8A8) half of the routed MoE-LoRA forward: the per-token-group
// activation quantizer and the grouped expert GEMMs on e4m3 weights and
// e4m3 activations.
//
// "[WIP][LoRA] BF16 support for the experimental_sgl_trtllm MoE-LoRA path &
// lora expert_outer_shared" (yushengsu-thu/sglang#4), Flow 1(A), draws the
// bf16 path as the FP8 one without two steps: a ``per_token_group_quant_fp8``
// of the hidden input before the gate_up GEMM and a post-activation quant
// before the down GEMM.  Their arithmetic is read as (per row and group of
// 128 consecutive columns, float32): scale = max(amax, 1e-10) / 448, code =
// e4m3(x / scale) rounded to nearest even and saturated at +-448; the
// activation is quantized from its float32 value; the LoRA deltas read the
// unquantized hidden row and activation.  Expert weights are e4m3 with one
// float32 scale per 128 x 128 block of (output rows, K).
//
// GEMM: as the bf16 kernel (swap AB: M = 128 weight rows, N = the token
// tile, TMEM accumulators, TMA with 128-byte swizzle), but every 128-K block
// is one ring stage of raw e4m3 weights and e4m3 token rows (128-byte rows,
// the same geometry as a 64-K bf16 block) multiplied by four
// tcgen05.mma.kind::f8f6f4 (K = 32 each) into a fresh TMEM partial.  The
// scales differ per weight row block, per token and per 128-K block, so the
// epilogue warps promote each partial: acc[col] += partial[col] *
// wscale[row block, kb] * xscale[token, kb], in registers, while the MMA
// fills the next partial slots.  The LoRA expand blocks stay bf16
// (kind::f16, B factor against the bf16 one-hot U) and are added unscaled.
// After the last block the epilogue applies SwiGLU (gate_up; the float32
// activation goes out for the post-activation quant) or stores y (down).
//
// Roles (192 threads): warp 0 = TMA producer, warp 1 = MMA issuer and TMEM
// owner, warps 2..5 = promotion + epilogue (TMEM lane quadrant = warp % 4).
// Persistent grid, one CTA per token tile unit.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/moe_lora.h"
#include "gemm_common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

// ------------------------------------------------------------- quantizer
// One warp per (row, 128-column group): four consecutive columns per lane.
__global__ void __launch_bounds__(256) quant_groups_kernel(const QuantParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const int G = (p.K + kActGroup - 1) / kActGroup;
  const int64_t task = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (task >= static_cast<int64_t>(p.rows) * G) return;
  const int lane = threadIdx.x & 31;
  const int row = static_cast<int>(task / G), g = static_cast<int>(task % G);
  const int k = g * kActGroup + 4 * lane;
  const bool in = k < p.K;  // K % 16 == 0: a lane's four columns are all in or all out
  int src = row;
  if (p.row_map != nullptr) {
    const int m = __ldg(p.row_map + row);
    src = m >= 0 ? m / p.map_div : -1;
  }
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  if (in && src >= 0) {
    if (p.x_f32) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p.x) +
                                                               static_cast<size_t>(src) * p.K + k));
      v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
    } else {
      const uint2 b = __ldg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(p.x) +
                                                             static_cast<size_t>(src) * p.K + k));
      const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&b.x));
      const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&b.y));
      v[0] = lo.x; v[1] = lo.y; v[2] = hi.x; v[3] = hi.y;
    }
  }
  // |x| of non-negative floats orders like their bit patterns
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) m = max(m, __float_as_uint(fabsf(v[i])));
  m = __reduce_max_sync(kFullMask, m);
  const float scale = __fdiv_rn(fmaxf(__uint_as_float(m), kActEps), kE4m3Max);
  if (in) {
    const uint32_t c01 = cvt_e4m3x2(__fdiv_rn(v[0], scale), __fdiv_rn(v[1], scale));
    const uint32_t c23 = cvt_e4m3x2(__fdiv_rn(v[2], scale), __fdiv_rn(v[3], scale));
    *reinterpret_cast<uint32_t*>(p.codes + static_cast<size_t>(row) * p.K + k) = c01 | (c23 << 16);
    if (p.copy != nullptr) {
      uint2 o;
      *reinterpret_cast<__nv_bfloat162*>(&o.x) = __floats2bfloat162_rn(v[0], v[1]);
      *reinterpret_cast<__nv_bfloat162*>(&o.y) = __floats2bfloat162_rn(v[2], v[3]);
      *reinterpret_cast<uint2*>(p.copy + static_cast<size_t>(row) * p.K + k) = o;
    }
  }
  if (lane == 0) p.scales[static_cast<size_t>(row) * G + g] = scale;
}

cudaError_t launch_quant_groups(const QuantParams& p, cudaStream_t s) {
  if (p.rows == 0) return cudaSuccess;
  const int64_t tasks = static_cast<int64_t>(p.rows) * ((p.K + kActGroup - 1) / kActGroup);
  const int64_t blocks = (tasks + 7) / 8;
  if (blocks >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  return launch_pdl(quant_groups_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, p);
}

// ------------------------------------------------------------------ GEMM
template <int BN>
struct Fp8Cfg {
  static constexpr int kCtasPerSm = BN <= 64 ? 2 : 1;
  static constexpr int kThreads = 192;
  static constexpr int kStageBudget = BN <= 64 ? 96 * 1024 : 200 * 1024;
  static constexpr int kABytes = 128 * 128;  // 128 rows x 128 B: 128 e4m3 or 64 bf16 of K
  static constexpr int kBBytes = BN * 128;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStagesRaw = kStageBudget / kStageBytes;
  static constexpr int kStages = kStagesRaw > 16 ? 16 : kStagesRaw;
  // TMEM partial slots of BN columns (a power-of-two allocation; two CTAs
  // of narrow tiles share an SM's 512 columns).  16-wide tiles take 16, so
  // the MMA can run two units of the down GEMM ahead of the epilogue warps
  // while they do the in-kernel shrink pass.
  static constexpr int kSlots = BN <= 16 ? 16 : (BN <= 32 ? 8 : 4);
  static constexpr int kTmemCols = kSlots * BN < 32 ? 32 : kSlots * BN;
  static constexpr int kMetaBytes = 512;
  static constexpr int kTableBytes = 2 * (MOE_MAX_EXPERTS + 1) * 4;
  static constexpr int kEpiOffset = (kMetaBytes + kTableBytes + 15) / 16 * 16;
  static constexpr int kEpiBytes = 4 * 1024;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kEpiOffset + kEpiBytes;
  static_assert((2 * kStages + 2 * kSlots + 2) * 8 + 16 <= kMetaBytes, "barriers, TMEM slot, flag, key fit");
  static_assert(kCtasPerSm * (kSmemBytes + 1024) <= 233472, "the CTAs of an SM fit its shared memory");
  static_assert(kCtasPerSm * kTmemCols <= 512, "the CTAs of an SM fit its tensor memory");
};

template <int BN, int MODE>
__global__ void __launch_bounds__(Fp8Cfg<BN>::kThreads, Fp8Cfg<BN>::kCtasPerSm)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                    const __grid_constant__ CUtensorMap tm_lb, const __grid_constant__ CUtensorMap tm_lu,
                    const GemmParams p) {
  using C = Fp8Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* meta = smem + C::kStages * C::kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(meta);
  uint64_t* empty = full + C::kStages;
  uint64_t* pfull = empty + C::kStages;
  uint64_t* pempty = pfull + C::kSlots;
  uint64_t* drain = pempty + C::kSlots;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  unsigned long long* s_grid_key = reinterpret_cast<unsigned long long*>(tmem_slot + 2);
  int* s_off = reinterpret_cast<int*>(meta + C::kMetaBytes);
  int* s_ts = s_off + (MOE_MAX_EXPERTS + 1);
  uint8_t* s_epi = meta + C::kEpiOffset;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool use_lora = p.num_adapters > 0 && p.rank > 0;
  const int nk = (p.K + kActGroup - 1) / kActGroup;  // 128-K blocks
  const int lkb = (p.rank + 63) / 64;                // 64-K blocks per adapter of the LoRA expand

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(&pfull[s], 1);
      mbar_init(&pempty[s], 4);  // the four epilogue warps
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    *s_grid_key = ~0ull;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tm_w);
    tma_prefetch_map(&tm_x);
    if (use_lora) {
      tma_prefetch_map(&tm_lb);
      tma_prefetch_map(&tm_lu);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  // Everything this kernel reads besides the weights (routing tables, the
  // quantized rows and their scales, the LoRA operand) comes from the
  // kernels before it.
  pdl_wait();
  for (int i = threadIdx.x; i <= p.E; i += blockDim.x) {
    s_off[i] = __ldcg(p.expert_offsets + i);
    s_ts[i] = __ldcg(p.tile_start + i);
  }
  pdl_launch_dependents();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const int FBg = p.feat_blocks;
  const int total_work = s_ts[p.E] * FBg;
  // Units are dealt round robin over the first unit_step CTAs of the grid,
  // a count that evens out the last round; the rest take none.
  const int unit_step = balanced_grid(total_work, static_cast<int>(gridDim.x), s_grid_key);
  const int unit0 = static_cast<int>(blockIdx.x) < unit_step ? static_cast<int>(blockIdx.x) : total_work;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_x = l2_policy_evict_last();
    uint32_t stage = 0, phase = 0, armed = 0, armed_parity = 0;
    bool ok = true;
    for (int w = unit0; w < total_work && ok; w += unit_step) {
      if (__shfl_sync(kFullMask, *abort_flag, 0)) break;
      const Work wk = decode_work<BN>(w, 0, 1, s_off, s_ts, p.E, FBg);
      uint64_t amask = use_lora ? tile_adapter_mask<BN>(p.row_adapter, wk.row0, wk.nrows, lane) : 0;
      const int nblocks = nk + __popcll(amask) * lkb;
      int adapter = -1, j = 0;
      for (int b = 0; b < nblocks; ++b) {
        if (b >= nk && j == 0) {
          adapter = __ffsll(static_cast<long long>(amask)) - 1;
          amask &= amask - 1;
        }
        if (lane == 0 && p.fuse_shrink && b == nk) {
          // the tile's LoRA rows come from the in-kernel shrink of running
          // CTAs (this one included): wait until all of them are published
          ok = wait_tile_rows(p.tile_flags + w / FBg, wk.nrows, p.timeout_ns, abort_flag);
          if (!ok && !*abort_flag) raise_timeout_at(p.status, abort_flag, kWaitShrinkFlag, w, b, stage);
        }
        if (lane == 0 && ok) {
          ok = wait_or_abort(&empty[stage], phase ^ 1, p.timeout_ns, abort_flag);
          if (ok) {
            uint8_t* sA = smem + stage * C::kStageBytes;
            uint8_t* sB = sA + C::kABytes;
            mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
            if (b < nk) {
              if (MODE == kGateUp)  // map dims {H, 16 rows, 2 halves, I/16 groups, E}, bytes
                tma_load_5d(sA, &tm_w, &full[stage], b * 128, 0, 0, wk.fb * 4, wk.e, pol_w);
              else
                tma_load_2d(sA, &tm_w, &full[stage], b * 128, wk.e * p.rows_per_expert + wk.fb * 128, pol_w);
              tma_load_2d(sB, &tm_x, &full[stage], b * 128, wk.row0, pol_x);
            } else {
              const int64_t frow = static_cast<int64_t>(adapter) * p.lb_row_stride_adapter +
                                   static_cast<int64_t>(wk.e) * p.lb_row_stride_expert;
              load_lora_b_block<MODE, false>(sA, &tm_lb, &full[stage], 0u, j * 64, frow, wk.fb, p.n_feat,
                                             pol_x);
              tma_load_2d(sB, &tm_lu, &full[stage], adapter * p.rank + j * 64, wk.row0, pol_x);
            }
            armed |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          } else {
            raise_timeout_at(p.status, abort_flag, kWaitProducer, w, b, stage);
          }
        }
        ok = __shfl_sync(kFullMask, ok, 0);
        if (!ok) break;
        if (b >= nk) j = (j + 1 == lkb) ? 0 : j + 1;
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (lane == 0) {  // every load issued must have landed before the CTA leaves
      const uint64_t lim = *abort_flag ? 1000000ull : p.timeout_ns;
      for (int s = 0; s < C::kStages; ++s)
        if (armed & (1u << s))
          if (!mbar_wait(&full[s], (armed_parity >> s) & 1u, lim)) note_drain_timeout(p.status, kWaitDrainProducer, s);
    }
    __syncwarp();
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer
    uint32_t stage = 0, phase = 0, slot = 0, sphase = 0;
    bool ok = true;
    for (int w = unit0; w < total_work && ok; w += unit_step) {
      if (__shfl_sync(kFullMask, *abort_flag, 0)) break;
      const Work wk = decode_work<BN>(w, 0, 1, s_off, s_ts, p.E, FBg);
      const uint64_t amask = use_lora ? tile_adapter_mask<BN>(p.row_adapter, wk.row0, wk.nrows, lane) : 0;
      const int nblocks = nk + __popcll(amask) * lkb;
      const int ncols = ((wk.nrows + 15) / 16) * 16;
      const uint32_t idesc8 = make_idesc_e4m3(128, ncols);
      const uint32_t idesc16 = make_idesc_bf16(128, ncols);
      int j = 0;
      for (int b = 0; b < nblocks; ++b) {
        if (lane == 0) {
          ok = wait_or_abort(&full[stage], phase, p.timeout_ns, abort_flag);
          if (!ok) {
            raise_timeout_at(p.status, abort_flag, kWaitMmaFull, w, b, stage);
          } else {
            ok = wait_or_abort(&pempty[slot], sphase ^ 1, p.timeout_ns, abort_flag);
            if (!ok) raise_timeout_at(p.status, abort_flag, kWaitMmaAccEmpty, w, b, slot);
          }
          if (ok) {
            tc_fence_after_sync();
            const uint32_t a_addr = smem_u32(smem + stage * C::kStageBytes);
            const uint64_t adesc = make_sdesc_sw128(a_addr);
            const uint64_t bdesc = make_sdesc_sw128(a_addr + C::kABytes);
            const uint32_t d_tmem = tmem_base + slot * BN;
            if (b < nk) {
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                tc_mma_e4m3(d_tmem, adesc + 2 * ks, bdesc + 2 * ks, idesc8, ks > 0 ? 1u : 0u);
            } else {
              const int rem = p.rank - j * 64;
              const int ksteps = rem >= 64 ? 4 : (rem + 15) / 16;
              for (int ks = 0; ks < ksteps; ++ks)
                tc_mma_bf16(d_tmem, adesc + 2 * ks, bdesc + 2 * ks, idesc16, ks > 0 ? 1u : 0u);
            }
            tc_commit(&empty[stage]);
            tc_commit(&pfull[slot]);
          }
        }
        ok = __shfl_sync(kFullMask, ok, 0);
        if (!ok) break;
        if (b >= nk) j = (j + 1 == lkb) ? 0 : j + 1;
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1;
        }
        if (++slot == C::kSlots) {
          slot = 0;
          sphase ^= 1;
        }
      }
    }
    // Every MMA issued must be complete before TMEM is released.
    if (lane == 0) {
      tc_commit(drain);
      if (!mbar_wait(drain, 0, p.timeout_ns)) note_drain_timeout(p.status, kWaitDrainMma, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------- promotion and epilogue
    const int q = warp & 3;
    const int r = q * 32 + lane;  // this thread's TMEM lane: the unit's weight row r
    const int ldx = nk;           // token scales per row
    uint32_t slot = 0, sphase = 0;
    uint8_t* stg = s_epi + q * 1024;
    // Decode-sized tiles: the LoRA shrink of the rows (u from the bf16
    // hidden rows, v from the bf16 activation) runs here, before the first
    // partial is ready (GemmParams::fuse_shrink).
    if (p.fuse_shrink) shrink_rows_in_gemm<BN>(p, s_off, s_ts, warp - 2, lane, reinterpret_cast<float*>(s_epi));
    for (int w = unit0; w < total_work; w += unit_step) {
      if (__shfl_sync(kFullMask, *abort_flag, 0)) break;
      const Work wk = decode_work<BN>(w, 0, 1, s_off, s_ts, p.E, FBg);
      const uint64_t amask = use_lora ? tile_adapter_mask<BN>(p.row_adapter, wk.row0, wk.nrows, lane) : 0;
      const int nblocks = nk + __popcll(amask) * lkb;
      const int ncols = ((wk.nrows + 15) / 16) * 16;
      // the weight row behind this thread's lane, and its scale row
      int wrow;
      if (MODE == kGateUp) wrow = ((r >> 4) & 1) * p.n_feat + wk.fb * 64 + (r >> 5) * 16 + (r & 15);
      else wrow = wk.fb * 128 + r;
      const bool wrow_in = wrow < p.rows_per_expert;
      const float* wsrow = p.w_scale + (static_cast<size_t>(wk.e) * p.scale_nb + (wrow_in ? wrow >> 7 : 0)) *
                                           p.scale_kb;
      // token scales of K block kb for columns 32 c + lane (0 past the tile)
      constexpr int NC = (BN + 31) / 32;
      auto load_xs = [&](int kb, float (&xs)[NC]) {
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const int col = c * 32 + lane;
          xs[c] = (col < wk.nrows && kb < nk) ? __ldg(p.x_scale + static_cast<size_t>(wk.row0 + col) * ldx + kb)
                                              : 0.f;
        }
      };
      float xs_cur[NC], xs_nxt[NC];
      load_xs(0, xs_cur);
      float ws_cur = wrow_in ? __ldg(wsrow) : 0.f;
      float acc[BN];
#pragma unroll
      for (int c = 0; c < BN; ++c) acc[c] = 0.f;
      bool ok = true;
      for (int b = 0; b < nblocks; ++b) {
        // the next block's scales are in flight while this one waits and adds
        load_xs(b + 1, xs_nxt);
        const float ws_nxt = (wrow_in && b + 1 < nk) ? __ldg(wsrow + b + 1) : 0.f;
        if (lane == 0) {
          ok = wait_or_abort(&pfull[slot], sphase, p.timeout_ns, abort_flag);
          if (!ok) raise_timeout_at(p.status, abort_flag, kWaitEpilogue, w, b, slot);
        }
        ok = __shfl_sync(kFullMask, ok, 0);
        if (!ok) break;
        tc_fence_after_sync();
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + slot * BN;
        const bool main_block = b < nk;
#pragma unroll
        for (int c0 = 0; c0 < BN; c0 += 16) {
          if (c0 < ncols) {
            float v[16];
            tmem_ld16(t_row + c0, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int col = c0 + i;
              const float ts = __shfl_sync(kFullMask, xs_cur[col / 32], col % 32);
              acc[col] = main_block ? fmaf(v[i], ws_cur * ts, acc[col]) : acc[col] + v[i];
            }
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pempty[slot]);
        if (++slot == C::kSlots) {
          slot = 0;
          sphase ^= 1;
        }
#pragma unroll
        for (int c = 0; c < NC; ++c) xs_cur[c] = xs_nxt[c];
        ws_cur = ws_nxt;
      }
      if (!ok) break;
      // output: per 16 columns, registers -> (SwiGLU) -> staging tile -> rows
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 16) {
        if (c0 < ncols) {
          const int col = c0 + (lane >> 1);  // the column this lane writes out
          if (MODE == kGateUp) {
            // lanes < 16 hold gate rows, lanes >= 16 the up rows of the same
            // 16 features; the float32 activation goes out for its quant
            float* stg32 = reinterpret_cast<float*>(stg);
            const bool hi = lane >= 16;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float send = hi ? acc[c0 + 2 * i] : acc[c0 + 2 * i + 1];
              const float recv = __shfl_xor_sync(kFullMask, send, 16);
              const float gate = hi ? recv : acc[c0 + 2 * i];
              const float up = hi ? acc[c0 + 2 * i + 1] : recv;
              stg32[(2 * i + (hi ? 1 : 0)) * 16 + (lane & 15)] = __fdividef(gate, 1.0f + __expf(-gate)) * up;
            }
            __syncwarp();
            // lane L: column L / 2, features 8 (L % 2) .. + 7 of the warp's 16
            const int feat = wk.fb * 64 + q * 16 + 8 * (lane & 1);
            const float4 o0 = *reinterpret_cast<const float4*>(stg + lane * 32);
            const float4 o1 = *reinterpret_cast<const float4*>(stg + lane * 32 + 16);
            if (col < wk.nrows && feat < p.n_feat) {
              float* dst = p.out_f32 + static_cast<size_t>(wk.row0 + col) * p.n_feat + feat;
              *reinterpret_cast<float4*>(dst) = o0;
              *reinterpret_cast<float4*>(dst + 4) = o1;
            }
          } else {
            __nv_bfloat16* stg16 = reinterpret_cast<__nv_bfloat16*>(stg);
#pragma unroll
            for (int i = 0; i < 16; ++i) stg16[i * 32 + lane] = __float2bfloat16_rn(acc[c0 + i]);
            __syncwarp();
            // lane L: column L / 2, features 16 (L % 2) .. + 15 of the warp's 32
            const int feat = wk.fb * 128 + q * 32 + 16 * (lane & 1);
            const uint4 o0 = *reinterpret_cast<const uint4*>(stg + lane * 32);
            const uint4 o1 = *reinterpret_cast<const uint4*>(stg + lane * 32 + 16);
            if (col < wk.nrows) {
              __nv_bfloat16* dst = p.out + static_cast<size_t>(wk.row0 + col) * p.n_feat + feat;
              if (feat < p.n_feat) *reinterpret_cast<uint4*>(dst) = o0;
              if (feat + 8 < p.n_feat) *reinterpret_cast<uint4*>(dst + 8) = o1;
            }
          }
          __syncwarp();  // the staging tile is free again
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

int fp8_gemm_ctas_per_sm(int bn) { return bn <= 64 ? 2 : 1; }

template <int BN, int MODE>
static cudaError_t launch_fp8_one(const CUtensorMap& tm_w, const CUtensorMap& tm_x, const CUtensorMap& tm_lb,
                                  const CUtensorMap& tm_lu, const GemmParams& p, int grid, cudaStream_t s) {
  using C = Fp8Cfg<BN>;
  auto kern = fp8_gemm_kernel<BN, MODE>;
  cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(kern), C::kSmemBytes);
  if (err != cudaSuccess) return err;
  return launch_pdl(kern, dim3(grid), dim3(C::kThreads), C::kSmemBytes, s, tm_w, tm_x, tm_lb, tm_lu, p);
}

cudaError_t launch_fp8_gemm(int mode, int bn, const CUtensorMap& tm_w, const CUtensorMap& tm_x,
                            const CUtensorMap& tm_lb, const CUtensorMap& tm_lu, const GemmParams& p, int grid,
                            cudaStream_t s) {
#define MOE_FP8_CASE(BNV)                                                                    \
  if (bn == BNV)                                                                             \
    return mode == kGateUp ? launch_fp8_one<BNV, kGateUp>(tm_w, tm_x, tm_lb, tm_lu, p, grid, s) \
                           : launch_fp8_one<BNV, kDown>(tm_w, tm_x, tm_lb, tm_lu, p, grid, s);
  MOE_FP8_CASE(16)
  MOE_FP8_CASE(32)
  MOE_FP8_CASE(64)
  MOE_FP8_CASE(128)
#undef MOE_FP8_CASE
  return cudaErrorInvalidValue;
}

}  // namespace moe
