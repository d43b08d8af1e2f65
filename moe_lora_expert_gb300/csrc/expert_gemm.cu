// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM),
// operands staged by TMA.
//
// The gate_up GEMM (K = hidden, N = 2*inter) and the down GEMM (K = inter,
// N = hidden) of the launcher row in the "Files changed" table of
// "[WIP][LoRA] BF16 support for the experimental_sgl_trtllm MoE-LoRA path &
// lora expert_outer_shared" (yushengsu-thu/sglang#4), with
//   * the LoRA expand (s * B u, u = A x computed by the shrink kernel) run as
//     extra K blocks of the same accumulation: for each adapter present in
//     the token tile, B[a, e] (rows = output features, K = rank) against the
//     one-hot operand U[:, a*r : a*r + r] whose rows are zero for tokens of
//     other adapters;
//   * for gate_up, the LoRA-aware SwiGLU in the epilogue: the delta is
//     already inside the accumulator when h = silu(gate) * up is taken,
//     which is the "adds gate_up_lora_delta pre-SwiGLU" order of the
//     launcher row.
//
// Orientation ("swap AB"): the MMA's M side is 128 weight rows (output
// features), its N side is the token tile.  D[feature, token] lives in TMEM,
// lane = feature row, column = token.  Both operands are K-major, loaded by
// TMA with 128-byte swizzle.
//
// gate_up feature block fb covers gate features [64 fb, 64 fb + 64) and the
// matching up features.  Its 128 A rows are eight 16-row boxes interleaved
// so that TMEM lanes [32q, 32q + 16) hold gate rows 64 fb + 16q + (0..15)
// and lanes [32q + 16, 32q + 32) the up rows of the same features: warp q of
// the epilogue then pairs gate and up with one shuffle.
//
// Roles (192 threads): warp 0 = TMA producer, warp 1 = MMA issuer and TMEM
// owner, warps 2..5 = epilogue (TMEM lane quadrant = warp % 4).  The kernel
// is persistent: CTA b < P takes work items b, b + P, ... (P, at most the
// grid, chosen on the device so that the last round is not a thin one; see
// balanced_grid); the TMEM accumulator is double-buffered so the epilogue of
// one item overlaps the MMAs of the next.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "../../include/moe_lora.h"
#include "gemm_common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

template <int BN, bool PAIR = false, bool W8 = false>
struct GemmCfg {
  // Narrow (decode) tiles run two CTAs per SM so that two producers keep TMA
  // loads in flight; wide tiles run one CTA per SM with deeper stages.
  static constexpr int kCtasPerSm = BN <= 64 ? 2 : 1;
  // FP8 weights add kConvWarps converter warps (warps 6, 7, ...).
  static constexpr int kConvWarps = 4;
  static constexpr int kThreads = W8 ? 192 + 32 * kConvWarps : 192;
  static constexpr int kStageBudget = BN <= 64 ? (W8 ? 104 : 96) * 1024 : 200 * 1024;
  // 64-K sub-blocks per ring stage.  The MMA role commits once per stage
  // (that releases it to the producer), and on sm_103a each commit costs
  // about as much as a few MMAs, so wide tiles take two sub-blocks (eight
  // MMAs per commit).  FP8 weights keep one.
  static constexpr int kKSub = W8 ? 1 : (BN >= 128 ? 2 : 1);
  static constexpr int kASub = 128 * 64 * 2;     // 128 rows x 64 K of bf16
  // A CTA of a pair holds half of the token tile.
  static constexpr int kBSub = (PAIR ? BN / 2 : BN) * 64 * 2;
  // Tiles of a few rows (an expert's last, nearly empty tile) load their
  // token rows through a second tensor map whose box is kSmallRows high.
  static constexpr int kSmallRows = 32;
  static constexpr int kBSubSmall = kSmallRows * 64 * 2;
  static constexpr int kABytes = kKSub * kASub;
  static constexpr int kBBytes = kKSub * kBSub;
  static constexpr int kStageBytes = kABytes + kBBytes;
  // FP8: a deep ring of (raw 128 x 64 e4m3 weight tile, token tile) stages
  // filled by TMA; the converter warps write the bf16 A tiles into a short
  // ring of A-only stages.
  static constexpr int kW8Bytes = 128 * 64;
  static constexpr int kW8Stage = (kW8Bytes + kBBytes + 1023) / 1024 * 1024;
  static constexpr int kStagesRaw = W8 ? (BN <= 64 ? 3 : 4) : kStageBudget / kStageBytes;
  static constexpr int kStages = kStagesRaw > 16 ? 16 : kStagesRaw;
  static constexpr int kARingBytes = W8 ? kStages * kABytes : kStages * kStageBytes;
  static constexpr int kStages8Raw = W8 ? (kStageBudget - kARingBytes) / kW8Stage : 0;
  static constexpr int kStages8 = kStages8Raw > 16 ? 16 : kStages8Raw;
  static constexpr int kTmemCols = (2 * BN < 32) ? 32 : 2 * BN;
  static constexpr int kMetaBytes = 512;                         // barriers, flags
  static constexpr int kTableBytes = 2 * (MOE_MAX_EXPERTS + 1) * 4;
  // Per-unit descriptors (K blocks, MMA width) that the producer publishes
  // for the MMA role: a ring of more entries than there are stages, so the
  // producer (at most kStages stages ahead) never overwrites one in use.
  static constexpr int kUnitRing = 32;
  static constexpr int kUnitBytes = kUnitRing * 8;
  // Epilogue: a 1 KB staging tile per epilogue warp (16 token columns of its
  // features), so the output leaves in 16-byte row segments.
  static constexpr int kEpiOffset = (kMetaBytes + kTableBytes + kUnitBytes + 15) / 16 * 16;
  static constexpr int kEpiBytes = 4 * 1024;
  static constexpr int kSmemBytes =
      1024 + kARingBytes + kStages8 * kW8Stage + kEpiOffset + kEpiBytes;
  static_assert((2 * kStages + 2 * kStages8 + 6) * 8 + 16 <= kMetaBytes, "barriers, TMEM slot, flag, key fit");
  static_assert(kUnitRing > kStages, "a unit has at least one stage");
  static_assert(kCtasPerSm * (kSmemBytes + 1024) <= 233472, "the CTAs of an SM fit its shared memory");
};

// PAIR (CL == 2): the two CTAs of the cluster take adjacent feature blocks
// of the same token tile and share one M = 256 MMA (cta_group::2).  Each
// loads its 128 weight rows and half of the token rows; all those bytes
// complete on the even CTA's barrier, whose MMA warp alone issues the MMAs
// and commits to both CTAs' barriers.  Each CTA's TMEM receives its own
// feature block for the whole token tile, so the epilogue is unchanged; the
// epilogue warps of both CTAs release the even CTA's accumulator barrier.
//
// W8 (FP8 block-scaled weights, CL == 1): warp 0 streams each K block's raw
// e4m3 weight tile and its token tile through the deep ring (full8/empty8);
// the converter warps wait for a free bf16 A stage, write the dequantized
// weight tile (e4m3 value times its 128 x 128 block scale, rounded to bf16)
// in the 128-byte-swizzled layout the MMA reads, and arrive on full, one
// arrival per warp.  A LoRA block's bf16 B-factor tile goes straight to the
// A stage by TMA.  The MMA reads A from the A ring and the token tile from
// the deep ring; the epilogue is unchanged.
template <int BN, int MODE, int CL, bool PAIR, bool W8>
__global__ void __launch_bounds__(GemmCfg<BN, PAIR, W8>::kThreads, GemmCfg<BN, PAIR, W8>::kCtasPerSm)
    expert_gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                       const __grid_constant__ CUtensorMap tm_lb, const __grid_constant__ CUtensorMap tm_lu,
                       const __grid_constant__ CUtensorMap tm_xs, const __grid_constant__ CUtensorMap tm_lus,
                       const GemmParams p) {
  static_assert(PAIR == (CL == 2) && CL <= 2, "one CTA per tile, or a pair (a cluster of two)");
  static_assert(!W8 || (CL == 1 && !PAIR), "FP8 weights: one CTA per tile");
  using C = GemmCfg<BN, PAIR, W8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* w8ring = smem + C::kARingBytes;  // FP8 only
  uint8_t* meta = w8ring + C::kStages8 * C::kW8Stage;
  uint64_t* full = reinterpret_cast<uint64_t*>(meta);
  uint64_t* empty = full + C::kStages;
  uint64_t* accf = empty + C::kStages;
  uint64_t* acce = accf + 2;
  uint64_t* drain = acce + 2;
  uint64_t* never = drain + 1;  // test hook: a barrier nothing arrives on
  uint64_t* full8 = never + 1;
  uint64_t* empty8 = full8 + C::kStages8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(empty8 + C::kStages8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  unsigned long long* s_grid_key = reinterpret_cast<unsigned long long*>(tmem_slot + 2);
  int* s_off = reinterpret_cast<int*>(meta + C::kMetaBytes);
  int* s_ts = s_off + (MOE_MAX_EXPERTS + 1);
  int2* s_units = reinterpret_cast<int2*>(meta + C::kMetaBytes + C::kTableBytes);
  uint8_t* s_epi = meta + C::kEpiOffset;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool use_lora = p.num_adapters > 0 && p.rank > 0;
  constexpr int kBlockK = 64 * C::kKSub;  // K elements per ring stage
  const int nk = (p.K + kBlockK - 1) / kBlockK;
  const int lkb = (p.rank + kBlockK - 1) / kBlockK;  // K blocks per adapter of the LoRA expand
  // 64-K sub-blocks of block b that hold any K (the rest are neither loaded
  // nor multiplied); j: the block's index within its adapter's LoRA blocks
  auto subs_of = [&](int b, int j) {
    const int left = b < nk ? p.K - b * kBlockK : p.rank - j * kBlockK;
    return min(C::kKSub, (left + 63) / 64);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages8; ++s) {
      mbar_init(&full8[s], 1);
      mbar_init(&empty8[s], 1);
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], W8 ? C::kConvWarps : 1);  // FP8: one arrival per converter warp
      // pair: the leader's commit arrives once in each CTA
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], PAIR ? 8 : 4);  // epilogue warps (of both CTAs of a pair)
    }
    mbar_init(drain, 1);
    mbar_init(never, 1);
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
    if constexpr (PAIR) {  // collective with the peer's warp 1
      tmem_alloc_pair(tmem_slot, C::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, C::kTmemCols);
      tmem_relinquish();
    }
  }
  // Programmatic dependent launch: this grid may start while the previous
  // kernel drains.  When that kernel is the shrink (tables_ready), it waited
  // for its own predecessor before letting this grid launch, so the routing
  // tables the permute wrote are complete: they are read now (L2 loads, no
  // stale L1 line possible), the weight stream starts at once, and only the
  // token-side loads, which read what the shrink wrote, wait (producer warp,
  // below).  Otherwise every thread waits here first.
  if (!p.tables_ready) pdl_wait();
  for (int i = threadIdx.x; i <= p.E; i += blockDim.x) {
    s_off[i] = __ldcg(p.expert_offsets + i);
    s_ts[i] = __ldcg(p.tile_start + i);
  }
  pdl_launch_dependents();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  // The pair leader's loads and commits arrive on this CTA's barriers: all of
  // them must be initialised.
  if (CL > 1) cluster_sync_all();
  const uint32_t tmem_base = *tmem_slot;
  const int crank = CL > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int FBg = (p.feat_blocks + CL - 1) / CL;
  const int total_work = s_ts[p.E] * FBg;
  // Units are dealt round robin over the first unit_step CTAs of the grid,
  // a count that evens out the last round of these HBM-bound tiles; the rest
  // take none.  CTA pairs (wide tiles, bound by the tensor pipe) and FP8
  // weights (bound by the converter warps) run no faster with fewer units in
  // the last round: there every CTA takes units.
  const int unit_step = CL > 1 ? static_cast<int>(cluster_count_x())
                        : W8   ? static_cast<int>(gridDim.x)
                               : balanced_grid(total_work, static_cast<int>(gridDim.x), s_grid_key);
  const int unit_id = CL > 1 ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int unit0 = unit_id < unit_step ? unit_id : total_work;
  const bool leader = !PAIR || crank == 0;

  if (W8 && warp == 0) {
    // ---------------------------------------------------- FP8 producer
    // Per K block one ring stage: the raw e4m3 weight tile (main blocks) and
    // the token tile (x, or the one-hot u of a LoRA block), 128-byte
    // swizzled, that the MMA reads in place.  Weights are static and go out
    // at once; the token tiles of the first ring pass wait for the previous
    // kernel (griddepcontrol.wait).
    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_x = l2_policy_evict_last();
    uint32_t s8 = 0, ph8 = 0, armed = 0, armed_parity = 0;
    bool ok = true;
    bool waited = !p.tables_ready;
    int n_pend = 0;
    const CUtensorMap* pend_map[C::kStages8 > 0 ? C::kStages8 : 1];
    int pend_c0[C::kStages8 > 0 ? C::kStages8 : 1], pend_c1[C::kStages8 > 0 ? C::kStages8 : 1],
        pend_stage[C::kStages8 > 0 ? C::kStages8 : 1];
    auto release_pending = [&]() {
      pdl_wait();
      waited = true;
      for (int i = 0; i < n_pend; ++i)
        tma_load_2d(w8ring + pend_stage[i] * C::kW8Stage + C::kW8Bytes, pend_map[i], &full8[pend_stage[i]],
                    pend_c0[i], pend_c1[i], pol_x);
      n_pend = 0;
    };
    for (int w = unit0; w < total_work && ok; w += unit_step) {
      if (__shfl_sync(kFullMask, *abort_flag, 0)) break;
      const Work wk = decode_work<BN>(w, crank, CL, s_off, s_ts, p.E, FBg);
      uint64_t amask = use_lora ? tile_adapter_mask<BN>(p.row_adapter, wk.row0, wk.nrows, lane) : 0;
      const int nblocks = nk + __popcll(amask) * lkb;
      int adapter = -1, j = 0;
      for (int b = 0; b < nblocks; ++b) {
        if (b >= nk && j == 0) {
          adapter = __ffsll(static_cast<long long>(amask)) - 1;
          amask &= amask - 1;
        }
        if (lane == 0 && p.fuse_shrink && b == (p.gather_src != nullptr ? 0 : nk)) {
          // the tile's token / LoRA rows come from the in-kernel pass
          ok = wait_tile_rows(p.tile_flags + w / FBg, wk.nrows, p.timeout_ns, abort_flag);
          if (!ok && !*abort_flag) raise_timeout_at(p.status, abort_flag, kWaitShrinkFlag, w, b, s8);
        }
        if (lane == 0 && ok) {
          ok = wait_or_abort(&empty8[s8], ph8 ^ 1, p.timeout_ns, abort_flag);
          if (ok) {
            uint8_t* st = w8ring + s8 * C::kW8Stage;
            mbar_arrive_expect_tx(&full8[s8], (b < nk ? C::kW8Bytes : 0) + C::kBBytes);
            const CUtensorMap* tmap;
            int tc0;
            if (b < nk) {
              load_weight_block<MODE, false, 1>(st, &tm_w, &full8[s8], 0u, b * 64, wk.e, wk.fb,
                                                p.rows_per_expert, p.gu_single_box, pol_w);
              tmap = &tm_x;
              tc0 = b * 64;
            } else {
              tmap = &tm_lu;
              tc0 = adapter * p.rank + j * 64;
            }
            if (waited) {
              tma_load_2d(st + C::kW8Bytes, tmap, &full8[s8], tc0, wk.row0, pol_x);
            } else {
              pend_map[n_pend] = tmap;
              pend_c0[n_pend] = tc0;
              pend_c1[n_pend] = wk.row0;
              pend_stage[n_pend] = s8;
              ++n_pend;
              if (static_cast<int>(s8) == C::kStages8 - 1) release_pending();  // before the ring wraps
            }
            armed |= 1u << s8;
            armed_parity = (armed_parity & ~(1u << s8)) | (ph8 << s8);
          } else {
            raise_timeout_at(p.status, abort_flag, kWaitProducerW8, w, b, s8);
          }
        }
        ok = __shfl_sync(kFullMask, ok, 0);
        if (!ok) break;
        if (b >= nk) j = (j + 1 == lkb) ? 0 : j + 1;
        if (++s8 == C::kStages8) {
          s8 = 0;
          ph8 ^= 1;
        }
      }
    }
    if (lane == 0 && !waited) release_pending();
    if (lane == 0) {  // every load issued must have landed before the CTA leaves
      const uint64_t lim = *abort_flag ? 1000000ull : p.timeout_ns;
      for (int s = 0; s < C::kStages8; ++s)
        if (armed & (1u << s))
          if (!mbar_wait(&full8[s], (armed_parity >> s) & 1u, lim))
            note_drain_timeout(p.status, kWaitDrainProducerW8, s);
    }
    __syncwarp();
  } else if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_x = l2_policy_evict_last();
    uint32_t stage = 0, phase = 0;
    uint32_t armed = 0, armed_parity = 0;
    bool ok = true;
    // Token-side loads of the first ring pass are held back until the
    // previous kernel has completed (griddepcontrol.wait).
    bool waited = !p.tables_ready;
    int n_pend = 0;
    constexpr int kPend = C::kStages * C::kKSub;
    const CUtensorMap* pend_map[kPend];
    int pend_c0[kPend], pend_c1[kPend], pend_stage[kPend];
    // Pair: c1 already names this CTA's half of the token tile.  c0 is the
    // sub-block's first K element; st * kKSub + sub names stage and sub-block.
    auto issue_token_load = [&](const CUtensorMap* map, int st_sub, int c0, int c1) {
      const int st = st_sub / C::kKSub, sub = st_sub % C::kKSub;
      uint8_t* sB = smem + st * C::kStageBytes + C::kABytes + sub * C::kBSub;
      if constexpr (PAIR)
        tma_load_2d_pair(sB, map, mapa_shared(smem_u32(&full[st]), 0), c0, c1, pol_x);
      else
        tma_load_2d(sB, map, &full[st], c0, c1, pol_x);
    };
    auto release_pending = [&]() {
      pdl_wait();
      waited = true;
      for (int i = 0; i < n_pend; ++i) issue_token_load(pend_map[i], pend_stage[i], pend_c0[i], pend_c1[i]);
      n_pend = 0;
    };
    // The next unit's tile and row adapters are worked out while this unit's
    // loads go out, so no gap opens in the load stream between units.
    Work next_wk{};
    TileAdapters<BN> next_ad;
    if (unit0 < total_work) {
      next_wk = decode_work<BN>(unit0, crank, CL, s_off, s_ts, p.E, FBg);
      if (use_lora) load_tile_adapters<BN>(p.row_adapter, next_wk.row0, next_wk.nrows, lane, next_ad);
    }
    for (int w = unit0, ul = 0; w < total_work && ok; w += unit_step, ++ul) {
      if (__shfl_sync(kFullMask, *abort_flag, 0)) break;
      const Work wk = next_wk;
      uint64_t amask = use_lora ? reduce_tile_adapters<BN>(next_ad) : 0;
      if (w + unit_step < total_work) {
        next_wk = decode_work<BN>(w + unit_step, crank, CL, s_off, s_ts, p.E, FBg);
        if (use_lora) load_tile_adapters<BN>(p.row_adapter, next_wk.row0, next_wk.nrows, lane, next_ad);
      }
      const int nblocks = nk + __popcll(amask) * lkb;
      // the MMA role reads this after the unit's first full barrier, whose
      // arrival below releases it
      if (lane == 0)
        s_units[ul % C::kUnitRing] =
            make_int2(nblocks, PAIR ? ((wk.nrows + 31) / 32) * 32 : ((wk.nrows + 15) / 16) * 16);
      // first token row this CTA loads: a pair splits the MMA's N in halves
      const int trow = PAIR ? wk.row0 + crank * (((wk.nrows + 31) / 32) * 16) : wk.row0;
      // token rows this CTA's MMA operand needs; few: the small-box maps
      const int my_rows = PAIR ? ((wk.nrows + 31) / 32) * 16 : ((wk.nrows + 15) / 16) * 16;
      const bool small = BN > C::kSmallRows && my_rows <= C::kSmallRows;
      const int bsub = small ? C::kBSubSmall : C::kBSub;
      int adapter = -1, j = 0;
      for (int b = 0; b < nblocks; ++b) {
        if (b >= nk) {  // next LoRA block: adapters in ascending order, lkb blocks each
          if (j == 0) {
            adapter = __ffsll(static_cast<long long>(amask)) - 1;
            amask &= amask - 1;
          }
        }
        if (lane == 0 && p.fuse_shrink && b == (p.gather_src != nullptr ? 0 : nk)) {
          // the tile's LoRA rows (and, gathering, its token rows) come from
          // the in-kernel pass of other CTAs (or this one): wait until all
          // of them are published
          ok = wait_tile_rows(p.tile_flags + w / FBg, wk.nrows, p.timeout_ns, abort_flag);
          if (!ok && !*abort_flag) raise_timeout_at(p.status, abort_flag, kWaitShrinkFlag, w, b, stage);
        }
        if (lane == 0 && ok) {
          ok = wait_or_abort<PAIR>(&empty[stage], phase ^ 1, p.timeout_ns, abort_flag);
          if (ok) {
            const int nsub = subs_of(b, j);
            // the pair leader counts the bytes of both CTAs
            if (leader) mbar_arrive_expect_tx(&full[stage], (PAIR ? 2 : 1) * nsub * (C::kASub + bsub));
            const uint32_t cbar = PAIR ? mapa_shared(smem_u32(&full[stage]), 0) : 0u;
            for (int sub = 0; sub < nsub; ++sub) {
              uint8_t* sA = smem + stage * C::kStageBytes + sub * C::kASub;
              const CUtensorMap* tmap;
              int tc0;
              if (b < nk) {
                const int kc = b * kBlockK + sub * 64;
                load_weight_block<MODE, PAIR>(sA, &tm_w, &full[stage], cbar, kc, wk.e, wk.fb,
                                              p.rows_per_expert, p.gu_single_box, pol_w);
                tmap = small ? &tm_xs : &tm_x;
                tc0 = kc;
              } else {
                const int kc = j * kBlockK + sub * 64;
                const int64_t frow = static_cast<int64_t>(adapter) * p.lb_row_stride_adapter +
                                     static_cast<int64_t>(wk.e) * p.lb_row_stride_expert;
                load_lora_b_block<MODE, PAIR>(sA, &tm_lb, &full[stage], cbar, kc, frow, wk.fb,
                                              p.n_feat, pol_x);
                tmap = small ? &tm_lus : &tm_lu;
                tc0 = adapter * p.rank + kc;
              }
              const int st_sub = stage * C::kKSub + sub;
              if (waited) {
                issue_token_load(tmap, st_sub, tc0, trow);
              } else {
                pend_map[n_pend] = tmap;
                pend_c0[n_pend] = tc0;
                pend_c1[n_pend] = trow;
                pend_stage[n_pend] = st_sub;
                ++n_pend;
              }
            }
            // before the ring wraps onto a stage whose token loads still wait
            if (!waited && stage == C::kStages - 1) release_pending();
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
    if (lane == 0 && !waited) release_pending();
    // Every load issued must have landed before the CTA leaves.  A pair's
    // odd CTA cannot wait on the leader's barriers: it waits until the MMA
    // released each stage it filled last (the data had landed by then).
    // After an abort nothing may consume the stages any more; loads in
    // flight land within microseconds, so a short wait suffices then.
    if (lane == 0) {
      const uint64_t lim = *abort_flag ? 1000000ull : p.timeout_ns;
      for (int s = 0; s < C::kStages; ++s)
        if (armed & (1u << s)) {
          uint64_t* bar = leader ? &full[s] : &empty[s];
          if (!mbar_wait(bar, (armed_parity >> s) & 1u, lim)) note_drain_timeout(p.status, kWaitDrainProducer, s);
        }
    }
    __syncwarp();
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer
    uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
    uint32_t s8 = 0, ph8 = 0;  // FP8: the ring stage holding this block's token tile
    bool ok = leader;  // a pair's odd CTA issues no MMA
    if (p.debug_stall_mma && leader) {  // failure-path test: this wait can only run out
      if (lane == 0 && !wait_or_abort(never, 0, p.timeout_ns, abort_flag))
        raise_timeout(p.status, abort_flag);
      ok = false;
    }
    // bf16: each unit's K-block count and MMA width come from the
    // producer's descriptor ring (the producer works them out stages
    // ahead), so the MMA role does no per-unit decoding between MMAs.
    for (int w = unit0, ul = 0; w < total_work && ok; w += unit_step, ++ul) {
      if (__shfl_sync(kFullMask, *abort_flag, 0)) break;
      int nblocks_w8 = 0, ncols_w8 = 0;
      if constexpr (W8) {
        const Work wk = decode_work<BN>(w, crank, CL, s_off, s_ts, p.E, FBg);
        const uint64_t amask = use_lora ? tile_adapter_mask<BN>(p.row_adapter, wk.row0, wk.nrows, lane) : 0;
        nblocks_w8 = nk + __popcll(amask) * lkb;
        ncols_w8 = ((wk.nrows + 15) / 16) * 16;
      }
      if (lane == 0) {
        ok = wait_or_abort<PAIR>(&acce[acc], acc_phase ^ 1, p.timeout_ns, abort_flag);
        if (!ok) raise_timeout_at(p.status, abort_flag, kWaitMmaAccEmpty, w, 0, acc);
      }
      ok = __shfl_sync(kFullMask, ok, 0);
      if (!ok) break;
      tc_fence_after_sync();
      const uint32_t d_tmem = tmem_base + acc * BN;
      // The unit's K loop runs in lane 0 alone: no warp-wide exchange per
      // block between the MMA issues.
      if (lane == 0) {
        int j = 0;
        int nblocks = W8 ? nblocks_w8 : 1;  // bf16: known once the first block is in
        uint32_t idesc = make_idesc_bf16(PAIR ? 256 : 128, W8 ? ncols_w8 : 16);
        for (int b = 0; b < nblocks; ++b) {
          ok = wait_or_abort<PAIR>(&full[stage], phase, p.timeout_ns, abort_flag);
          int site = kWaitMmaFull;
          if (W8 && ok) {
            ok = wait_or_abort(&full8[s8], ph8, p.timeout_ns, abort_flag);
            site = kWaitMmaFull8;
          }
          if (!ok) {
            raise_timeout_at(p.status, abort_flag, site, w, b, site == kWaitMmaFull8 ? s8 : stage);
            break;
          }
          if (!W8 && b == 0) {
            const int2 d = s_units[ul % C::kUnitRing];
            nblocks = d.x;
            idesc = make_idesc_bf16(PAIR ? 256 : 128, d.y);
          }
          tc_fence_after_sync();
          const uint32_t a_base = smem_u32(smem + stage * (W8 ? C::kABytes : C::kStageBytes));
          const uint32_t b_base =
              W8 ? smem_u32(w8ring + s8 * C::kW8Stage + C::kW8Bytes) : a_base + C::kABytes;
          const int nsub = subs_of(b, j);
          for (int sub = 0; sub < nsub; ++sub) {
            const uint64_t adesc = make_sdesc_sw128(a_base + sub * C::kASub);
            const uint64_t bdesc = make_sdesc_sw128(b_base + sub * C::kBSub);
            int ksteps = 4;
            if (b >= nk) {
              const int rem = p.rank - j * kBlockK - sub * 64;
              ksteps = rem >= 64 ? 4 : (rem + 15) / 16;
            }
            for (int ks = 0; ks < ksteps; ++ks) {
              const uint32_t accum = (b > 0 || sub > 0 || ks > 0) ? 1u : 0u;
              if constexpr (PAIR)
                tc_mma_bf16_pair(d_tmem, adesc + 2 * ks, bdesc + 2 * ks, idesc, accum);
              else
                tc_mma_bf16(d_tmem, adesc + 2 * ks, bdesc + 2 * ks, idesc, accum);
            }
          }
          if constexpr (PAIR) tc_commit_pair(&empty[stage], 0x3);
          else tc_commit(&empty[stage]);
          if constexpr (W8) tc_commit(&empty8[s8]);
          if (b >= nk) j = (j + 1 == lkb) ? 0 : j + 1;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
          if (W8 && ++s8 == C::kStages8) {
            s8 = 0;
            ph8 ^= 1;
          }
        }
      }
      ok = __shfl_sync(kFullMask, ok, 0);
      if (!ok) break;
      if (lane == 0) {
        if constexpr (PAIR) tc_commit_pair(&accf[acc], 0x3);
        else tc_commit(&accf[acc]);
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    // Every MMA issued must be complete before TMEM is released.
    if (lane == 0 && leader) {
      if constexpr (PAIR) tc_commit_pair(drain, 0x1);
      else tc_commit(drain);
      if (!mbar_wait(drain, 0, p.timeout_ns)) note_drain_timeout(p.status, kWaitDrainMma, 0);
    }
    __syncwarp();
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    uint32_t acc = 0, acc_phase = 0;
    if constexpr (CL == 1) {
      if (p.fuse_shrink) {  // the LoRA rows of this CTA's tiles, before any accumulator is ready
        pdl_wait();
        shrink_rows_in_gemm<BN>(p, s_off, s_ts, warp - 2, lane, reinterpret_cast<float*>(s_epi));
      }
    }
    for (int w = unit0; w < total_work; w += unit_step) {
      if (__shfl_sync(kFullMask, *abort_flag, 0)) break;
      const Work wk = decode_work<BN>(w, crank, CL, s_off, s_ts, p.E, FBg);
      const int ncols = PAIR ? ((wk.nrows + 31) / 32) * 32 : ((wk.nrows + 15) / 16) * 16;
      bool ok = true;
      if (lane == 0) {
        ok = wait_or_abort<PAIR>(&accf[acc], acc_phase, p.timeout_ns, abort_flag);
        if (!ok) raise_timeout_at(p.status, abort_flag, kWaitEpilogue, w, 0, acc);
      }
      ok = __shfl_sync(kFullMask, ok, 0);
      if (!ok) break;
      tc_fence_after_sync();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      // Per 16 columns: TMEM -> registers -> (SwiGLU) -> bf16 staging tile
      // [column][feature] -> 16-byte row segments to global memory.  The
      // output feature count is a multiple of 8, so an 8-feature segment is
      // either wholly inside or wholly outside the output.
      uint8_t* stg = s_epi + q * 1024;
      __nv_bfloat16* stg16 = reinterpret_cast<__nv_bfloat16*>(stg);
      for (int c0 = 0; c0 < ncols; c0 += 16) {
        float v[16];
        tmem_ld16(t_row + c0, v);
        const int col = c0 + (lane >> 1);  // the column this lane writes out
        if (MODE == kGateUp) {
          // lanes < 16 hold gate rows, lanes >= 16 the up rows of the same
          // 16 features.  Column pairs (2i, 2i+1): the low half finishes
          // column 2i, the high half column 2i+1, after one exchange.
          const bool hi = lane >= 16;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float send = hi ? v[2 * i] : v[2 * i + 1];
            const float recv = __shfl_xor_sync(kFullMask, send, 16);
            const float gate = hi ? recv : v[2 * i];
            const float up = hi ? v[2 * i + 1] : recv;
            const float h = __fdividef(gate, 1.0f + __expf(-gate)) * up;
            stg16[(2 * i + (hi ? 1 : 0)) * 16 + (lane & 15)] = __float2bfloat16_rn(h);
          }
          __syncwarp();
          // lane L: column L / 2, features 8 (L % 2) .. + 7 of the warp's 16
          const int feat = wk.fb * 64 + q * 16 + 8 * (lane & 1);
          const uint4 o = *reinterpret_cast<const uint4*>(stg + lane * 16);
          if (col < wk.nrows && feat < p.n_feat)
            *reinterpret_cast<uint4*>(p.out + static_cast<size_t>(wk.row0 + col) * p.n_feat + feat) = o;
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) stg16[i * 32 + lane] = __float2bfloat16_rn(v[i]);
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
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if constexpr (PAIR) mbar_arrive_cluster(mapa_shared(smem_u32(&acce[acc]), 0));
        else mbar_arrive(&acce[acc]);
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  } else if constexpr (W8) {
    // ------------------------------------------------- FP8 converters
    // Warps 6.., each on its own: converter warp cw writes tile rows
    // [kRows cw, kRows (cw + 1)).  Lane l takes 16-byte chunks
    // 4 kRows cw + l + 32 i of the 8 KB e4m3 tile (row = chunk / 4, columns
    // 16 (chunk % 4) + 0..15) and writes them as two 16-byte bf16 chunks of
    // the row at the 128-byte swizzle positions (chunk j of row r at
    // j ^ (r % 8)), then arrives on the stage's full barrier (kConvWarps
    // arrivals complete it; for a LoRA block warp 6's arrival also carries
    // the byte count of the B-factor tile).
    constexpr int kRows = 128 / C::kConvWarps;
    const int cw = warp - 6;
    const uint64_t pol_b = l2_policy_evict_last();
    uint32_t sa = 0, pha = 0, s8 = 0, ph8 = 0, armed = 0, armed_parity = 0;
    bool ok = true;
    for (int w = unit0; w < total_work && ok; w += unit_step) {
      if (__shfl_sync(kFullMask, *abort_flag, 0)) break;
      const Work wk = decode_work<BN>(w, crank, CL, s_off, s_ts, p.E, FBg);
      uint64_t amask = use_lora ? tile_adapter_mask<BN>(p.row_adapter, wk.row0, wk.nrows, lane) : 0;
      const int nblocks = nk + __popcll(amask) * lkb;
      int adapter = -1, j = 0;
      for (int b = 0; b < nblocks; ++b) {
        if (b >= nk && j == 0) {  // next LoRA block: adapters in ascending order
          adapter = __ffsll(static_cast<long long>(amask)) - 1;
          amask &= amask - 1;
        }
        uint8_t* sA = smem + sa * C::kABytes;
        if (lane == 0) {
          int site = kWaitConvEmpty;
          ok = wait_or_abort(&empty[sa], pha ^ 1, p.timeout_ns, abort_flag);
          if (ok && b < nk) {
            ok = wait_or_abort(&full8[s8], ph8, p.timeout_ns, abort_flag);
            site = kWaitConvFull8;
            // a main block reuses the stage: its earlier B-factor load (if
            // any) was consumed, so nothing of it is left to drain
            armed &= ~(1u << sa);
          }
          if (ok && b >= nk && cw == 0) {  // LoRA block: the B factor tile (bf16) to the A stage
            const int64_t frow = static_cast<int64_t>(adapter) * p.lb_row_stride_adapter +
                                 static_cast<int64_t>(wk.e) * p.lb_row_stride_expert;
            mbar_arrive_expect_tx(&full[sa], C::kABytes);
            load_lora_b_block<MODE, false>(sA, &tm_lb, &full[sa], 0u, j * 64, frow, wk.fb, p.n_feat,
                                           pol_b);
            armed |= 1u << sa;
            armed_parity = (armed_parity & ~(1u << sa)) | (pha << sa);
          }
          if (!ok && !*abort_flag)
            raise_timeout_at(p.status, abort_flag, site, w, b, site == kWaitConvFull8 ? s8 : sa);
        }
        ok = __shfl_sync(kFullMask, ok, 0);
        if (!ok) break;
        if (b < nk) {
          const uint8_t* src8 = w8ring + s8 * C::kW8Stage;
          const int kblk = (b * 64) >> 7;
#pragma unroll
          for (int i = 0; i < kRows / 8; ++i) {
            const int c = 4 * kRows * cw + lane + 32 * i;
            const int r = c >> 2, part = c & 3;
            int wrow;  // the weight row behind tile row r
            if (MODE == kGateUp) wrow = ((r >> 4) & 1) * p.n_feat + wk.fb * 64 + (r >> 5) * 16 + (r & 15);
            else wrow = wk.fb * 128 + r;
            const float sc = wrow < p.rows_per_expert
                                 ? __ldg(p.w_scale + (static_cast<size_t>(wk.e) * p.scale_nb + (wrow >> 7)) *
                                                         p.scale_kb + kblk)
                                 : 0.f;
            const uint4 raw = *reinterpret_cast<const uint4*>(src8 + c * 16);
            const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
            uint32_t ov[8];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(
                  static_cast<__nv_fp8x2_storage_t>(wv[u] & 0xFFFFu), __NV_E4M3);
              const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(
                  static_cast<__nv_fp8x2_storage_t>(wv[u] >> 16), __NV_E4M3);
              const float2 flo = __half22float2(__half2(lo));
              const float2 fhi = __half22float2(__half2(hi));
              const __nv_bfloat162 blo = __floats2bfloat162_rn(flo.x * sc, flo.y * sc);
              const __nv_bfloat162 bhi = __floats2bfloat162_rn(fhi.x * sc, fhi.y * sc);
              ov[2 * u] = *reinterpret_cast<const uint32_t*>(&blo);
              ov[2 * u + 1] = *reinterpret_cast<const uint32_t*>(&bhi);
            }
            uint8_t* rowp = sA + r * 128;
            const int j0 = 2 * part;
            *reinterpret_cast<uint4*>(rowp + ((j0 ^ (r & 7)) << 4)) = make_uint4(ov[0], ov[1], ov[2], ov[3]);
            *reinterpret_cast<uint4*>(rowp + (((j0 + 1) ^ (r & 7)) << 4)) =
                make_uint4(ov[4], ov[5], ov[6], ov[7]);
          }
          fence_proxy_async_shared();  // the tensor cores read what this thread wrote
        }
        __syncwarp();
        if (lane == 0 && !(b >= nk && cw == 0)) mbar_arrive(&full[sa]);
        if (b >= nk) j = (j + 1 == lkb) ? 0 : j + 1;
        if (++s8 == C::kStages8) {  // one ring stage per block, main and LoRA
          s8 = 0;
          ph8 ^= 1;
        }
        if (++sa == C::kStages) {
          sa = 0;
          pha ^= 1;
        }
      }
    }
    if (lane == 0 && cw == 0) {  // every load issued must have landed before the CTA leaves
      const uint64_t lim = *abort_flag ? 1000000ull : p.timeout_ns;
      for (int s = 0; s < C::kStages; ++s)
        if (armed & (1u << s))
          if (!mbar_wait(&full[s], (armed_parity >> s) & 1u, lim)) note_drain_timeout(p.status, kWaitDrainConv, s);
    }
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  // No CTA leaves while a peer may still signal its barriers or write its
  // shared memory.
  if (CL > 1) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after_sync();
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, C::kTmemCols);  // collective with the peer
    else tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

int gemm_ctas_per_sm(int bn) {
  switch (bn) {
    case 16: return GemmCfg<16>::kCtasPerSm;
    case 32: return GemmCfg<32>::kCtasPerSm;
    case 64: return GemmCfg<64>::kCtasPerSm;
    case 128: return GemmCfg<128>::kCtasPerSm;
    default: return GemmCfg<256>::kCtasPerSm;
  }
}

int gemm_stage_count(int bn, bool pair) {
  switch (bn) {
    case 16: return GemmCfg<16>::kStages;
    case 32: return GemmCfg<32>::kStages;
    case 64: return GemmCfg<64>::kStages;
    case 128: return pair ? GemmCfg<128, true>::kStages : GemmCfg<128>::kStages;
    default: return pair ? GemmCfg<256, true>::kStages : GemmCfg<256>::kStages;
  }
}

size_t gemm_smem_bytes(int bn, bool pair) {
  switch (bn) {
    case 16: return GemmCfg<16>::kSmemBytes;
    case 32: return GemmCfg<32>::kSmemBytes;
    case 64: return GemmCfg<64>::kSmemBytes;
    case 128: return pair ? GemmCfg<128, true>::kSmemBytes : GemmCfg<128>::kSmemBytes;
    default: return pair ? GemmCfg<256, true>::kSmemBytes : GemmCfg<256>::kSmemBytes;
  }
}

template <int BN, int MODE, int CL, bool PAIR, bool W8 = false>
static cudaError_t launch_one(const CUtensorMap& tm_w, const CUtensorMap& tm_x,
                              const CUtensorMap& tm_lb, const CUtensorMap& tm_lu,
                              const CUtensorMap& tm_xs, const CUtensorMap& tm_lus,
                              const GemmParams& p, int grid, cudaStream_t s) {
  using C = GemmCfg<BN, PAIR, W8>;
  auto kern = expert_gemm_kernel<BN, MODE, CL, PAIR, W8>;
  const int smem = C::kSmemBytes;
  cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(kern), smem);
  if (err != cudaSuccess) return err;
  if (CL == 1)
    return launch_pdl(kern, dim3(grid), dim3(C::kThreads), smem, s, tm_w, tm_x, tm_lb, tm_lu, tm_xs, tm_lus,
                      p);

  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // The persistent grid is as many clusters as can be resident at once.
  cfg.gridDim = dim3(CL * 64);
  int max_clusters = 0;
  err = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg);
  if (err != cudaSuccess) return err;
  int clusters = grid / CL;
  if (max_clusters > 0 && clusters > max_clusters) clusters = max_clusters;
  if (clusters < 1) clusters = 1;
  cfg.gridDim = dim3(clusters * CL);
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, tm_w, tm_x, tm_lb, tm_lu, tm_xs, tm_lus, p);
}

// Wide token tiles run as CTA pairs (cta_group::2): each SM then lands half
// of the token tile per stage, which leaves room for deeper stages.
bool gemm_use_pair(int bn) { return bn == 256; }

cudaError_t launch_expert_gemm(int mode, int bn, bool pair, bool w8, const CUtensorMap& tm_w,
                               const CUtensorMap& tm_x, const CUtensorMap& tm_lb,
                               const CUtensorMap& tm_lu, const CUtensorMap& tm_xs,
                               const CUtensorMap& tm_lus, const GemmParams& p, int grid,
                               cudaStream_t s) {
  const int cl = pair ? 2 : 1;
  if (w8) {
    if (pair) return cudaErrorInvalidValue;
#define MOE_GEMM_W8_CASE(BNV)                                                                     \
    if (bn == BNV)                                                                                \
      return mode == kGateUp                                                                      \
                 ? launch_one<BNV, kGateUp, 1, false, true>(tm_w, tm_x, tm_lb, tm_lu, tm_xs, tm_lus, p, grid, s) \
                 : launch_one<BNV, kDown, 1, false, true>(tm_w, tm_x, tm_lb, tm_lu, tm_xs, tm_lus, p, grid, s);
    MOE_GEMM_W8_CASE(16)
    MOE_GEMM_W8_CASE(32)
    MOE_GEMM_W8_CASE(64)
    MOE_GEMM_W8_CASE(128)
    MOE_GEMM_W8_CASE(256)
#undef MOE_GEMM_W8_CASE
    return cudaErrorInvalidValue;
  }
#define MOE_GEMM_CASE(BNV, CLV, PV)                                                               \
  if (bn == BNV && cl == CLV && pair == PV)                                                       \
    return mode == kGateUp                                                                        \
               ? launch_one<BNV, kGateUp, CLV, PV>(tm_w, tm_x, tm_lb, tm_lu, tm_xs, tm_lus, p, grid, s)          \
               : launch_one<BNV, kDown, CLV, PV>(tm_w, tm_x, tm_lb, tm_lu, tm_xs, tm_lus, p, grid, s);
  MOE_GEMM_CASE(16, 1, false)
  MOE_GEMM_CASE(32, 1, false)
  MOE_GEMM_CASE(64, 1, false)
  MOE_GEMM_CASE(128, 1, false)
  MOE_GEMM_CASE(256, 1, false)
  MOE_GEMM_CASE(128, 2, true)
  MOE_GEMM_CASE(256, 2, true)
#undef MOE_GEMM_CASE
  return cudaErrorInvalidValue;
}

}  // namespace moe
