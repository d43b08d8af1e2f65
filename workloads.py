"""Seeded synthetic inputs for the routed MoE-LoRA layer forward.

This module only draws random numbers and lays them out; it holds none of the
layer's arithmetic.  Both sides of every parity check (the CPU oracle and the
CUDA library) receive the arrays built here.

The shapes mirror a 30B-A3B-class MoE layer (hidden 2048, expert intermediate
768, 128 experts, top-8), the model the LoRA perf tables of
"[WIP][LoRA] BF16 support for the experimental_sgl_trtllm MoE-LoRA path &
lora expert_outer_shared" (yushengsu-thu/sglang#4, "Verification" and the
Qwen3-30B-A3B decode perf matrix) were measured on.  No trained weights or
datasets exist here, so every tensor is drawn from the stated distribution.

Draw order for one workload (one ``numpy.random.default_rng(seed)``):
  1. router logits [T, E] ~ N(0, 1) float32; skewed configs then draw a
     per-expert bias [E] ~ N(0, bias_sigma) and add it to the logits;
  2. hidden [T, H] ~ N(0, 1), rounded to bf16 (round-to-nearest-even);
  3. w13 [E, 2I, H] then w2 [E, H, I] ~ N(0, 0.02) -> bf16, drawn one expert
     at a time;
  4. LoRA factors ~ N(0, 0.02) -> bf16 in the order A_gu, B_gu, A_dn, B_dn
     (shared-outer factors have no expert axis);
  5. token_lora_mapping [T] int32, uniform over the config's adapter set
     (-1 = no adapter).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    I: int
    E: int
    top_k: int
    num_adapters: int
    rank: int
    scaling: float
    map_lo: int            # token_lora_mapping drawn uniformly from [map_lo, map_hi]
    map_hi: int
    shared_outer: bool = False   # gate_up A and down B shared across experts
    bias_sigma: float = 0.0      # per-expert router bias std (0 = none)
    seed: int = 0


# The five synthetic layers.  The first is small enough for the oracle to run
# in well under a second; the other four use the 30B-A3B layer shape.
WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_T8", T=8, H=256, I=128, E=8, top_k=2, num_adapters=2,
                 rank=8, scaling=2.0, map_lo=-1, map_hi=1),
        Workload("decode_T16", T=16, H=2048, I=768, E=128, top_k=8,
                 num_adapters=4, rank=16, scaling=2.0, map_lo=-1, map_hi=3),
        Workload("decode_T64_mixed8", T=64, H=2048, I=768, E=128, top_k=8,
                 num_adapters=8, rank=16, scaling=2.0, map_lo=0, map_hi=7),
        Workload("prefill_T4096", T=4096, H=2048, I=768, E=128, top_k=8,
                 num_adapters=1, rank=16, scaling=2.0, map_lo=0, map_hi=0),
        Workload("skewed_T256_shared_outer_r64", T=256, H=2048, I=768, E=128,
                 top_k=8, num_adapters=4, rank=64, scaling=2.0, map_lo=-1,
                 map_hi=3, shared_outer=True, bias_sigma=2.0),
    ]
}
WORKLOAD_ORDER = list(WORKLOADS)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits.

    Used only to store the drawn inputs in bf16.  Inputs here are finite.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def _normal_bf16(rng, shape, std):
    return f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))


@dataclasses.dataclass
class LayerInputs:
    """One layer's inputs.  bf16 tensors are held as uint16 bit patterns.

    LoRA factor layouts (row-major, rows contiguous within one factor):
      A_gu [A, E, r, H]  (shared-outer: [A, r, H])
      B_gu [A, E, 2I, r]
      A_dn [A, E, r, I]
      B_dn [A, E, H, r]  (shared-outer: [A, H, r])
    A factor is addressed as base + a*stride_adapter + e*stride_expert (in
    elements); a shared factor has stride_expert = 0.
    """
    wl: Workload
    logits: np.ndarray        # float32 [T, E]
    hidden: np.ndarray        # uint16  [T, H]
    w13: np.ndarray           # uint16  [E, 2I, H]
    w2: np.ndarray            # uint16  [E, H, I]
    A_gu: Optional[np.ndarray]
    B_gu: Optional[np.ndarray]
    A_dn: Optional[np.ndarray]
    B_dn: Optional[np.ndarray]
    mapping: np.ndarray       # int32   [T]

    def factor_strides(self):
        """(sA_adapter, sA_expert, sB_adapter, sB_expert) in elements, per projection."""
        wl = self.wl
        H, I, E, r = wl.H, wl.I, wl.E, wl.rank
        gu_a = (r * H, 0) if wl.shared_outer else (E * r * H, r * H)
        gu_b = (E * 2 * I * r, 2 * I * r)
        dn_a = (E * r * I, r * I)
        dn_b = (H * r, 0) if wl.shared_outer else (E * H * r, H * r)
        return {"gate_up": gu_a + gu_b, "down": dn_a + dn_b}


def make_inputs(wl: Workload, T: Optional[int] = None, seed: Optional[int] = None) -> LayerInputs:
    """Draw one layer's inputs in the documented order.  ``T`` overrides the token count."""
    T = wl.T if T is None else T
    rng = np.random.default_rng(wl.seed if seed is None else seed)
    H, I, E, A, r = wl.H, wl.I, wl.E, wl.num_adapters, wl.rank

    logits = rng.standard_normal((T, E), dtype=np.float32)
    if wl.bias_sigma > 0:
        bias = rng.standard_normal((E,), dtype=np.float32) * np.float32(wl.bias_sigma)
        logits = (logits + bias[None, :]).astype(np.float32)
    hidden = _normal_bf16(rng, (T, H), 1.0)

    w13 = np.empty((E, 2 * I, H), dtype=np.uint16)
    for e in range(E):
        w13[e] = _normal_bf16(rng, (2 * I, H), 0.02)
    w2 = np.empty((E, H, I), dtype=np.uint16)
    for e in range(E):
        w2[e] = _normal_bf16(rng, (H, I), 0.02)

    if A > 0 and r > 0:
        A_gu = _normal_bf16(rng, (A, r, H) if wl.shared_outer else (A, E, r, H), 0.02)
        B_gu = _normal_bf16(rng, (A, E, 2 * I, r), 0.02)
        A_dn = _normal_bf16(rng, (A, E, r, I), 0.02)
        B_dn = _normal_bf16(rng, (A, H, r) if wl.shared_outer else (A, E, H, r), 0.02)
    else:
        A_gu = B_gu = A_dn = B_dn = None

    mapping = rng.integers(wl.map_lo, wl.map_hi + 1, size=(T,), dtype=np.int64).astype(np.int32)
    return LayerInputs(wl, logits, hidden, w13, w2, A_gu, B_gu, A_dn, B_dn, mapping)


def small_workload(name="custom", T=8, H=64, I=32, E=4, top_k=2, num_adapters=2, rank=8,
                   scaling=2.0, map_lo=-1, map_hi=1, shared_outer=False, bias_sigma=0.0, seed=0):
    """A workload of arbitrary (small) shape, for edge cases and brute-force checks."""
    return Workload(name, T, H, I, E, top_k, num_adapters, rank, scaling, map_lo, map_hi,
                    shared_outer, bias_sigma, seed)


FP8_BLOCK = 128          # weight block (rows x K) sharing one scale
FP8_E4M3_MAX = 448.0    # largest finite float8 e4m3 value


def quantize_fp8_blocks(w_bits: np.ndarray):
    """Block-quantize bf16 weights [E, N, K] (uint16 bits) to float8 e4m3.

    How an FP8 block-scaled checkpoint is made (upstream of the layer): per
    expert and 128 x 128 block of (rows, K), scale = max|w| / 448 (1 for an
    all-zero block) and q = e4m3(w / scale), rounded to nearest even by
    torch's float8_e4m3fn conversion.  Returns (q bits uint8 [E, N, K],
    scales float32 [E, ceil(N/128), ceil(K/128)]).
    """
    import torch
    E, N, K = w_bits.shape
    B = FP8_BLOCK
    nb, kb = (N + B - 1) // B, (K + B - 1) // B
    w = (w_bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    pad = np.zeros((E, nb * B, kb * B), dtype=np.float32)
    pad[:, :N, :K] = w
    blocks = pad.reshape(E, nb, B, kb, B)
    amax = np.abs(blocks).max(axis=(2, 4))
    scale = np.where(amax > 0, amax / np.float32(FP8_E4M3_MAX), np.float32(1.0)).astype(np.float32)
    scaled = blocks / scale[:, :, None, :, None]
    q = torch.from_numpy(np.ascontiguousarray(scaled)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    q = q.reshape(E, nb * B, kb * B)[:, :N, :K]
    return np.ascontiguousarray(q), scale


def fp8_weights(inp: "LayerInputs"):
    """(w13_q, w13_scale, w2_q, w2_scale) for a layer's bf16 weights."""
    q13, s13 = quantize_fp8_blocks(inp.w13)
    q2, s2 = quantize_fp8_blocks(inp.w2)
    return q13, s13, q2, s2


def shard_experts(inp: "LayerInputs", offset: int, count: int) -> "LayerInputs":
    """The inputs of one expert-parallel shard: experts [offset, offset + count).

    Weights and per-expert LoRA factors are sliced along the expert axis (a
    shared factor is kept whole); the router logits keep all experts, since
    routing is global.  ``wl.E`` becomes ``count``, the number of local
    experts.
    """
    sl = slice(offset, offset + count)
    shared = inp.wl.shared_outer

    def cut(x, keep_whole=False):
        if x is None:
            return None
        return np.ascontiguousarray(x if keep_whole else x[:, sl])

    return LayerInputs(
        wl=dataclasses.replace(inp.wl, E=count),
        logits=inp.logits, hidden=inp.hidden,
        w13=np.ascontiguousarray(inp.w13[sl]), w2=np.ascontiguousarray(inp.w2[sl]),
        A_gu=cut(inp.A_gu, keep_whole=shared), B_gu=cut(inp.B_gu),
        A_dn=cut(inp.A_dn), B_dn=cut(inp.B_dn, keep_whole=shared),
        mapping=inp.mapping)


def make_peft_adapters(wl: Workload, specs, seed: int = 7):
    """Draw PEFT-style adapters for the layer shape of ``wl``.

    ``specs`` is a list, one entry per adapter slot, of (kind, rank, alpha):
    kind "separate" draws one LoRA pair per projection (gate, up, down);
    kind "fused" draws one pair on the fused gate_up projection and one on
    down.  Factors ~ N(0, 0.02) -> bf16 bits; scaling = alpha / rank.
    Order: for each adapter in turn, its gate/up (or gate_up) A then B, then
    down A then B.
    """
    rng = np.random.default_rng(seed)
    H, I, E = wl.H, wl.I, wl.E
    out = []
    for kind, r, alpha in specs:
        ad = {"scaling": float(alpha) / float(r)}
        if kind == "separate":
            ad["gate"] = (_normal_bf16(rng, (E, r, H), 0.02), _normal_bf16(rng, (E, I, r), 0.02))
            ad["up"] = (_normal_bf16(rng, (E, r, H), 0.02), _normal_bf16(rng, (E, I, r), 0.02))
        else:
            ad["gate_up"] = (_normal_bf16(rng, (E, r, H), 0.02), _normal_bf16(rng, (E, 2 * I, r), 0.02))
        ad["down"] = (_normal_bf16(rng, (E, r, I), 0.02), _normal_bf16(rng, (E, H, r), 0.02))
        out.append(ad)
    return out
