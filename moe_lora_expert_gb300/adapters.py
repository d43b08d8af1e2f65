"""Packing of PEFT-style adapters into the library's LoRA factor layout.

The library takes, per projection, one rank-``rank`` pair per (adapter,
expert): gate_up A [A, E, rank, H], B [A, E, 2I, rank]; down A [A, E, rank, I],
B [A, E, H, rank], plus one scale per adapter.  Adapters as trained carry a
pair per projection (gate_proj, up_proj, down_proj) with their own rank and
scale alpha / r.  This module lays them out once, at load time:

- separate gate and up pairs become the block-diagonal pair of rank 2r on the
  fused projection: A = [A_gate; A_up], B = [[B_gate, 0], [0, B_up]], which
  gives exactly the two per-projection deltas;
- adapters of smaller rank are padded with zero rows of A and zero columns of
  B to the common rank (a multiple of 8), which adds exactly 0;
- the per-adapter scales go to ``moe_lora_args_t.adapter_scaling``.

Device tensors only; nothing here runs per forward.
"""
from __future__ import annotations

from typing import Dict, List, Sequence, Tuple


def _round8(v: int) -> int:
    return (v + 7) // 8 * 8


def packed_rank(adapters: Sequence[Dict]) -> int:
    """Common rank of the packed factors (gate_up and down share it)."""
    r = 0
    for ad in adapters:
        if "gate_up" in ad:
            r = max(r, ad["gate_up"][0].shape[1])
        else:
            r = max(r, ad["gate"][0].shape[1] + ad["up"][0].shape[1])
        r = max(r, ad["down"][0].shape[1])
    return _round8(r)


def pack_adapters(adapters: Sequence[Dict], E: int, H: int, I: int):
    """adapters[a]: dict of bf16 CUDA tensors, per expert:
         'gate': (A [E, r, H], B [E, I, r]) and 'up': (A, B)   (separate), or
         'gate_up': (A [E, r, H], B [E, 2I, r])                 (fused);
         'down': (A [E, r, I], B [E, H, r]); 'scaling': float.
    Returns (A_gu, B_gu, A_dn, B_dn, scalings) ready for MoeLoraLayer.
    """
    import torch
    n = len(adapters)
    R = packed_rank(adapters)
    dev = next(iter(adapters[0]["down"])).device
    kw = dict(dtype=torch.bfloat16, device=dev)
    A_gu = torch.zeros((n, E, R, H), **kw)
    B_gu = torch.zeros((n, E, 2 * I, R), **kw)
    A_dn = torch.zeros((n, E, R, I), **kw)
    B_dn = torch.zeros((n, E, H, R), **kw)
    scalings: List[float] = []
    for a, ad in enumerate(adapters):
        if "gate_up" in ad:
            A, B = ad["gate_up"]
            r = A.shape[1]
            A_gu[a, :, :r] = A
            B_gu[a, :, :, :r] = B
        else:
            (Ag, Bg), (Au, Bu) = ad["gate"], ad["up"]
            rg, ru = Ag.shape[1], Au.shape[1]
            A_gu[a, :, :rg] = Ag
            A_gu[a, :, rg:rg + ru] = Au
            B_gu[a, :, :I, :rg] = Bg
            B_gu[a, :, I:, rg:rg + ru] = Bu
        Ad, Bd = ad["down"]
        rd = Ad.shape[1]
        A_dn[a, :, :rd] = Ad
        B_dn[a, :, :, :rd] = Bd
        scalings.append(float(ad["scaling"]))
    return A_gu, B_gu, A_dn, B_dn, scalings
