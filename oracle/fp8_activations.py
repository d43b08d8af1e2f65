"""FP8 activations of the pages' FP8 block-scale path (oracle).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only the tests may
import it; the CUDA library does not, and no code is shared with it.

Source: "[WIP][LoRA] BF16 support for the experimental_sgl_trtllm MoE-LoRA
path & lora expert_outer_shared" (yushengsu-thu/sglang#4), Flow 1(A): the
bf16 path is drawn as the FP8 one minus two steps, a
``per_token_group_quant_fp8`` of the hidden input before the gate_up GEMM
and a post-activation quant before the down GEMM.

Reading R12 (the pages give neither step's arithmetic; the plainest reading
of the function name, and of the sglang function of that name):
  * per token (row) and group of 128 consecutive columns, in float32:
    scale = max(amax, 1e-10) / 448 and code = e4m3(x / scale), rounded to the
    nearest finite e4m3 value, ties to an even mantissa, magnitudes above 448
    to 448 (the quotient can exceed 448 by one float32 rounding);
  * the quantized value is code * scale;
  * the activation is quantized from its float32 value (the activation
    kernel computes it in float32);
  * the LoRA deltas read the unquantized tensors: the gate_up delta the bf16
    hidden row, the down delta the activation (the pages feed the LoRA from
    the bf16 hidden states and from ``activation_lora_input``);
  * the expert weights are the block-scaled e4m3 ones of reading R11.
Every other step is the bf16 forward's, in float64.
"""
from __future__ import annotations

import numpy as np

from .moe_lora_oracle import (bf16_bits_to_f64, dequant_fp8_blocks, e4m3_to_f64,
                              f64_to_bf16_bits, route_topk, silu)

E4M3_MAX = 448.0
ACT_GROUP = 128
ACT_EPS = 1e-10

# the non-negative finite codes, 0x00 .. 0x7E, in ascending value order
_POS_CODES = np.arange(0, 0x7F, dtype=np.uint8)


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """Codes (uint8) of the finite e4m3 values nearest to ``v`` (float64
    holding float32 values): ties go to the code with an even mantissa
    (the lower code bit), magnitudes above 448 to 448; the sign bit is the
    sign of ``v``, negative zero included."""
    v = np.asarray(v, dtype=np.float64)
    vals = e4m3_to_f64(_POS_CODES)
    a = np.minimum(np.abs(v), E4M3_MAX)
    hi = np.minimum(np.searchsorted(vals, a, side="left"), len(vals) - 1)  # vals[hi] >= a
    lo = np.maximum(hi - 1, 0)
    d_hi = vals[hi] - a
    d_lo = a - vals[lo]
    take_lo = (lo != hi) & ((d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0)))
    code = np.where(take_lo, lo, hi).astype(np.uint8)
    return code | np.where(np.signbit(v), 0x80, 0).astype(np.uint8)


def quant_fp8_token_groups(x32: np.ndarray, group: int = ACT_GROUP):
    """Reading R12 on a [rows, K] float32 matrix: returns (codes uint8
    [rows, K], scales float32 [rows, ceil(K / group)])."""
    x32 = np.asarray(x32, dtype=np.float32)
    rows, K = x32.shape
    G = -(-K // group)
    codes = np.zeros((rows, K), dtype=np.uint8)
    scales = np.zeros((rows, G), dtype=np.float32)
    for g in range(G):
        blk = x32[:, g * group:(g + 1) * group]
        amax = np.max(np.abs(blk), axis=1)
        s = np.maximum(amax, np.float32(ACT_EPS)) / np.float32(E4M3_MAX)  # float32 division
        q = blk / s[:, None]                                               # float32 division
        codes[:, g * group:(g + 1) * group] = e4m3_encode(q.astype(np.float64))
        scales[:, g] = s
    return codes, scales


def dequant_token_groups(codes: np.ndarray, scales: np.ndarray, group: int = ACT_GROUP) -> np.ndarray:
    """code value times its group's scale, float64."""
    v = e4m3_to_f64(codes)
    s = np.repeat(np.asarray(scales, dtype=np.float64), group, axis=1)[:, :v.shape[1]]
    return v * s


def expert_slot_w8a8(x, xq, w13_e, w2_e, lora_gu, lora_dn, adapter, expert, scaling):
    """One (token, expert) evaluation of the FP8 path, float64: the base GEMMs
    read the quantized hidden row ``xq`` and the quantized activation, the
    LoRA deltas the unquantized ones."""
    I = w2_e.shape[1]
    g = w13_e @ xq
    if adapter >= 0 and lora_gu is not None:
        g = g + scaling * (lora_gu.b(adapter, expert) @ (lora_gu.a(adapter, expert) @ x))
    h = silu(g[:I]) * g[I:]
    hc, hs = quant_fp8_token_groups(h.astype(np.float32)[None, :])
    y = w2_e @ dequant_token_groups(hc, hs)[0]
    if adapter >= 0 and lora_dn is not None:
        y = y + scaling * (lora_dn.b(adapter, expert) @ (lora_dn.a(adapter, expert) @ h))
    return g, h, y


def moe_lora_forward_w8a8(hidden_bits, logits, w13_q, w13_scale, w2_q, w2_scale, mapping, top_k,
                          scaling=2.0, lora_gu=None, lora_dn=None, tokens=None):
    """The layer forward of the FP8 path (readings R11, R12): routing and
    finalize as in the bf16 forward; each touched expert's weights
    dequantized once; the slot sum in slot order."""
    hidden_bits = np.asarray(hidden_bits)
    T, H = hidden_bits.shape
    x_all = bf16_bits_to_f64(hidden_bits)
    xc, xs = quant_fp8_token_groups(x_all.astype(np.float32))
    xq_all = dequant_token_groups(xc, xs)
    E = w13_q.shape[0]
    ids, w = route_topk(logits, top_k)
    tokens = list(range(T)) if tokens is None else list(tokens)
    by_expert = {}
    for t in tokens:
        for j in range(top_k):
            e = int(ids[t, j])
            if 0 <= e < E:
                by_expert.setdefault(e, []).append((t, j))
    y_slot = {}
    for e in sorted(by_expert):
        w13_e = dequant_fp8_blocks(w13_q[e:e + 1], w13_scale[e:e + 1])[0]
        w2_e = dequant_fp8_blocks(w2_q[e:e + 1], w2_scale[e:e + 1])[0]
        for (t, j) in by_expert[e]:
            _, _, y = expert_slot_w8a8(x_all[t], xq_all[t], w13_e, w2_e, lora_gu, lora_dn,
                                       int(mapping[t]), e, scaling)
            y_slot[(t, j)] = y
    out = np.zeros((len(tokens), H), dtype=np.float64)
    for i, t in enumerate(tokens):
        acc = np.zeros(H, dtype=np.float64)
        for j in range(top_k):
            if (t, j) in y_slot:
                acc = acc + w[t, j] * y_slot[(t, j)]
        out[i] = acc
    return {"ids": ids, "w": w, "tokens": tokens, "out64": out, "out_bf16": f64_to_bf16_bits(out)}
