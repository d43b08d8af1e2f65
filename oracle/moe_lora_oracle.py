"""CPU oracle for the routed BF16 MoE layer forward with per-token multi-adapter LoRA.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  The CUDA library
never calls it, and it shares no code with the CUDA library.

It is a plain, slow, float64 restatement of the pipeline that the pages
describe, one step per function, in the pages' order:

  routing -> permute (gather) -> gate_up GEMM (+ gate_up LoRA delta)
  -> LoRA-aware SwiGLU -> down GEMM (+ down LoRA delta) -> finalize

Sources (page title, then section):
  [P1] prhub digest of sgl-project/sglang#28953 -- excerpts of
       ``lora_dispatch.py`` (single-stream docstring "routing -> gather ->
       gate_up GEMM -> LoRA-aware activation -> down GEMM -> finalize") and
       ``core.py`` (``trtllm_bf16_routed_moe_lora`` signature and docstring).
  [P2] "[WIP][LoRA] BF16 support for the experimental_sgl_trtllm MoE-LoRA path
       & lora expert_outer_shared" (yushengsu-thu/sglang#4) -- "Files changed"
       table (launcher row: activation "adds gate_up_lora_delta pre-SwiGLU";
       dispatch row: down-LoRA merged after the down GEMM), Flow 1(A) sequence
       diagram (gate_up shrink+expand -> delta; down LoRA with the routed
       weight), Flow 2 "Shared-outer (TML) LoRA" (shared gate_up A and shared
       down B, addressed by adapter id only).
  [P3] prhub report on sgl-project/sglang#28091 -- "关键源码片段" snippet sizing
       the gate_up LoRA intermediate as [tokens, top_k, lora_a.shape[2]].

Readings taken where the pages are silent (each one is also listed in the
design notes of the repository):
  R1 routing: softmax over the router logits, top-k, renormalise over the
     selected experts.  Selection compares the raw float32 logits (softmax is
     monotone), ties go to the lower expert id, slots are ordered by
     descending logit.  Weights are exp(l_j - m) / sum_j' exp(l_j' - m) with
     m the largest selected logit.
  R3 w13 rows [0, I) are the gate projection, rows [I, 2I) the up
     projection; h = silu(gate) * up, silu(z) = z / (1 + exp(-z)).
  R4 one rank-r LoRA pair per (adapter, expert) on the fused gate_up
     projection: A_gu [r, H], B_gu [2I, r]; one on down: A_dn [r, I],
     B_dn [H, r].
  R5 each delta is scaling * B (A x), added to the base GEMM result; the
     gate_up delta is added before SwiGLU.
  R6 the down delta is multiplied by the routing weight like the base
     expert output, so finalize sums w * (y + delta).
  R7 shared-outer: gate_up A is [r, H] per adapter, down B is [H, r] per
     adapter; the inner factors stay per expert.
  R8 no routed scaling factor (1.0), no shared expert.
  R9 mapping -1 (or rank 0, or no adapters) means the delta is absent.
Every intermediate is float64; the only rounding is the final bf16
round-to-nearest-even of the output.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np


# ---------------------------------------------------------------------------
# bf16 <-> float64 (exact decode; round-to-nearest-even encode)
# ---------------------------------------------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64.  Exact: bf16 is the top half of float32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float64 -> bf16 bits, rounding to the nearest bf16 value, ties to even.

    Written out on the exact binary value: the float64 is first split into
    sign, exponent and 53-bit significand, so no double rounding through
    float32 can occur.  Normal and subnormal bf16 results, overflow to inf,
    and NaN are handled.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    flat_in = x.ravel()
    flat_out = out.ravel()
    for i, v in enumerate(flat_in):
        flat_out[i] = _one_f64_to_bf16(float(v))
    return out


def _one_f64_to_bf16(v: float) -> int:
    if math.isnan(v):
        return 0x7FC0
    sign = 0x8000 if math.copysign(1.0, v) < 0 else 0
    a = abs(v)
    if a == 0.0:
        return sign
    if math.isinf(a):
        return sign | 0x7F80
    m, e = math.frexp(a)          # a = m * 2**e, 0.5 <= m < 1
    # bf16 normal: value = 1.f * 2**(E-127), 7 fraction bits; min normal 2**-126.
    exp_unbiased = e - 1          # a = (2m) * 2**(e-1), 1 <= 2m < 2
    if exp_unbiased >= -126:
        # Significand scaled to an integer with 7 fraction bits, then rounded.
        scaled = a / 2.0 ** (exp_unbiased - 7)   # in [128, 256), exact in float64
        q = _round_half_even(scaled)
        if q == 256:              # rounding carried into the next binade
            q = 128
            exp_unbiased += 1
        if exp_unbiased > 127:
            return sign | 0x7F80
        return sign | ((exp_unbiased + 127) << 7) | (q - 128)
    # Subnormal bf16: value = f * 2**-133, f in [0, 127].
    scaled = a / 2.0 ** -133
    q = _round_half_even(scaled)
    if q == 128:                  # rounds up to the smallest normal
        return sign | (1 << 7)
    return sign | q


def _round_half_even(s: float) -> int:
    f = math.floor(s)
    d = s - f
    if d > 0.5 or (d == 0.5 and (int(f) & 1)):
        return int(f) + 1
    return int(f)


# ---------------------------------------------------------------------------
# Step 1: routing  ([P1] lora_dispatch/moe_overlap excerpts take
# ``topk_output.topk_ids / topk_weights`` in the standard format; reading R1)
# ---------------------------------------------------------------------------

def route_topk(logits: np.ndarray, top_k: int):
    """Top-k softmax routing with renormalisation over the selected experts.

    Returns (topk_ids int32 [T, k], topk_w float64 [T, k]).
    """
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    ids = np.zeros((T, top_k), dtype=np.int32)
    w = np.zeros((T, top_k), dtype=np.float64)
    for t in range(T):
        row = [float(v) for v in logits[t]]
        # descending logit, ties broken by the lower expert id
        order = sorted(range(E), key=lambda e: (-row[e], e))
        sel = order[:top_k]
        m = row[sel[0]]
        ex = [math.exp(row[e] - m) for e in sel]
        z = sum(ex)
        ids[t] = sel
        w[t] = [v / z for v in ex]
    return ids, w


# ---------------------------------------------------------------------------
# Step 2: permute ([P1] core.py docstring: do_finalize=False returns
# ``expanded_idx_to_permuted_idx``; [P2] launcher row: "moe::dev::permute
# (bf16 gather)")
# ---------------------------------------------------------------------------

def permute(topk_ids: np.ndarray, E: int):
    """Expert-grouped, stable counting-sort permutation of the expanded slots.

    Expanded index x = t*k + j.  expert_offsets[e] = number of slots routed to
    experts < e; expanded_to_permuted[x] = offset[e] + (number of earlier
    slots x' < x routed to the same expert e); permuted_to_expanded is its
    inverse.  Slots with id -1 are dropped (permuted index -1).
    """
    flat = np.asarray(topk_ids, dtype=np.int64).ravel()
    n = flat.size
    counts = [0] * E
    for x in range(n):
        if 0 <= flat[x] < E:
            counts[int(flat[x])] += 1
    offsets = [0] * (E + 1)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    seen = [0] * E
    e2p = np.full(n, -1, dtype=np.int32)
    p2e = np.full(n, -1, dtype=np.int32)
    for x in range(n):
        e = int(flat[x])
        if not (0 <= e < E):
            continue
        p = offsets[e] + seen[e]
        seen[e] += 1
        e2p[x] = p
        p2e[p] = x
    return np.asarray(offsets, dtype=np.int32), e2p, p2e


# ---------------------------------------------------------------------------
# Steps 3-7: one expert slot, then the weighted sum.
# ---------------------------------------------------------------------------

def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z * sigmoid(z) = z / (1 + exp(-z))  (reading R3)."""
    return z / (1.0 + np.exp(-z))


class LoraFactors:
    """Per-(adapter, expert) LoRA factors of one projection, held as float64.

    ``A`` is [A, E, r, K] or, when shared across experts, [A, r, K]; ``B`` is
    [A, E, N, r] or, when shared, [A, N, r] (reading R4/R7).
    """

    def __init__(self, A_bits, B_bits, a_shared=False, b_shared=False):
        self.A = bf16_bits_to_f64(A_bits)
        self.B = bf16_bits_to_f64(B_bits)
        self.a_shared = a_shared
        self.b_shared = b_shared

    def a(self, adapter, expert):
        return self.A[adapter] if self.a_shared else self.A[adapter, expert]

    def b(self, adapter, expert):
        return self.B[adapter] if self.b_shared else self.B[adapter, expert]


def expert_slot(x, w13_e, w2_e, lora_gu: Optional[LoraFactors], lora_dn: Optional[LoraFactors],
                adapter: int, expert: int, scaling: float):
    """One (token, expert) evaluation, all in float64.

    g = w13[e] x                       (gate_up GEMM, K = H, N = 2I)
      + s * B_gu (A_gu x)              (gate_up LoRA delta, added pre-SwiGLU)
    h = silu(g[:I]) * g[I:]            (LoRA-aware SwiGLU activation)
    y = w2[e] h                        (down GEMM, K = I, N = H)
      + s * B_dn (A_dn h)              (down LoRA delta)
    Returns (g, h, y).
    """
    I = w2_e.shape[1]
    g = w13_e @ x
    if adapter >= 0 and lora_gu is not None:
        u = lora_gu.a(adapter, expert) @ x
        g = g + scaling * (lora_gu.b(adapter, expert) @ u)
    h = silu(g[:I]) * g[I:]
    y = w2_e @ h
    if adapter >= 0 and lora_dn is not None:
        v = lora_dn.a(adapter, expert) @ h
        y = y + scaling * (lora_dn.b(adapter, expert) @ v)
    return g, h, y


def moe_lora_forward(hidden_bits, logits, w13_bits, w2_bits, mapping, top_k, scaling=2.0,
                     lora_gu: Optional[LoraFactors] = None, lora_dn: Optional[LoraFactors] = None,
                     tokens: Optional[Sequence[int]] = None, keep_intermediates=False,
                     local_expert_offset: int = 0):
    """The whole layer forward for the listed tokens (default: all).

    Expert parallelism (the local_expert_offset / local_num_experts arguments
    of trtllm_bf16_routed_moe_lora, sglang PR #28953 summary page; the slots
    of other ranks' experts carry permuted index -1 there): the router scores
    all logits.shape[1] experts, while w13_bits, w2_bits and the LoRA factors
    hold only experts [local_expert_offset, local_expert_offset + E) and are
    indexed by the local expert.  Slots routed elsewhere contribute nothing,
    so ``out`` is this shard's part of the sum that the downstream all-reduce
    completes (Flow 1(A), "downstream all_reduce (in qwen3_moe)").

    Routing is computed for every token (it is cheap); the expert work and
    the output only for ``tokens``.  The expert loop visits the experts one
    at a time so that each expert's weights are decoded to float64 once; the
    per-slot arithmetic is exactly ``expert_slot``.

    Returns a dict with
      ids, w             routing (all tokens)
      out64 [n, H]       float64 output rows for ``tokens``
      out_bf16 [n, H]    the same rounded to bf16 bits
      and, with keep_intermediates, per (token, slot): g, h, y (float64).
    """
    hidden_bits = np.asarray(hidden_bits)
    T, H = hidden_bits.shape
    E = w13_bits.shape[0]
    ids, w = route_topk(logits, top_k)
    if tokens is None:
        tokens = list(range(T))
    tokens = list(tokens)
    row_of = {t: i for i, t in enumerate(tokens)}
    out = np.zeros((len(tokens), H), dtype=np.float64)
    inter = {}

    # slots grouped by local expert: expert -> [(token, slot)]
    by_expert = {}
    for t in tokens:
        for j in range(top_k):
            e = int(ids[t, j]) - local_expert_offset
            if 0 <= e < E:
                by_expert.setdefault(e, []).append((t, j))

    # y for every slot first; the weighted sum then runs in slot order.
    y_slot = {}
    for e in sorted(by_expert):
        w13_e = bf16_bits_to_f64(w13_bits[e])
        w2_e = bf16_bits_to_f64(w2_bits[e])
        for (t, j) in by_expert[e]:
            x = bf16_bits_to_f64(hidden_bits[t])
            a = int(mapping[t])
            g, h, y = expert_slot(x, w13_e, w2_e, lora_gu, lora_dn, a, e, scaling)
            y_slot[(t, j)] = y
            if keep_intermediates:
                inter[(t, j)] = (g, h, y)

    # Step 7: finalize -- out[t] = sum_j w[t, j] * y[t, j]   (reading R6)
    for t in tokens:
        acc = np.zeros(H, dtype=np.float64)
        for j in range(top_k):
            if (t, j) in y_slot:          # slots of other shards are skipped
                acc = acc + w[t, j] * y_slot[(t, j)]
        out[row_of[t]] = acc

    res = {"ids": ids, "w": w, "tokens": tokens, "out64": out, "out_bf16": f64_to_bf16_bits(out)}
    if keep_intermediates:
        res["intermediates"] = inter
    return res


# ---------------------------------------------------------------------------
# FP8 block-scaled expert weights (the FP8 block-quant checkpoints of the
# pages' sibling path, trtllm_fp8_block_scale_routed_moe_lora, summary of
# "[WIP][LoRA] BF16 support for the experimental_sgl_trtllm MoE-LoRA path &
# lora expert_outer_shared").  Reading: float8 e4m3 (finite-only variant: no
# infinities, 0x7F/0xFF are NaN, max 448) with one float32 scale per 128 x 128
# block of (rows, K); the activations stay bf16.
# ---------------------------------------------------------------------------

def e4m3_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode float8 e4m3 bit patterns (uint8): sign, 4 exponent bits with
    bias 7, 3 mantissa bits; exponent 0 is subnormal (m/8 * 2^-6); exponent 15
    with mantissa 7 is NaN (there is no infinity)."""
    table = np.empty(256, dtype=np.float64)
    for c in range(256):
        sgn = -1.0 if c & 0x80 else 1.0
        e = (c >> 3) & 0xF
        m = c & 0x7
        if e == 0xF and m == 0x7:
            table[c] = np.nan
        elif e == 0:
            table[c] = sgn * (m / 8.0) * 2.0 ** -6
        else:
            table[c] = sgn * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return table[np.asarray(bits, dtype=np.uint8)]


def dequant_fp8_blocks(q_bits: np.ndarray, scale: np.ndarray, block: int = 128) -> np.ndarray:
    """w[e, n, k] = e4m3(q[e, n, k]) * scale[e, n // block, k // block], float64."""
    q = e4m3_to_f64(q_bits)
    E, N, K = q.shape
    s = np.repeat(np.repeat(np.asarray(scale, dtype=np.float64), block, axis=1), block, axis=2)
    return q * s[:, :N, :K]


def f64_weights_to_bf16_bits_exact(w: np.ndarray) -> np.ndarray:
    """float64 weights -> the uint16 layout moe_lora_forward reads, only for
    values that bf16 holds exactly (checked)."""
    bits = (w.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    assert np.array_equal(bf16_bits_to_f64(bits), w), "weights not exact in bf16"
    return bits


def moe_lora_forward_fp8(hidden_bits, logits, w13_q, w13_scale, w2_q, w2_scale, mapping, top_k,
                         scaling=2.0, lora_gu=None, lora_dn=None, tokens=None,
                         local_expert_offset=0):
    """The layer forward with FP8 block-scaled expert weights: each touched
    expert's weights are dequantized (e4m3 value times its block's scale, in
    float64; one expert at a time, to bound memory) and the per-slot
    arithmetic is exactly ``expert_slot``; the slot sum runs in slot order."""
    hidden_bits = np.asarray(hidden_bits)
    T, H = hidden_bits.shape
    E = w13_q.shape[0]
    ids, w = route_topk(logits, top_k)
    tokens = list(range(T)) if tokens is None else list(tokens)
    by_expert = {}
    for t in tokens:
        for j in range(top_k):
            e = int(ids[t, j]) - local_expert_offset
            if 0 <= e < E:
                by_expert.setdefault(e, []).append((t, j))
    y_slot = {}
    for e in sorted(by_expert):
        w13_e = dequant_fp8_blocks(w13_q[e:e + 1], w13_scale[e:e + 1])[0]
        w2_e = dequant_fp8_blocks(w2_q[e:e + 1], w2_scale[e:e + 1])[0]
        for (t, j) in by_expert[e]:
            x = bf16_bits_to_f64(hidden_bits[t])
            _, _, y = expert_slot(x, w13_e, w2_e, lora_gu, lora_dn, int(mapping[t]), e, scaling)
            y_slot[(t, j)] = y
    out = np.zeros((len(tokens), H), dtype=np.float64)
    for i, t in enumerate(tokens):
        acc = np.zeros(H, dtype=np.float64)
        for j in range(top_k):
            if (t, j) in y_slot:
                acc = acc + w[t, j] * y_slot[(t, j)]
        out[i] = acc
    return {"ids": ids, "w": w, "tokens": tokens, "out64": out, "out_bf16": f64_to_bf16_bits(out)}


def forward_inputs_fp8(inp, fp8, tokens=None, with_lora=True):
    """``moe_lora_forward_fp8`` on a ``workloads.LayerInputs`` and its
    (w13_q, w13_scale, w2_q, w2_scale)."""
    gu, dn = factors_from_inputs(inp) if with_lora else (None, None)
    wl = inp.wl
    q13, s13, q2, s2 = fp8
    return moe_lora_forward_fp8(inp.hidden, inp.logits, q13, s13, q2, s2, inp.mapping, wl.top_k,
                                wl.scaling, gu, dn, tokens=tokens)


def factors_from_inputs(inp):
    """Wrap a ``workloads.LayerInputs`` LoRA set as oracle factors (None when absent)."""
    if inp.A_gu is None:
        return None, None
    shared = inp.wl.shared_outer
    gu = LoraFactors(inp.A_gu, inp.B_gu, a_shared=shared, b_shared=False)
    dn = LoraFactors(inp.A_dn, inp.B_dn, a_shared=False, b_shared=shared)
    return gu, dn


def forward_inputs(inp, tokens=None, keep_intermediates=False, with_lora=True,
                   local_expert_offset=0):
    """Run ``moe_lora_forward`` on a ``workloads.LayerInputs`` (for a shard of
    the experts: the sliced inputs and the shard's first expert)."""
    gu, dn = factors_from_inputs(inp) if with_lora else (None, None)
    wl = inp.wl
    return moe_lora_forward(inp.hidden, inp.logits, inp.w13, inp.w2, inp.mapping, wl.top_k,
                            wl.scaling, gu, dn, tokens=tokens, keep_intermediates=keep_intermediates,
                            local_expert_offset=local_expert_offset)


# ---------------------------------------------------------------------------
# General adapters: separate or fused gate/up LoRA, own rank and scale per
# adapter.  Real PEFT adapters carry one LoRA pair per projection (gate_proj,
# up_proj, down_proj) with scale alpha / r.  The pages' fused gate_up delta is
# the special case of one pair on the fused projection (readings R4, R5).
# ---------------------------------------------------------------------------

def expert_slot_general(x, w13_e, w2_e, adapter, expert):
    """One (token, expert) evaluation with a general adapter (or None).

    ``adapter`` is a dict of float64 arrays indexed by expert:
      'scaling': s,
      either 'gate_up': (A [E, r, H], B [E, 2I, r])
      or 'gate': (A [E, r, H], B [E, I, r]) and 'up': (A, B) of the same shapes,
      'down': (A [E, r, I], B [E, H, r]).
    gate = w13[e][:I] x + s B_g (A_g x);  up = w13[e][I:] x + s B_u (A_u x)
    y = w2[e] h + s B_dn (A_dn h),  h = silu(gate) * up.
    """
    I = w2_e.shape[1]
    g = w13_e @ x
    if adapter is not None:
        s = adapter["scaling"]
        if "gate_up" in adapter:
            A, B = adapter["gate_up"]
            g = g + s * (B[expert] @ (A[expert] @ x))
        else:
            Ag, Bg = adapter["gate"]
            Au, Bu = adapter["up"]
            g = g + s * np.concatenate([Bg[expert] @ (Ag[expert] @ x), Bu[expert] @ (Au[expert] @ x)])
    h = silu(g[:I]) * g[I:]
    y = w2_e @ h
    if adapter is not None:
        Ad, Bd = adapter["down"]
        y = y + adapter["scaling"] * (Bd[expert] @ (Ad[expert] @ h))
    return y


def decode_adapter(bits_adapter):
    """bf16-bit arrays of one adapter -> float64 (same structure)."""
    out = {"scaling": float(bits_adapter["scaling"])}
    for key in ("gate_up", "gate", "up", "down"):
        if key in bits_adapter:
            A, B = bits_adapter[key]
            out[key] = (bf16_bits_to_f64(A), bf16_bits_to_f64(B))
    return out


def moe_lora_forward_general(hidden_bits, logits, w13_bits, w2_bits, mapping, top_k, adapters,
                             tokens=None):
    """Layer forward with general adapters (list indexed by adapter slot).

    Routing and the weighted sum are those of ``moe_lora_forward``; each slot
    is ``expert_slot_general``.  Returns (out64 [n, H], out_bf16).
    """
    T, H = np.asarray(hidden_bits).shape
    ids, w = route_topk(logits, top_k)
    tokens = list(range(T)) if tokens is None else list(tokens)
    dec = [decode_adapter(a) for a in adapters]
    by_expert = {}
    for t in tokens:
        for j in range(top_k):
            by_expert.setdefault(int(ids[t, j]), []).append((t, j))
    y_slot = {}
    for e in sorted(by_expert):
        w13_e = bf16_bits_to_f64(w13_bits[e])
        w2_e = bf16_bits_to_f64(w2_bits[e])
        for (t, j) in by_expert[e]:
            a = int(mapping[t])
            y_slot[(t, j)] = expert_slot_general(bf16_bits_to_f64(hidden_bits[t]), w13_e, w2_e,
                                                 dec[a] if a >= 0 else None, e)
    out = np.zeros((len(tokens), H))
    for i, t in enumerate(tokens):
        acc = np.zeros(H)
        for j in range(top_k):
            acc = acc + w[t, j] * y_slot[(t, j)]
        out[i] = acc
    return out, f64_to_bf16_bits(out)
