"""Pins for the CPU oracle, against facts that do not come from the oracle itself.

* a hand-worked example whose output is a closed form derived on paper;
* brute force: every expert evaluated densely with merged weights
  W' = W + s*B*A, selection by a library sort, weights by a full softmax;
* library routines: numpy's stable argsort for routing order and for the
  permutation, torch's float32->bf16 conversion for the rounding;
* special cases: one expert (a plain SwiGLU MLP with LoRA), k = E (a full
  softmax mixture);
* invariants: weights sum to 1, no-adapter / rank-0 / zero-scaling reproduce
  plain MoE, token permutation equivariance;
* planted mistakes: each plausible slip (swapped gate/up, dropped scaling,
  delta after the activation, wrong tie-break, ...) planted in a copy of the
  oracle on the CPU must make one of the checks above fail.
"""
import math

import numpy as np
import pytest

import oracle.moe_lora_oracle as O
import workloads as W


# --------------------------------------------------------------------------
# bf16 rounding
# --------------------------------------------------------------------------

def test_bf16_round_hand_values():
    cases = {
        1.0: 0x3F80,
        -2.5: 0xC020,
        1.0 + 2.0 ** -8: 0x3F80,                  # tie -> even (0x3F80)
        1.0 + 3 * 2.0 ** -8: 0x3F82,              # tie -> even (0x3F82)
        1.0 + 2.0 ** -8 + 2.0 ** -40: 0x3F81,     # just above the tie
        3.3895313892515355e38: 0x7F7F,            # largest finite bf16
        3.4e38: 0x7F80,                           # rounds past the largest -> inf
        2.0 ** -126: 0x0080,                      # smallest normal
        2.0 ** -133: 0x0001,                      # smallest subnormal
        2.0 ** -134: 0x0000,                      # tie between 0 and 2^-133 -> even
        3 * 2.0 ** -135: 0x0001,                  # 0.75 ulp -> 1
        -0.0: 0x8000,
        float("inf"): 0x7F80,
    }
    for v, bits in cases.items():
        assert int(O.f64_to_bf16_bits(np.array([v]))[0]) == bits, (v, hex(bits))
    assert int(O.f64_to_bf16_bits(np.array([float("nan")]))[0]) & 0x7FFF > 0x7F80


def test_bf16_round_matches_torch_on_float32_values():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-30, 30, 4000),
                        rng.standard_normal(1000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = O.f64_to_bf16_bits(x.astype(np.float64))
    assert np.array_equal(ref, got)


def test_bf16_decode_exact():
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]      # finite only
    f = O.bf16_bits_to_f64(bits)
    back = O.f64_to_bf16_bits(f)
    assert np.array_equal(back, bits)


# --------------------------------------------------------------------------
# Hand-worked example (closed form derived on paper)
# --------------------------------------------------------------------------

def _bits(a):
    return W.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def test_hand_worked_example():
    """T=1, H=2, I=1, E=3, top_k=2, rank 1, adapter 0, scaling 2.

    logits (0.5, 1.5, -2.0) -> experts (1, 0); w1 = 1/(1+e^-1), w0 = e^-1/(1+e^-1).
    x = (1, 2).
    expert 1: gate = x0 = 1, up = x1 = 2; LoRA u = 0.5*x0 = 0.5, delta = 2*(1, 0)*0.5
              -> gate 2, up 2 -> h1 = silu(2)*2 = 4/(1+e^-2);
              y = (h1, 2 h1) + 2*(0, 1)*(1*h1) = (h1, 4 h1).
    expert 0: gate = 0.5*x1 = 1, up = x0 + x1 = 3; LoRA u = x0 - x1 = -1,
              delta = 2*(0, 0.25)*(-1) = (0, -0.5) -> gate 1, up 2.5
              -> h0 = silu(1)*2.5 = 2.5/(1+e^-1);  y = (-h0, 0.5 h0) (A_dn = 0).
    out = w1*y1 + w0*y0.
    """
    E, H, I = 3, 2, 1
    logits = np.array([[0.5, 1.5, -2.0]], dtype=np.float32)
    hidden = _bits([[1.0, 2.0]])
    w13 = _bits([[[0.0, 0.5], [1.0, 1.0]],      # expert 0: gate row, up row
                 [[1.0, 0.0], [0.0, 1.0]],      # expert 1
                 [[3.0, 3.0], [3.0, 3.0]]])     # expert 2 (not selected)
    w2 = _bits([[[-1.0], [0.5]], [[1.0], [2.0]], [[7.0], [7.0]]])
    A_gu = _bits([[[[1.0, -1.0]], [[0.5, 0.0]], [[9.0, 9.0]]]])        # [A=1, E, r=1, H]
    B_gu = _bits([[[[0.0], [0.25]], [[1.0], [0.0]], [[9.0], [9.0]]]])  # [1, E, 2I, r]
    A_dn = _bits([[[[0.0]], [[1.0]], [[9.0]]]])                        # [1, E, r, I]
    B_dn = _bits([[[[5.0], [5.0]], [[0.0], [1.0]], [[9.0], [9.0]]]])  # [1, E, H, r]
    gu = O.LoraFactors(A_gu, B_gu)
    dn = O.LoraFactors(A_dn, B_dn)
    res = O.moe_lora_forward(hidden, logits, w13, w2, np.array([0], np.int32), 2, 2.0, gu, dn)

    w1 = 1.0 / (1.0 + math.exp(-1.0))
    w0 = math.exp(-1.0) / (1.0 + math.exp(-1.0))
    h1 = 4.0 / (1.0 + math.exp(-2.0))
    h0 = 2.5 / (1.0 + math.exp(-1.0))
    expect = np.array([w1 * h1 - w0 * h0, 4.0 * w1 * h1 + 0.5 * w0 * h0])
    assert list(res["ids"][0]) == [1, 0]
    np.testing.assert_allclose(res["w"][0], [w1, w0], rtol=1e-15)
    np.testing.assert_allclose(res["out64"][0], expect, rtol=1e-14)


# --------------------------------------------------------------------------
# Routing
# --------------------------------------------------------------------------

def test_routing_against_library_sort_and_full_softmax():
    rng = np.random.default_rng(3)
    for T, E, k in [(16, 8, 2), (5, 128, 8), (3, 16, 16), (7, 33, 5)]:
        logits = rng.standard_normal((T, E)).astype(np.float32)
        ids, w = O.route_topk(logits, k)
        order = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")[:, :k]
        assert np.array_equal(ids, order)
        p = np.exp(logits.astype(np.float64))
        p /= p.sum(axis=1, keepdims=True)
        psel = np.take_along_axis(p, order, axis=1)
        np.testing.assert_allclose(w, psel / psel.sum(axis=1, keepdims=True), rtol=1e-13)
        np.testing.assert_allclose(w.sum(axis=1), 1.0, atol=1e-14)
        assert np.all(np.diff(w, axis=1) <= 0)


def test_routing_ties_go_to_lower_expert():
    logits = np.array([[1.0, 2.0, 2.0, 0.0, 2.0],
                       [0.0, 0.0, 0.0, 0.0, 0.0],
                       [-0.0, 0.0, -1.0, 0.0, -0.0]], dtype=np.float32)
    ids, w = O.route_topk(logits, 3)
    assert ids.tolist() == [[1, 2, 4], [0, 1, 2], [0, 1, 3]]
    np.testing.assert_allclose(w[1], [1 / 3] * 3, rtol=1e-15)


def test_k_equals_E_is_full_softmax():
    rng = np.random.default_rng(4)
    logits = rng.standard_normal((4, 6)).astype(np.float32)
    ids, w = O.route_topk(logits, 6)
    for t in range(4):
        p = np.exp(logits[t].astype(np.float64))
        p /= p.sum()
        np.testing.assert_allclose(w[t], p[ids[t]], rtol=1e-14)


# --------------------------------------------------------------------------
# Permutation
# --------------------------------------------------------------------------

def test_permute_against_stable_argsort():
    rng = np.random.default_rng(5)
    for T, k, E in [(8, 2, 8), (37, 8, 128), (64, 8, 4), (1, 1, 1)]:
        ids = np.stack([rng.permutation(max(E, k))[:k] % E for _ in range(T)]).astype(np.int32)
        off, e2p, p2e = O.permute(ids, E)
        flat = ids.ravel()
        ref_p2e = np.argsort(flat, kind="stable")
        assert np.array_equal(p2e, ref_p2e)
        assert np.array_equal(e2p[p2e], np.arange(flat.size))
        assert np.array_equal(off, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
        assert off[-1] == T * k and np.all(np.diff(off) >= 0)


def test_permute_drops_minus_one_slots():
    ids = np.array([[2, -1], [0, 2], [-1, 1]], dtype=np.int32)
    off, e2p, p2e = O.permute(ids, 3)
    assert off.tolist() == [0, 1, 2, 4]
    assert e2p.tolist() == [2, -1, 0, 3, -1, 1]
    assert p2e.tolist() == [2, 5, 0, 3, -1, -1]


# --------------------------------------------------------------------------
# Brute force with merged weights
# --------------------------------------------------------------------------

def brute_force(inp):
    """Every expert evaluated densely with merged weights; selection by argsort."""
    wl = inp.wl
    H, I, E, k, s = wl.H, wl.I, wl.E, wl.top_k, wl.scaling
    w13 = O.bf16_bits_to_f64(inp.w13)
    w2 = O.bf16_bits_to_f64(inp.w2)
    A_gu = O.bf16_bits_to_f64(inp.A_gu) if inp.A_gu is not None else None
    B_gu = O.bf16_bits_to_f64(inp.B_gu) if inp.B_gu is not None else None
    A_dn = O.bf16_bits_to_f64(inp.A_dn) if inp.A_dn is not None else None
    B_dn = O.bf16_bits_to_f64(inp.B_dn) if inp.B_dn is not None else None
    x = O.bf16_bits_to_f64(inp.hidden)
    out = np.zeros((wl.T, H))
    for t in range(wl.T):
        a = int(inp.mapping[t])
        y_all = np.zeros((E, H))
        for e in range(E):
            W13, W2 = w13[e].copy(), w2[e].copy()
            if a >= 0 and A_gu is not None:
                Agu = A_gu[a] if wl.shared_outer else A_gu[a, e]
                Bdn = B_dn[a] if wl.shared_outer else B_dn[a, e]
                W13 = W13 + s * (B_gu[a, e] @ Agu)
                W2 = W2 + s * (Bdn @ A_dn[a, e])
            gate, up = W13[:I] @ x[t], W13[I:] @ x[t]
            y_all[e] = W2 @ (gate * (1.0 / (1.0 + np.exp(-gate))) * up)
        l = inp.logits[t].astype(np.float64)
        sel = np.argsort(-l, kind="stable")[:k]
        p = np.exp(l - l.max())
        p = p / p.sum()
        wsel = p[sel] / p[sel].sum()
        out[t] = (wsel[:, None] * y_all[sel]).sum(axis=0)
    return out


BRUTE_CASES = [
    W.WORKLOADS["tiny_T8"],
    W.small_workload("odd_shapes", T=5, H=24, I=40, E=5, top_k=3, num_adapters=3, rank=8,
                     map_lo=-1, map_hi=2, seed=11),
    W.small_workload("shared_outer", T=6, H=32, I=16, E=4, top_k=2, num_adapters=2, rank=8,
                     map_lo=-1, map_hi=1, shared_outer=True, bias_sigma=2.0, seed=12),
    W.small_workload("one_expert", T=3, H=16, I=8, E=1, top_k=1, num_adapters=1, rank=8,
                     map_lo=0, map_hi=0, seed=13),
    W.small_workload("k_eq_E", T=4, H=16, I=24, E=3, top_k=3, num_adapters=2, rank=8,
                     map_lo=-1, map_hi=1, seed=14),
]


@pytest.mark.parametrize("wl", BRUTE_CASES, ids=lambda w: w.name)
def test_oracle_matches_brute_force(wl):
    inp = W.make_inputs(wl)
    res = O.forward_inputs(inp)
    ref = brute_force(inp)
    np.testing.assert_allclose(res["out64"], ref, rtol=1e-10, atol=1e-12 * np.abs(ref).max())
    ids, w = res["ids"], res["w"]
    np.testing.assert_allclose(w.sum(axis=1), 1.0, atol=1e-14)


def test_one_expert_is_a_swiglu_mlp_with_lora():
    """E = 1, k = 1: out = W2' (silu(W1' x) * (W3' x)) with merged LoRA weights."""
    wl = W.small_workload("mlp", T=4, H=32, I=16, E=1, top_k=1, num_adapters=1, rank=8,
                          map_lo=0, map_hi=0, seed=21)
    inp = W.make_inputs(wl)
    s = wl.scaling
    f = O.bf16_bits_to_f64
    w13, w2 = f(inp.w13)[0], f(inp.w2)[0]
    merged13 = w13 + s * f(inp.B_gu)[0, 0] @ f(inp.A_gu)[0, 0]
    W1, W3 = merged13[:16], merged13[16:]
    W2m = w2 + s * f(inp.B_dn)[0, 0] @ f(inp.A_dn)[0, 0]
    X = f(inp.hidden)
    G = X @ W1.T
    ref = ((G / (1 + np.exp(-G))) * (X @ W3.T)) @ W2m.T
    np.testing.assert_allclose(O.forward_inputs(inp)["out64"], ref, rtol=1e-11)


# --------------------------------------------------------------------------
# Invariants
# --------------------------------------------------------------------------

def test_no_adapter_rank0_and_zero_scaling_reproduce_plain_moe():
    wl = W.WORKLOADS["tiny_T8"]
    inp = W.make_inputs(wl)
    plain = O.forward_inputs(inp, with_lora=False)["out64"]
    # all tokens -1
    inp_none = W.make_inputs(wl)
    inp_none.mapping[:] = -1
    assert np.array_equal(O.forward_inputs(inp_none)["out64"], plain)
    # scaling 0
    import dataclasses
    inp0 = W.make_inputs(dataclasses.replace(wl, scaling=0.0))
    assert np.array_equal(O.forward_inputs(inp0)["out64"], plain)
    # rank 0 (no factors drawn): same routing and base weights only if drawn identically;
    # the draw order puts LoRA after the base weights, so base tensors are unchanged.
    inpr0 = W.make_inputs(dataclasses.replace(wl, rank=0))
    assert inpr0.A_gu is None
    assert np.array_equal(O.forward_inputs(inpr0)["out64"], plain)
    # tokens without an adapter in a mixed batch match the plain rows exactly
    mixed = O.forward_inputs(inp)["out64"]
    no_ad = inp.mapping < 0
    assert no_ad.any() and (~no_ad).any()
    assert np.array_equal(mixed[no_ad], plain[no_ad])
    assert not np.allclose(mixed[~no_ad], plain[~no_ad])


def test_token_permutation_equivariance():
    wl = W.WORKLOADS["tiny_T8"]
    inp = W.make_inputs(wl)
    base = O.forward_inputs(inp)["out64"]
    perm = np.random.default_rng(9).permutation(wl.T)
    inp.hidden = inp.hidden[perm]
    inp.logits = inp.logits[perm]
    inp.mapping = inp.mapping[perm]
    np.testing.assert_allclose(O.forward_inputs(inp)["out64"], base[perm], rtol=1e-13, atol=1e-15)


def test_token_subset_matches_full_run():
    wl = W.WORKLOADS["tiny_T8"]
    inp = W.make_inputs(wl)
    full = O.forward_inputs(inp)
    sub = O.forward_inputs(inp, tokens=[6, 1, 3])
    assert np.array_equal(sub["out64"], full["out64"][[6, 1, 3]])


# --------------------------------------------------------------------------
# Planted mistakes: each must be caught by the pins above.
# --------------------------------------------------------------------------

ORIGINAL_SLOT = O.expert_slot
ORIGINAL_ROUTE = O.route_topk


def _make_slot(**mut):
    """expert_slot with one slip planted (selected by keyword)."""
    def slot(x, w13_e, w2_e, gu, dn, a, e, s):
        I = w2_e.shape[1]
        fe = 0 if mut.get("factor_of_expert_0") else e
        fa = (a + 1) % gu.A.shape[0] if (mut.get("wrong_adapter") and a >= 0) else a
        g = w13_e @ x
        delta = np.zeros_like(g)
        if a >= 0 and gu is not None and not mut.get("drop_gu"):
            delta = (1.0 if mut.get("drop_scale") else s) * (gu.b(fa, fe) @ (gu.a(fa, fe) @ x))
        if mut.get("delta_after_act"):
            h = O.silu(g[:I]) * g[I:] + delta[:I]
        elif mut.get("gate_up_swapped"):
            g = g + delta
            h = O.silu(g[I:]) * g[:I]
        else:
            g = g + delta
            h = O.silu(g[:I]) * g[I:]
        y = w2_e @ h
        if a >= 0 and dn is not None and not mut.get("drop_dn"):
            y = y + s * (dn.b(fa, e) @ (dn.a(fa, e) @ h))
        return g, h, y
    return slot


def _route_ties_to_higher(logits, top_k):
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    ids = np.zeros((T, top_k), np.int32)
    w = np.zeros((T, top_k))
    for t in range(T):
        row = [float(v) for v in logits[t]]
        order = sorted(range(E), key=lambda e: (-row[e], -e))
        sel = order[:top_k]
        ex = [math.exp(row[e] - row[sel[0]]) for e in sel]
        ids[t], w[t] = sel, [v / sum(ex) for v in ex]
    return ids, w


def _route_no_renorm(logits, top_k):
    ids, _ = ORIGINAL_ROUTE(logits, top_k)
    l = np.asarray(logits, np.float64)
    p = np.exp(l - l.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    return ids, np.take_along_axis(p, ids.astype(np.int64), axis=1)


def _silu_sigmoid_only(z):
    return 1.0 / (1.0 + np.exp(-z))


MUTANTS = {
    "gate_up_swapped": ("expert_slot", _make_slot(gate_up_swapped=True)),
    "drop_gate_up_lora": ("expert_slot", _make_slot(drop_gu=True)),
    "drop_down_lora": ("expert_slot", _make_slot(drop_dn=True)),
    "drop_scaling": ("expert_slot", _make_slot(drop_scale=True)),
    "delta_after_activation": ("expert_slot", _make_slot(delta_after_act=True)),
    "wrong_adapter": ("expert_slot", _make_slot(wrong_adapter=True)),
    "factor_of_expert_0": ("expert_slot", _make_slot(factor_of_expert_0=True)),
    "ties_to_higher_id": ("route_topk", _route_ties_to_higher),
    "no_renormalisation": ("route_topk", _route_no_renorm),
    "silu_is_sigmoid": ("silu", _silu_sigmoid_only),
}


def _pins_pass():
    """Runs the value-level pins; returns False as soon as one fails."""
    try:
        test_hand_worked_example()
        test_routing_ties_go_to_lower_expert()
        for wl in BRUTE_CASES:
            test_oracle_matches_brute_force(wl)
        test_one_expert_is_a_swiglu_mlp_with_lora()
    except AssertionError:
        return False
    return True


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(O, attr, fn)
    assert not _pins_pass(), f"planted mistake {name!r} went unnoticed"


def test_unmodified_oracle_passes_pins():
    assert _pins_pass()


def test_unplanted_slot_copy_passes_pins(monkeypatch):
    """The mutant scaffold itself, with nothing planted, must pass."""
    monkeypatch.setattr(O, "expert_slot", _make_slot())
    assert _pins_pass()
