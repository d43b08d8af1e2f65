"""Pins for the oracle's general adapters (separate gate/up pairs, own rank and
scale per adapter) and for the packing of such adapters into the library's
fused layout.  CPU only."""
import numpy as np
import pytest

import oracle
import oracle.moe_lora_oracle as O
import workloads as W


def _fused_from_inputs(inp):
    wl = inp.wl
    ads = []
    for a in range(wl.num_adapters):
        ads.append({"scaling": wl.scaling, "gate_up": (inp.A_gu[a], inp.B_gu[a]),
                    "down": (inp.A_dn[a], inp.B_dn[a])})
    return ads


def test_general_form_equals_fused_oracle():
    wl = W.WORKLOADS["tiny_T8"]
    inp = W.make_inputs(wl)
    out_general, _ = oracle.moe_lora_forward_general(inp.hidden, inp.logits, inp.w13, inp.w2,
                                                     inp.mapping, wl.top_k, _fused_from_inputs(inp))
    np.testing.assert_allclose(out_general, oracle.forward_inputs(inp)["out64"], rtol=1e-13, atol=1e-15)


def brute_force_general(inp, adapters):
    """Dense evaluation of every expert with merged weights per projection."""
    wl = inp.wl
    f = O.bf16_bits_to_f64
    H, I, E, k = wl.H, wl.I, wl.E, wl.top_k
    w13, w2, X = f(inp.w13), f(inp.w2), f(inp.hidden)
    dec = [O.decode_adapter(a) for a in adapters]
    out = np.zeros((wl.T, H))
    for t in range(wl.T):
        a = int(inp.mapping[t])
        y_all = np.zeros((E, H))
        for e in range(E):
            Wg, Wu, Wd = w13[e][:I].copy(), w13[e][I:].copy(), w2[e].copy()
            if a >= 0:
                ad, s = dec[a], dec[a]["scaling"]
                if "gate_up" in ad:
                    merged = s * ad["gate_up"][1][e] @ ad["gate_up"][0][e]
                    Wg, Wu = Wg + merged[:I], Wu + merged[I:]
                else:
                    Wg = Wg + s * ad["gate"][1][e] @ ad["gate"][0][e]
                    Wu = Wu + s * ad["up"][1][e] @ ad["up"][0][e]
                Wd = Wd + s * ad["down"][1][e] @ ad["down"][0][e]
            gate, up = Wg @ X[t], Wu @ X[t]
            y_all[e] = Wd @ (gate / (1 + np.exp(-gate)) * up)
        l = inp.logits[t].astype(np.float64)
        sel = np.argsort(-l, kind="stable")[:k]
        p = np.exp(l - l.max())
        wsel = p[sel] / p[sel].sum()
        out[t] = (wsel[:, None] * y_all[sel]).sum(axis=0)
    return out


SPECS = [("separate", 8, 16.0), ("fused", 16, 32.0), ("separate", 4, 4.0)]


def _general_case(seed=71):
    wl = W.small_workload("peft", T=9, H=48, I=24, E=4, top_k=2, num_adapters=3, rank=8,
                          map_lo=-1, map_hi=2, seed=seed)
    inp = W.make_inputs(wl)
    return inp, W.make_peft_adapters(wl, SPECS, seed=seed + 1)


def test_general_form_matches_brute_force():
    inp, ads = _general_case()
    got, _ = oracle.moe_lora_forward_general(inp.hidden, inp.logits, inp.w13, inp.w2, inp.mapping,
                                             inp.wl.top_k, ads)
    ref = brute_force_general(inp, ads)
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12 * np.abs(ref).max())


def test_planted_gate_up_swap_is_caught(monkeypatch):
    inp, ads = _general_case()
    orig = O.expert_slot_general

    def swapped(x, w13_e, w2_e, adapter, expert):
        if adapter is not None and "gate" in adapter:
            adapter = dict(adapter, gate=adapter["up"], up=adapter["gate"])
        return orig(x, w13_e, w2_e, adapter, expert)

    monkeypatch.setattr(O, "expert_slot_general", swapped)
    got, _ = O.moe_lora_forward_general(inp.hidden, inp.logits, inp.w13, inp.w2, inp.mapping,
                                        inp.wl.top_k, ads)
    ref = brute_force_general(inp, ads)
    assert not np.allclose(got, ref, rtol=1e-6)


def test_packing_gives_the_same_deltas():
    """Packed block-diagonal, zero-padded factors reproduce each adapter's
    per-projection deltas (float64 on the CPU)."""
    torch = pytest.importorskip("torch")
    from moe_lora_expert_gb300 import adapters as pk
    inp, ads = _general_case()
    wl = inp.wl
    to_t = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)
    ads_t = []
    for ad in ads:
        d = {"scaling": ad["scaling"]}
        for key in ("gate_up", "gate", "up", "down"):
            if key in ad:
                d[key] = (to_t(ad[key][0]), to_t(ad[key][1]))
        ads_t.append(d)
    A_gu, B_gu, A_dn, B_dn, scales = pk.pack_adapters(ads_t, wl.E, wl.H, wl.I)
    assert A_gu.shape[2] % 8 == 0 and A_gu.shape[2] == pk.packed_rank(ads_t)
    rng = np.random.default_rng(3)
    x = rng.standard_normal(wl.H)
    hvec = rng.standard_normal(wl.I)
    for a, ad in enumerate(O.decode_adapter(ad) for ad in ads):
        for e in range(wl.E):
            Agu, Bgu = A_gu[a, e].double().numpy(), B_gu[a, e].double().numpy()
            Adn, Bdn = A_dn[a, e].double().numpy(), B_dn[a, e].double().numpy()
            packed = scales[a] * Bgu @ (Agu @ x)
            if "gate_up" in ad:
                direct = ad["scaling"] * ad["gate_up"][1][e] @ (ad["gate_up"][0][e] @ x)
            else:
                direct = ad["scaling"] * np.concatenate([ad["gate"][1][e] @ (ad["gate"][0][e] @ x),
                                                         ad["up"][1][e] @ (ad["up"][0][e] @ x)])
            np.testing.assert_allclose(packed, direct, rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(scales[a] * Bdn @ (Adn @ hvec),
                                       ad["scaling"] * ad["down"][1][e] @ (ad["down"][0][e] @ hvec),
                                       rtol=1e-12, atol=1e-14)
