"""Pins for the FP8-activation half of the FP8 path (oracle/fp8_activations.py).

Reading R12 (the pages name a per_token_group_quant_fp8 step on the hidden
input and a post-activation quant, Flow 1(A) of "[WIP][LoRA] BF16 support for
the experimental_sgl_trtllm MoE-LoRA path & lora expert_outer_shared", without
their arithmetic): per row and 128-column group, scale = max(amax, 1e-10) /
448 and code = e4m3(x / scale), both in float32.

Pins:
  * the encoder against torch's float8_e4m3fn conversion (a library routine),
    on exact values, every tie between neighbours and random values;
  * closed-form properties of the group quantizer: the group maximum encodes
    to +-448, the 3-bit rounding bound, the all-zero group, exact
    power-of-two scaling;
  * a planted mistake (groups along the wrong axis) is caught;
  * the whole forward against a brute-force scalar evaluation of a tiny
    layer that quantizes through torch's conversion.
"""
import math

import numpy as np
import pytest

import oracle
import workloads
from oracle import fp8_activations as fa

torch = pytest.importorskip("torch")


def torch_codes(v32):
    t = torch.from_numpy(np.asarray(v32, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_encoder_matches_torch_on_exact_values_and_ties():
    vals = oracle.e4m3_to_f64(np.arange(0, 0x7F, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2          # every tie between neighbours (exact in float32)
    probe = np.concatenate([vals, mids, -vals, -mids, [0.0, -0.0]]).astype(np.float32)
    assert np.array_equal(fa.e4m3_encode(probe.astype(np.float64)), torch_codes(probe))


def test_encoder_matches_torch_on_random_values():
    rng = np.random.default_rng(7)
    v = np.concatenate([rng.uniform(-448, 448, 20000), rng.normal(0, 1e-2, 20000),
                        rng.normal(0, 1e-3, 5000)]).astype(np.float32)
    assert np.array_equal(fa.e4m3_encode(v.astype(np.float64)), torch_codes(v))


def test_encoder_saturates_above_448():
    assert fa.e4m3_encode(np.array([448.00003, 1e6, -500.0])).tolist() == [0x7E, 0x7E, 0xFE]


def _groups(rows, K, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return (rng.normal(0, scale, (rows, K))).astype(np.float32)


def test_group_maximum_encodes_to_448_and_error_bound():
    x = _groups(5, 300, 1)                     # groups of 128, 128, 44
    codes, scales = fa.quant_fp8_token_groups(x)
    assert scales.shape == (5, 3)
    deq = fa.dequant_token_groups(codes, scales)
    for g in range(3):
        blk = x[:, g * 128:(g + 1) * 128].astype(np.float64)
        i = np.argmax(np.abs(blk), axis=1)
        c = codes[np.arange(5), g * 128 + i]
        assert np.all((c & 0x7F) == 0x7E)
    s = np.repeat(scales.astype(np.float64), 128, axis=1)[:, :300]
    xa = x.astype(np.float64)
    # 3 mantissa bits: |err| <= 2^-4 |x| (normal) or 2^-10 * scale (subnormal);
    # the float32 quotient adds one rounding
    bound = np.maximum(2.0 ** -4 * np.abs(xa), 2.0 ** -10 * s) * (1 + 1e-6)
    assert np.all(np.abs(deq - xa) <= bound)


def test_all_zero_group_and_power_of_two_scaling():
    x = _groups(3, 256, 2)
    x[1, 128:] = 0.0
    codes, scales = fa.quant_fp8_token_groups(x)
    assert np.all(codes[1, 128:] == 0)
    assert scales[1, 1] == np.float32(1e-10) / np.float32(448.0)
    codes2, scales2 = fa.quant_fp8_token_groups(x * np.float32(2.0 ** -5))
    nz = scales > np.float32(1e-9)
    assert np.array_equal(codes2[:, :128], codes[:, :128])
    assert np.array_equal(scales2[nz], scales[nz] * np.float32(2.0 ** -5))


def test_planted_wrong_group_axis_is_caught():
    x = _groups(128, 128, 3) * np.linspace(0.1, 10, 128, dtype=np.float32)[:, None]
    c, s = fa.quant_fp8_token_groups(x)
    good = fa.dequant_token_groups(c, s)
    ct, st = fa.quant_fp8_token_groups(np.ascontiguousarray(x.T))   # groups along tokens
    bad = fa.dequant_token_groups(ct, st).T
    assert np.max(np.abs(good - bad)) > 1e-3 * np.max(np.abs(x))


# ----------------------------------------------------------- brute force
def _torch_quant_scalar(vals):
    """Reading R12 on one group, scalar float32 steps, torch's e4m3 conversion."""
    amax = np.float32(0.0)
    for v in vals:
        amax = max(amax, np.float32(abs(v)))
    s = np.float32(max(amax, np.float32(1e-10)) / np.float32(448.0))
    out = []
    for v in vals:
        q = min(max(np.float32(np.float32(v) / s), np.float32(-448.0)), np.float32(448.0))
        qt = torch.tensor([float(q)], dtype=torch.float32).to(torch.float8_e4m3fn).to(torch.float64)
        out.append(float(qt.item()) * float(s))
    return out


def _quant_vec(vec):
    res = []
    for g0 in range(0, len(vec), 128):
        res.extend(_torch_quant_scalar([np.float32(v) for v in vec[g0:g0 + 128]]))
    return res


def test_forward_against_brute_force_on_a_tiny_layer():
    wl = workloads.small_workload("w8a8", T=3, H=136, I=132, E=2, top_k=1, num_adapters=2, rank=8,
                                  map_lo=-1, map_hi=1, seed=17)
    inp = workloads.make_inputs(wl)
    q13, s13, q2, s2 = workloads.fp8_weights(inp)
    gu, dn = oracle.factors_from_inputs(inp)
    got = fa.moe_lora_forward_w8a8(inp.hidden, inp.logits, q13, s13, q2, s2, inp.mapping,
                                   wl.top_k, wl.scaling, gu, dn)["out64"]

    def deq(q, s, e, n, k):
        code = torch.tensor([int(q[e, n, k])], dtype=torch.uint8).view(torch.float8_e4m3fn)
        return float(code.to(torch.float64).item()) * float(s[e, n // 128, k // 128])

    ids, w = oracle.route_topk(inp.logits, wl.top_k)
    H, I, r = wl.H, wl.I, wl.rank
    for t in range(wl.T):
        x = [float(v) for v in oracle.bf16_bits_to_f64(inp.hidden[t])]
        xq = _quant_vec(x)
        acc = [0.0] * H
        for j in range(wl.top_k):
            e, a = int(ids[t, j]), int(inp.mapping[t])
            g = [math.fsum(deq(q13, s13, e, n, k) * xq[k] for k in range(H)) for n in range(2 * I)]
            if a >= 0:
                A, B = gu.a(a, e), gu.b(a, e)
                u = [math.fsum(A[i, k] * x[k] for k in range(H)) for i in range(r)]
                g = [g[n] + wl.scaling * math.fsum(B[n, i] * u[i] for i in range(r)) for n in range(2 * I)]
            h = [g[n] / (1.0 + math.exp(-g[n])) * g[I + n] for n in range(I)]
            hq = _quant_vec(h)
            y = [math.fsum(deq(q2, s2, e, m, n) * hq[n] for n in range(I)) for m in range(H)]
            if a >= 0:
                A, B = dn.a(a, e), dn.b(a, e)
                v = [math.fsum(A[i, n] * h[n] for n in range(I)) for i in range(r)]
                y = [y[m] + wl.scaling * math.fsum(B[m, i] * v[i] for i in range(r)) for m in range(H)]
            acc = [acc[m] + float(w[t, j]) * y[m] for m in range(H)]
        ref = np.array(acc)
        assert np.abs(got[t] - ref).max() <= 1e-9 * max(np.abs(ref).max(), 1e-30), t
