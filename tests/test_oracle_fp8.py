"""Pins for the FP8 block-scaled weight path of the oracle.

Reading (the pages name the FP8 block-quant path, trtllm_fp8_block_scale_
routed_moe_lora, without its format): float8 e4m3 weights, finite-only
variant, one float32 scale per 128 x 128 block of (rows, K); activations
bf16.  Pins: the e4m3 decoding against torch's float8_e4m3fn (a library
routine) and hand values; the block-scale indexing on a worked example; the
quantize/dequantize error bound of 3 mantissa bits; and, with power-of-two
scales (dequantized weights exact in bf16), the FP8 forward equals the bf16
forward, which is pinned on its own.
"""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")


def test_e4m3_decoding_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.array_equal(ours[~both_nan], ref[~both_nan])


def test_e4m3_hand_values():
    v = oracle.e4m3_to_f64(np.array([0x7E, 0xFE, 0x38, 0x08, 0x07, 0x01, 0x00, 0x80, 0x7F],
                                    dtype=np.uint8))
    assert list(v[:8]) == [448.0, -448.0, 1.0, 2.0 ** -6, 7 / 8 * 2.0 ** -6, 2.0 ** -9, 0.0, -0.0]
    assert np.isnan(v[8])


def test_block_scales_are_indexed_by_row_block_then_k_block():
    # one expert, 256 x 384 weights: 2 row blocks x 3 K blocks, all codes 1.0
    q = np.full((1, 256, 384), 0x38, dtype=np.uint8)
    scale = np.array([[[1.0, 2.0, 4.0], [8.0, 16.0, 32.0]]], dtype=np.float32)
    w = oracle.dequant_fp8_blocks(q, scale)
    assert w[0, 0, 0] == 1.0 and w[0, 127, 127] == 1.0
    assert w[0, 0, 128] == 2.0 and w[0, 5, 300] == 4.0
    assert w[0, 128, 0] == 8.0 and w[0, 200, 200] == 16.0 and w[0, 255, 383] == 32.0


def test_planted_transposed_scale_is_caught():
    """Indexing the scale grid (K block, row block) instead of (row block, K
    block) — planted here as a transposed square grid — changes the weights."""
    q = np.full((1, 256, 256), 0x38, dtype=np.uint8)
    scale = np.array([[[1.0, 2.0], [8.0, 16.0]]], dtype=np.float32)
    good = oracle.dequant_fp8_blocks(q, scale)
    bad = oracle.dequant_fp8_blocks(q, scale.transpose(0, 2, 1).copy())
    assert good[0, 0, 128] == 2.0 and bad[0, 0, 128] == 8.0


def test_quantize_dequantize_error_bound():
    wl = workloads.small_workload("fp8", T=4, H=300, I=136, E=2, top_k=1, num_adapters=0, rank=0,
                                  seed=3)
    inp = workloads.make_inputs(wl)
    q13, s13, q2, s2 = workloads.fp8_weights(inp)
    for bits, q, s in [(inp.w13, q13, s13), (inp.w2, q2, s2)]:
        w = oracle.bf16_bits_to_f64(bits)
        back = oracle.dequant_fp8_blocks(q, s)
        scale_full = np.repeat(np.repeat(s.astype(np.float64), 128, 1), 128, 2)[:, :w.shape[1], :w.shape[2]]
        # round to nearest with 3 mantissa bits: |err| <= 2^-4 |w| for normal
        # values, <= 2^-10 * scale in the subnormal range; the quantizer rounds
        # the float32 quotient w / scale, hence the 1e-6 relative slack
        bound = np.maximum(2.0 ** -4 * np.abs(w), 2.0 ** -10 * scale_full) * (1 + 1e-6)
        assert np.all(np.abs(back - w) <= bound)
        # the block maximum is 448 * scale: exact
        assert np.max(np.abs(back)) == pytest.approx(np.max(np.abs(w)), rel=1e-7)


def test_fp8_forward_equals_bf16_forward_when_weights_are_exact_in_bf16():
    wl = workloads.small_workload("fp8eq", T=9, H=256, I=136, E=3, top_k=2, num_adapters=2, rank=8,
                                  map_lo=-1, map_hi=1, seed=4)
    inp = workloads.make_inputs(wl)
    rng = np.random.default_rng(11)
    fin = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)

    def draw(shape):
        q = rng.choice(fin, size=shape).astype(np.uint8)
        nb, kb = -(-shape[1] // 128), -(-shape[2] // 128)
        s = (2.0 ** rng.integers(-12, -6, size=(shape[0], nb, kb))).astype(np.float32)
        return q, s

    q13, s13 = draw(inp.w13.shape)
    q2, s2 = draw(inp.w2.shape)
    w13 = oracle.f64_weights_to_bf16_bits_exact(oracle.dequant_fp8_blocks(q13, s13))
    w2 = oracle.f64_weights_to_bf16_bits_exact(oracle.dequant_fp8_blocks(q2, s2))
    gu, dn = oracle.factors_from_inputs(inp)
    ref = oracle.moe_lora_forward(inp.hidden, inp.logits, w13, w2, inp.mapping, wl.top_k,
                                  wl.scaling, gu, dn)["out64"]
    got = oracle.forward_inputs_fp8(inp, (q13, s13, q2, s2))["out64"]
    assert np.array_equal(got, ref)
