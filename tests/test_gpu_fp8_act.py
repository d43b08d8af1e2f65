"""The FP8 path with FP8 activations (W8A8) through the C ABI (needs a GB300).

Reading R12 of the activation quant (per row and 128-column group, float32:
scale = max(amax, 1e-10) / 448, code = e4m3(x / scale)) is the oracle's
``oracle/fp8_activations.py``, pinned on the CPU by tests/test_oracle_fp8_act.py.

* ``moe_per_token_group_quant_fp8`` is compared with the oracle's quantizer
  bit for bit (codes and scales): both divide in float32 with IEEE rounding
  and round to e4m3 nearest-even, so the integer codes must agree exactly.
* The W8A8 forward is compared with ``moe_lora_forward_w8a8`` at the
  forward's output tolerance (per element |gpu - ref| <= 3e-2 + 2e-2 |ref|,
  relative Frobenius error <= 1e-2).  The kernels compute the activation in float32 with
  fast exp before its quant, so an activation code can differ from the
  float64 oracle's by one step where the value sits on a rounding boundary;
  one step is 2^-3 relative of that element, far inside the tolerance once
  summed over the down GEMM.
"""
import numpy as np
import pytest

import oracle
import workloads
from gpu_util import (assert_output_close, bf16_tensor, check_routing, dev, run_gpu, to_f64,
                      torch_mod)
from oracle import fp8_activations as fa

pytestmark = pytest.mark.gpu


def _bf16_rows(rng, shape, scale):
    return workloads.f32_to_bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


@pytest.mark.parametrize("K", [128, 144, 2048, 768])
def test_quant_groups_bit_exact_bf16_rows(K):
    """bf16 source rows through a row map (the permuted-row gather of the
    forward): partial last groups (K = 144), an all-zero row, a row of one
    large value, mixed scales, and negative map entries (zero rows)."""
    import moe_lora_expert_gb300 as m
    torch = torch_mod()
    rng = np.random.default_rng(K)
    T = 37
    x = _bf16_rows(rng, (T, K), 1.0)
    x[3] = 0
    x[5] = workloads.f32_to_bf16_bits(np.where(np.arange(K) == 7, 300.0, 1e-3).astype(np.float32))
    x[6] = _bf16_rows(rng, (1, K), 1e-6)[0]
    row_map = rng.integers(-1, T * 4, size=91).astype(np.int32)     # source row = row_map // 4
    codes, scales = m.moe_per_token_group_quant_fp8(bf16_tensor(x), torch.from_numpy(row_map).to(dev()),
                                                    map_div=4)
    src = oracle.bf16_bits_to_f64(x).astype(np.float32)
    rows = np.where(row_map[:, None] >= 0, src[np.maximum(row_map, 0) // 4], 0).astype(np.float32)
    ref_c, ref_s = fa.quant_fp8_token_groups(rows)
    assert np.array_equal(scales.cpu().numpy(), ref_s)
    assert np.array_equal(codes.cpu().numpy(), ref_c)


def test_quant_groups_bit_exact_f32_rows():
    """float32 source rows (the activation quant): values spread over many
    binades, exact ties between e4m3 neighbours after the scaling, and values
    that round past 448 before saturating."""
    import moe_lora_expert_gb300 as m
    torch = torch_mod()
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((64, 256)) * np.exp(rng.uniform(-8, 8, (64, 1)))).astype(np.float32)
    # row 0: group max 448 (scale 1), then every tie between e4m3 neighbours
    vals = oracle.e4m3_to_f64(np.arange(0, 0x7F, dtype=np.uint8))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    x[0, :] = 0
    x[0, 0] = 448.0
    x[0, 1:1 + 126] = mids[:126]
    x[0, 128] = 448.0
    x[0, 129:129 + 125] = -mids[:125]
    codes, scales = m.moe_per_token_group_quant_fp8(torch.from_numpy(x).to(dev()))
    ref_c, ref_s = fa.quant_fp8_token_groups(x)
    assert np.array_equal(scales.cpu().numpy(), ref_s)
    assert np.array_equal(codes.cpu().numpy(), ref_c)


def w8a8_layer(inp, fp8, with_lora=True):
    import moe_lora_expert_gb300 as m
    torch = torch_mod()
    q13, s13, q2, s2 = fp8
    wl = inp.wl
    lora = []
    if with_lora and inp.A_gu is not None:
        lora = [bf16_tensor(inp.A_gu), bf16_tensor(inp.B_gu), bf16_tensor(inp.A_dn), bf16_tensor(inp.B_dn)]
    return m.MoeLoraLayer(torch.from_numpy(q13).to(dev()), torch.from_numpy(q2).to(dev()), wl.top_k,
                          *lora, scaling=wl.scaling, w13_scale=torch.from_numpy(s13).to(dev()),
                          w2_scale=torch.from_numpy(s2).to(dev()), fp8_activations=True)


def w8a8_ref(inp, fp8, tokens=None, with_lora=True):
    gu, dn = oracle.factors_from_inputs(inp) if with_lora else (None, None)
    q13, s13, q2, s2 = fp8
    wl = inp.wl
    return fa.moe_lora_forward_w8a8(inp.hidden, inp.logits, q13, s13, q2, s2, inp.mapping, wl.top_k,
                                    wl.scaling, gu, dn, tokens=tokens)["out64"]


def _check(inp, fp8, tokens=None, tile_n=0, with_lora=True, label=""):
    res = run_gpu(inp, layer=w8a8_layer(inp, fp8, with_lora), tile_n=tile_n, with_lora=with_lora)
    assert res["status"] == 0, res["status_str"]
    check_routing(res, inp)
    got = res["out64"] if tokens is None else res["out64"][tokens]
    return assert_output_close(got, w8a8_ref(inp, fp8, tokens, with_lora), label)


@pytest.mark.parametrize("with_lora", [True, False])
@pytest.mark.parametrize("tile_n", [16, 32, 64, 128, 256])
def test_w8a8_every_tile_width(tile_n, with_lora):
    """Every token-tile width of the W8A8 GEMMs (256 runs as 128); H=192 and
    I=144 leave partial 128-wide scale blocks and activation groups and a
    partial last 128-K block in both GEMMs; rows of three adapters and
    unadapted rows share tiles."""
    wl = workloads.small_workload("w8a8_tiles", T=96, H=192, I=144, E=6, top_k=3, num_adapters=3,
                                  rank=16, map_lo=-1, map_hi=2, seed=61)
    inp = workloads.make_inputs(wl)
    _check(inp, workloads.fp8_weights(inp), tile_n=tile_n, with_lora=with_lora,
           label=f"w8a8 tile_n={tile_n} lora={with_lora}")


def test_w8a8_rank_and_shared_outer():
    """Rank 72 (two LoRA K blocks per adapter, the second partial) with
    shared-outer factors (the per-token gate_up shrink)."""
    wl = workloads.small_workload("w8a8_so", T=50, H=256, I=128, E=5, top_k=2, num_adapters=2,
                                  rank=72, map_lo=-1, map_hi=1, shared_outer=True, seed=63)
    inp = workloads.make_inputs(wl)
    _check(inp, workloads.fp8_weights(inp), label="w8a8 r72 shared-outer")


@pytest.mark.parametrize("name,tokens", [("decode_T16", None), ("decode_T64_mixed8", None),
                                         ("skewed_T256_shared_outer_r64", None),
                                         ("prefill_T4096", list(range(0, 4096, 211)) + [4095])])
def test_w8a8_workloads(name, tokens):
    inp = workloads.make_inputs(workloads.WORKLOADS[name])
    rel = _check(inp, workloads.fp8_weights(inp), tokens=tokens, label=f"w8a8 {name}")
    print(f"w8a8 {name}: relative Frobenius error {rel:.3e}")


def test_w8a8_no_adapter_tokens_match_plain_w8a8():
    """Mapping all -1: the LoRA K blocks are skipped for every tile, so the
    output equals the W8A8 layer built without LoRA bit for bit."""
    torch = torch_mod()
    inp = workloads.make_inputs(workloads.small_workload("w8a8_none", T=24, H=256, I=128, E=4, top_k=2,
                                                         num_adapters=2, rank=16, seed=64))
    fp8 = workloads.fp8_weights(inp)
    none = np.full(inp.wl.T, -1, dtype=np.int32)
    a = run_gpu(inp, layer=w8a8_layer(inp, fp8), mapping=none)["out"]
    b = run_gpu(inp, layer=w8a8_layer(inp, fp8, with_lora=False), with_lora=False)["out"]
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_w8a8_shrink_flag_wait_timeout_is_reported_and_recoverable():
    """The W8A8 GEMM holds a tile's LoRA operand loads until the in-kernel
    shrink has published the tile's rows.  With permuted row 0 never counted
    (test flag) that tile never completes: the held load's wait runs out,
    the forward reports MOE_ERR_DEVICE_TIMEOUT and the kernels drain and
    exit; the next call on the same workspace is correct."""
    import moe_lora_expert_gb300 as m
    torch = torch_mod()
    inp = workloads.make_inputs(workloads.WORKLOADS["decode_T16"])
    fp8 = workloads.fp8_weights(inp)
    layer = w8a8_layer(inp, fp8)
    hid = bf16_tensor(inp.hidden)
    lg = torch.from_numpy(inp.logits).to(dev())
    mp = torch.from_numpy(inp.mapping).to(dev())
    layer.forward(hid, lg, mp, wait_timeout_ms=20, debug_flags=m.MOE_DEBUG_HOLD_SHRINK_ROW)
    assert layer.device_status() == m.MOE_ERR_DEVICE_TIMEOUT
    out = layer.forward(hid, lg, mp)
    assert layer.device_status() == m.MOE_OK
    assert_output_close(to_f64(out), w8a8_ref(inp, fp8), "w8a8 after flag timeout")
