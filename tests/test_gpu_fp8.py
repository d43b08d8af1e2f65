"""FP8 block-scaled expert weights through the C ABI (needs a GB300).

The weights are the bf16 ones block-quantized (e4m3, one float32 scale per
128 x 128 block); the oracle dequantizes them in float64.  The kernels
dequantize to bf16 before the tensor cores (2^-9 relative per weight), well
inside the output tolerance.
"""
import numpy as np
import pytest

import oracle
import workloads
from gpu_util import assert_output_close, bf16_tensor, check_routing, dev, run_gpu, torch_mod

pytestmark = pytest.mark.gpu


def fp8_layer(inp, fp8, with_lora=True):
    import moe_lora_expert_gb300 as m
    torch = torch_mod()
    q13, s13, q2, s2 = fp8
    wl = inp.wl
    args = dict(scaling=wl.scaling,
                w13_scale=torch.from_numpy(s13).to(dev()), w2_scale=torch.from_numpy(s2).to(dev()))
    lora = []
    if with_lora and inp.A_gu is not None:
        lora = [bf16_tensor(inp.A_gu), bf16_tensor(inp.B_gu), bf16_tensor(inp.A_dn), bf16_tensor(inp.B_dn)]
    return m.MoeLoraLayer(torch.from_numpy(q13).to(dev()), torch.from_numpy(q2).to(dev()), wl.top_k,
                          *lora, **args)


def _check(inp, fp8, tokens=None, tile_n=0, with_lora=True, label=""):
    layer = fp8_layer(inp, fp8, with_lora)
    res = run_gpu(inp, layer=layer, tile_n=tile_n, with_lora=with_lora)
    assert res["status"] == 0, res["status_str"]
    check_routing(res, inp)
    got = res["out64"] if tokens is None else res["out64"][tokens]
    ref = oracle.forward_inputs_fp8(inp, fp8, tokens=tokens, with_lora=with_lora)["out64"]
    return assert_output_close(got, ref, label)


@pytest.mark.parametrize("with_lora", [True, False])
@pytest.mark.parametrize("tile_n", [16, 32, 64, 128, 256])
def test_fp8_every_tile_width(tile_n, with_lora):
    """Every token-tile width of the FP8 GEMMs; H=192 and I=144 leave partial
    128-wide scale blocks and a partial 64-wide K block of the down GEMM."""
    wl = workloads.small_workload("fp8_tiles", T=96, H=192, I=144, E=6, top_k=3, num_adapters=3,
                                  rank=16, map_lo=-1, map_hi=2, seed=61)
    inp = workloads.make_inputs(wl)
    _check(inp, workloads.fp8_weights(inp), tile_n=tile_n, with_lora=with_lora,
           label=f"fp8 tile_n={tile_n} lora={with_lora}")


@pytest.mark.parametrize("name,tokens", [("decode_T16", None),
                                         ("prefill_T4096", list(range(0, 4096, 211)) + [4095])])
def test_fp8_workloads(name, tokens):
    inp = workloads.make_inputs(workloads.WORKLOADS[name])
    rel = _check(inp, workloads.fp8_weights(inp), tokens=tokens, label=f"fp8 {name}")
    print(f"fp8 {name}: relative Frobenius error {rel:.3e}")


def test_fp8_exact_weights_match_bf16_layer():
    """With power-of-two block scales the dequantized weights are exact in
    bf16: the FP8 layer and a bf16 layer holding those weights then run the
    same tensor-core arithmetic and agree bit for bit."""
    import moe_lora_expert_gb300 as m  # noqa: F401
    torch = torch_mod()
    wl = workloads.small_workload("fp8_exact", T=40, H=256, I=128, E=4, top_k=2, num_adapters=2,
                                  rank=8, map_lo=-1, map_hi=1, seed=62)
    inp = workloads.make_inputs(wl)
    rng = np.random.default_rng(5)
    fin = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)

    def draw(shape):
        q = rng.choice(fin, size=shape).astype(np.uint8)
        s = (2.0 ** rng.integers(-12, -6, size=(shape[0], -(-shape[1] // 128), -(-shape[2] // 128))))
        return q, s.astype(np.float32)

    q13, s13 = draw(inp.w13.shape)
    q2, s2 = draw(inp.w2.shape)
    out8 = run_gpu(inp, layer=fp8_layer(inp, (q13, s13, q2, s2)))["out"]
    inp16 = workloads.LayerInputs(inp.wl, inp.logits, inp.hidden,
                                  oracle.f64_weights_to_bf16_bits_exact(oracle.dequant_fp8_blocks(q13, s13)),
                                  oracle.f64_weights_to_bf16_bits_exact(oracle.dequant_fp8_blocks(q2, s2)),
                                  inp.A_gu, inp.B_gu, inp.A_dn, inp.B_dn, inp.mapping)
    out16 = run_gpu(inp16)["out"]
    assert torch.equal(out8.view(torch.int16), out16.view(torch.int16))
