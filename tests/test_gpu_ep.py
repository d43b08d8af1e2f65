"""Expert-parallel shards through the C ABI (needs a GB300).

Each shard is a layer holding a contiguous slice of the experts with
local_expert_offset / num_router_experts set; the shards run one after the
other on one GPU.  Per shard: routing (global ids) bit-exact, the partial
output against the oracle's shard forward.  Over the shards: the partial
outputs summed in float32 against the unsharded oracle (the all-reduce a
multi-GPU run does; its host side is tested with gloo ranks on the CPU).
"""
import numpy as np
import pytest

import oracle
import workloads
from gpu_util import (assert_output_close, cached_inputs, check_routing, make_layer, run_gpu,
                      to_f64)
from moe_lora_expert_gb300 import ep

pytestmark = pytest.mark.gpu

FULL_SAMPLE = {"prefill_T4096": list(range(0, 4096, 97)) + [4095]}


@pytest.mark.parametrize("name,world", [("tiny_T8", 3), ("decode_T16", 2), ("decode_T16", 3),
                                        ("skewed_T256_shared_outer_r64", 2), ("prefill_T4096", 2)])
def test_expert_shards_sum_to_the_layer(name, world):
    inp = cached_inputs(name)
    E = inp.wl.E
    tokens = FULL_SAMPLE.get(name)
    total = None
    for rank in range(world):
        off, cnt = ep.expert_shard(E, world, rank)
        part = workloads.shard_experts(inp, off, cnt)
        layer = make_layer(part, local_expert_offset=off, num_router_experts=E)
        res = run_gpu(part, layer=layer)
        assert res["status"] == 0, res["status_str"]
        check_routing(res, inp, shard=(off, cnt))   # global ids, shard-local permutation
        y = res["out64"] if tokens is None else res["out64"][tokens]
        ref = oracle.forward_inputs(part, tokens=tokens, local_expert_offset=off)["out64"]
        assert_output_close(y, ref, f"{name} shard {rank}/{world}")
        total = y if total is None else total + y
    full = oracle.forward_inputs(inp, tokens=tokens)["out64"]
    assert_output_close(total, full, f"{name} sum over {world} shards")


def test_shard_without_routed_slots_writes_zeros():
    inp = cached_inputs("decode_T16")
    logits = inp.logits.copy()
    logits[:, 96:] = -1e9               # experts 96..127 are never selected
    inp2 = workloads.LayerInputs(inp.wl, logits, inp.hidden, inp.w13, inp.w2, inp.A_gu, inp.B_gu,
                                 inp.A_dn, inp.B_dn, inp.mapping)
    part = workloads.shard_experts(inp2, 96, 32)
    layer = make_layer(part, local_expert_offset=96, num_router_experts=inp.wl.E)
    res = run_gpu(part, layer=layer)
    assert res["status"] == 0, res["status_str"]
    assert np.count_nonzero(to_f64(res["out"])) == 0
    assert np.all(res["e2p"] == -1)
