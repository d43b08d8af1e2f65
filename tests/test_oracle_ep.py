"""Expert-parallel sharding: the oracle's shard forward against the unsharded one.

Pins (the local_expert_offset / local_num_experts arguments of
trtllm_bf16_routed_moe_lora, sglang PR #28953 summary page; the layer output
is completed by a downstream all-reduce, Flow 1(A) of "[WIP][LoRA] BF16
support for the experimental_sgl_trtllm MoE-LoRA path & lora
expert_outer_shared"):
  * linearity: the shards' partial outputs over any partition of the experts
    sum to the unsharded output (the unsharded oracle is pinned on its own in
    test_oracle_pins.py);
  * a shard holding every expert is the unsharded forward, bit for bit;
  * a shard no slot is routed to contributes exactly zero;
  * a planted mistake (shard weights indexed without the offset) breaks the sum.
"""
import numpy as np
import pytest

import oracle
import workloads
from moe_lora_expert_gb300 import ep


def _inputs(shared_outer=False, seed=5):
    wl = workloads.small_workload("ep", T=12, H=48, I=24, E=8, top_k=3, num_adapters=2, rank=8,
                                  map_lo=-1, map_hi=1, shared_outer=shared_outer, seed=seed)
    return workloads.make_inputs(wl)


def _sharded_sum(inp, world, offset_fn=None):
    total = None
    for rank in range(world):
        off, cnt = ep.expert_shard(inp.wl.E, world, rank)
        part = workloads.shard_experts(inp, off, cnt)
        used_off = off if offset_fn is None else offset_fn(off)
        y = oracle.forward_inputs(part, local_expert_offset=used_off)["out64"]
        total = y if total is None else total + y
    return total


@pytest.mark.parametrize("shared_outer", [False, True])
@pytest.mark.parametrize("world", [2, 3, 8])
def test_partials_over_a_partition_sum_to_the_layer(world, shared_outer):
    inp = _inputs(shared_outer)
    full = oracle.forward_inputs(inp)["out64"]
    got = _sharded_sum(inp, world)
    scale = np.abs(full).max()
    assert np.abs(got - full).max() <= 1e-12 * scale


def test_shard_with_every_expert_is_the_unsharded_forward():
    inp = _inputs()
    full = oracle.forward_inputs(inp)
    part = oracle.forward_inputs(workloads.shard_experts(inp, 0, inp.wl.E), local_expert_offset=0)
    assert np.array_equal(full["out64"], part["out64"])
    assert np.array_equal(full["ids"], part["ids"])


def test_shard_without_routed_slots_contributes_zero():
    inp = _inputs()
    logits = inp.logits.copy()
    logits[:, 6:] = -1e9          # experts 6 and 7 are never among the top 3
    inp.logits = logits
    part = workloads.shard_experts(inp, 6, 2)
    y = oracle.forward_inputs(part, local_expert_offset=6)["out64"]
    assert np.count_nonzero(y) == 0
    # routing stays global: the ids are the unsharded ones
    assert np.array_equal(oracle.forward_inputs(part, local_expert_offset=6)["ids"],
                          oracle.route_topk(logits, inp.wl.top_k)[0])


def test_planted_offset_mistake_breaks_the_sum():
    inp = _inputs()
    full = oracle.forward_inputs(inp)["out64"]
    # every shard told it starts at expert 0: slots of experts 0..cnt-1 are
    # evaluated with the shard's own (wrong) weights, the rest dropped
    wrong = _sharded_sum(inp, 2, offset_fn=lambda off: 0)
    assert np.abs(wrong - full).max() > 1e-3 * np.abs(full).max()


@pytest.mark.parametrize("E,world", [(128, 1), (128, 2), (128, 3), (128, 4), (10, 4), (7, 7)])
def test_expert_shard_partition(E, world):
    seen = []
    sizes = []
    prev_end = 0
    for rank in range(world):
        off, cnt = ep.expert_shard(E, world, rank)
        assert off == prev_end and cnt >= 1          # contiguous, in rank order
        prev_end = off + cnt
        seen.extend(range(off, off + cnt))
        sizes.append(cnt)
    assert seen == list(range(E))
    assert max(sizes) - min(sizes) <= 1


def test_expert_shard_rejects_empty_ranks():
    with pytest.raises(ValueError):
        ep.expert_shard(3, 4, 0)
    with pytest.raises(ValueError):
        ep.expert_shard(8, 2, 2)
