"""The multi-GPU bench path on the CPU: two gloo ranks, each an independent
replica (no data-path collective), barrier plus max-over-ranks timing and
the whole-job throughput that bench.py reports for N > 1."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        # rank r "took" 10 + 5r ms per step for 4 steps of 16 tokens each
        per_rank_total = 4 * (10.0 + 5.0 * rank)
        value, slowest = bench.job_throughput(16, 4, world, per_rank_total, dist, "cpu")
        e2e = bench.max_over_ranks(3.0 * (rank + 1), dist, "cpu")
        dist.barrier()
        q.put((rank, value, slowest, e2e))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=10) for _ in range(world))
    slowest_ms = 4 * (10.0 + 5.0)
    for rank, value, slowest, e2e in res:
        assert slowest == pytest.approx(slowest_ms)
        assert value == pytest.approx(world * 16 * 4 / (slowest_ms / 1e3))
        assert e2e == pytest.approx(6.0)


def test_single_rank_needs_no_process_group():
    import bench
    value, slowest = bench.job_throughput(16, 10, 1, 20.0)
    assert slowest == 20.0 and value == pytest.approx(16 * 10 / 0.02)


def _ep_worker(rank, world, port, q):
    """One expert-parallel rank: its slice of the experts, the oracle's partial
    output for it, then the all-reduce that completes the layer."""
    import numpy as np

    import oracle
    import workloads
    from moe_lora_expert_gb300 import ep
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = workloads.small_workload("ep", T=10, H=40, I=16, E=7, top_k=3, num_adapters=2, rank=8,
                                      map_lo=-1, map_hi=1, seed=9)
        inp = workloads.make_inputs(wl)
        off, cnt = ep.expert_shard(wl.E, world, rank)
        part = oracle.forward_inputs(workloads.shard_experts(inp, off, cnt), local_expert_offset=off)
        y64 = torch.from_numpy(part["out64"].copy())
        ep.all_reduce_partial(y64)
        # the same through bf16 partials, summed in float32 and rounded once
        bits = part["out_bf16"].astype(np.int32) << 16
        y16 = torch.from_numpy(bits.view(np.float32)).to(torch.bfloat16)
        ep.all_reduce_partial(y16)
        q.put((rank, y64.numpy(), y16.float().numpy(), np.abs(part["out64"])))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_expert_parallel_ranks_all_reduce_to_the_layer(world):
    import numpy as np

    import oracle
    import workloads
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_ep_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted((q.get(timeout=10) for _ in range(world)), key=lambda r: r[0])
    wl = workloads.small_workload("ep", T=10, H=40, I=16, E=7, top_k=3, num_adapters=2, rank=8,
                                  map_lo=-1, map_hi=1, seed=9)
    full = oracle.forward_inputs(workloads.make_inputs(wl))["out64"]
    scale = np.abs(full).max()
    sum_abs_parts = sum(r[3] for r in res)
    for _, y64, y16, _ in res:
        assert np.abs(y64 - full).max() <= 1e-12 * scale
        # one bf16 rounding (unit roundoff 2^-8: 8 significant bits) of each
        # partial and one of the sum; partials may exceed the sum when shards cancel
        bound = 2.0 ** -8 * (sum_abs_parts + np.abs(full)) * 1.01 + 1e-30
        assert np.all(np.abs(y16 - full) <= bound)
