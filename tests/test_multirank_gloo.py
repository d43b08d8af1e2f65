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
