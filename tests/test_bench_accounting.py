"""Host-side accounting in bench.py (no GPU): the default token-tile width,
the kernels one forward launches, and the algorithmic bytes charged to the
expert GEMMs.  These mirror choices the library makes in api.cu; the values
below are worked out by hand from the rules stated there."""
import pytest

import bench
import oracle
import workloads


@pytest.mark.parametrize("n_rows,E,bn", [
    (128, 128, 16),     # decode_T16: one row per expert
    (512, 128, 16),     # decode_T64: four rows per expert (4 * 4 = 16 stays)
    (1024, 128, 32),    # eight rows: 2 * 8 = 16, 4 * 8 = 32
    (2048, 128, 64),    # sixteen rows: 2 * 16 = 32, raised to 64 by 4 * 16
    (32768, 128, 256),  # prefill: 256 rows per expert
    (5, 8, 16),         # fewer rows than experts: avg over touched experts = 1
])
def test_auto_tile_n(n_rows, E, bn):
    assert bench.auto_tile_n(n_rows, E) == bn


def test_kernel_counts_per_forward():
    W = workloads.WORKLOADS
    # decode: permute (routing fused) + row gather + two GEMMs (shrinks inside) + finalize
    assert bench.kernels_per_forward(W["decode_T16"]) == 5
    assert bench.kernels_per_forward(W["decode_T64_mixed8"]) == 5
    assert bench.kernels_per_forward(W["decode_T16"], fp8=True) == 5
    # the row gather inside the gate_up GEMM as well
    assert bench.kernels_per_forward(W["decode_T16"], gather_in_gemm=True) == 4
    # W8A8: permute, row quant (the gather), GEMM, activation quant, GEMM, finalize
    assert bench.kernels_per_forward(W["decode_T16"], fp8=True, w8a8=True) == 6
    # shared-outer rank 64: routing, permute, gather+shrink, GEMM, shrink, GEMM, finalize
    assert bench.kernels_per_forward(W["skewed_T256_shared_outer_r64"]) == 7
    # prefill: routing, count, scan+scatter, row shrink, GEMM, row shrink, GEMM, finalize
    assert bench.kernels_per_forward(W["prefill_T4096"]) == 8
    # more experts than the two-kernel permute takes: routing + count, scan, scatter
    big_e = workloads.small_workload("e512", T=4096, H=256, I=128, E=512, top_k=8, num_adapters=1, rank=16)
    assert bench.kernels_per_forward(big_e) == 9


def test_shrink_in_gemm_conditions():
    W = workloads.WORKLOADS
    assert bench.shrink_in_gemm(W["decode_T16"])
    assert not bench.shrink_in_gemm(W["skewed_T256_shared_outer_r64"])   # shared gate_up A, rank 64
    assert not bench.shrink_in_gemm(W["prefill_T4096"])                  # 256-wide tiles
    big_rank = workloads.small_workload("r64", T=16, H=256, I=128, E=128, top_k=8, num_adapters=2,
                                        rank=64)
    assert not bench.shrink_in_gemm(big_rank)
    no_lora = workloads.small_workload("plain", T=16, H=256, I=128, E=128, top_k=8, num_adapters=0,
                                       rank=0)
    assert not bench.shrink_in_gemm(no_lora)


def test_gemm_bytes_charge_the_in_gemm_shrink():
    """Each expert GEMM is charged the weights and LoRA factors it reads and
    none of the intermediates (permuted rows, LoRA operands, activation,
    expert outputs).  With the shrinks inside the GEMMs, the gate_up kernel
    is also charged the A factors it reads, and the hidden input where it
    reads that itself (W8A8, or the row gather inside it); the down kernel
    the down A factors.  The sums are rebuilt here term by term from the
    routing of the seeded inputs."""
    wl = workloads.WORKLOADS["decode_T16"]
    inp = workloads.make_inputs(wl)
    ids, _ = oracle.route_topk(inp.logits, wl.top_k)
    work = bench.algorithmic_work(wl, ids, inp.mapping)
    own = bench.algorithmic_work(wl, ids, inp.mapping, gemm_reads_hidden=True)
    T, H, I, E, k, r = wl.T, wl.H, wl.I, wl.E, wl.top_k, wl.rank
    n = T * k
    experts = len(set(int(e) for e in ids.ravel()))
    adapted = [(t, int(inp.mapping[t])) for t in range(T) if inp.mapping[t] >= 0]
    pairs = len({(a, int(e)) for t, a in adapted for e in ids[t]})
    n_ad = len(adapted) * k
    gu = experts * 2 * I * H * 2 + pairs * 2 * I * r * 2
    gu += pairs * r * H * 2
    dn = experts * H * I * 2 + pairs * H * r * 2
    dn += pairs * r * I * 2
    assert work["gemm_gate_up"]["bytes"] == gu
    assert own["gemm_gate_up"]["bytes"] == gu + T * H * 2
    assert own["bytes"] == work["bytes"] and own["gemm_down"] == work["gemm_down"]
    assert work["gemm_down"]["bytes"] == dn
    assert work["gemm_gate_up"]["flops"] == n * 2 * 2 * I * H + n_ad * 2 * 2 * I * r + n_ad * 2 * r * H
    assert work["gemm_down"]["flops"] == n * 2 * H * I + n_ad * 2 * H * r + n_ad * 2 * r * I


def test_gemm_bytes_without_the_in_gemm_shrink():
    """Separate shrink kernels (prefill, or the in-GEMM shrink turned off):
    the GEMMs are charged only their weights and B factors; the forward's
    bytes are the same either way."""
    wl = workloads.WORKLOADS["decode_T16"]
    inp = workloads.make_inputs(wl)
    ids, _ = oracle.route_topk(inp.logits, wl.top_k)
    fused = bench.algorithmic_work(wl, ids, inp.mapping)
    sep = bench.algorithmic_work(wl, ids, inp.mapping, in_gemm_allowed=False)
    H, I, r = wl.H, wl.I, wl.rank
    experts = len(set(int(e) for e in ids.ravel()))
    pairs = fused["lora_pairs"]
    assert sep["gemm_gate_up"]["bytes"] == experts * 2 * I * H * 2 + pairs * 2 * I * r * 2
    assert sep["gemm_down"]["bytes"] == experts * H * I * 2 + pairs * H * r * 2
    assert sep["bytes"] == fused["bytes"] and sep["flops"] == fused["flops"]


def test_kernel_counts_of_the_other_schedules():
    W = workloads.WORKLOADS
    # separate shrinks: permute, gather+shrink, GEMM, shrink, GEMM, finalize
    assert bench.kernels_per_forward(W["decode_T16"], in_gemm_allowed=False) == 6
    # two streams: the gather and the gate_up shrink are two kernels
    assert bench.kernels_per_forward(W["decode_T16"], two_streams=True) == 7
    assert bench.kernels_per_forward(W["prefill_T4096"], two_streams=True) == 9
