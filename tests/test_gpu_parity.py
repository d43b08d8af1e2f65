"""CUDA path against the CPU oracle, through the C ABI (needs a GB300).

Routing ids and the permutation are compared bit for bit; routing weights
within a float32 error bound; the bf16 layer output per element within
3e-2 + 2e-2*|ref| and in relative Frobenius norm within 1e-2.
"""
import dataclasses

import numpy as np
import pytest

import oracle
import workloads
from gpu_util import (assert_output_close, bf16_tensor, cached_inputs, check_routing, dev,
                      make_layer, run_gpu, to_f64, torch_mod, W_RTOL)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import moe_lora_expert_gb300 as m
    m.lib()
    yield


# ----------------------------------------------------------------- routing

@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (37, 128, 8), (300, 33, 5), (64, 1024, 32),
                                   (5, 16, 16), (4096, 128, 8), (3, 1, 1)])
def test_route_topk_matches_oracle(T, E, k):
    import moe_lora_expert_gb300 as m
    torch = torch_mod()
    logits = np.random.default_rng(T * 7 + E).standard_normal((T, E)).astype(np.float32)
    ids, w = m.moe_route_topk(torch.from_numpy(logits).to(dev()), k)
    ids_ref, w_ref = oracle.route_topk(logits, k)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=W_RTOL, atol=1e-9)


def test_route_topk_ties_and_signed_zero():
    import moe_lora_expert_gb300 as m
    torch = torch_mod()
    logits = np.array([[1.0, 2.0, 2.0, 0.0, 2.0] + [-5.0] * 35,
                       [0.0] * 40,
                       [-0.0, 0.0, -1.0, 0.0, -0.0] + [-7.0] * 35], dtype=np.float32)
    ids, w = m.moe_route_topk(torch.from_numpy(logits).to(dev()), 3)
    ids_ref, w_ref = oracle.route_topk(logits, 3)
    assert ids.cpu().numpy().tolist() == ids_ref.tolist() == [[1, 2, 4], [0, 1, 2], [0, 1, 3]]
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=W_RTOL)


# ----------------------------------------------------------------- permute

@pytest.mark.parametrize("T,k,E,H", [(1, 1, 1, 8), (8, 2, 8, 256), (300, 8, 128, 72),
                                     (4096, 8, 128, 2048), (1000, 3, 1024, 16), (129, 4, 4, 40)])
def test_permute_matches_oracle(T, k, E, H):
    import moe_lora_expert_gb300 as m
    torch = torch_mod()
    rng = np.random.default_rng(T + E)
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    hidden = workloads.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    off, e2p, p2e, xp, ws = m.moe_permute(torch.from_numpy(ids).to(dev()), E, bf16_tensor(hidden))
    assert m.moe_read_device_status(ws) == m.MOE_OK
    off_r, e2p_r, p2e_r = oracle.permute(ids, E)
    assert np.array_equal(off.cpu().numpy(), off_r)
    assert np.array_equal(e2p.cpu().numpy(), e2p_r)
    assert np.array_equal(p2e.cpu().numpy(), p2e_r)
    xp_bits = xp.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(xp_bits, hidden[p2e_r // k])


def test_permute_unrouted_and_invalid_ids():
    import moe_lora_expert_gb300 as m
    torch = torch_mod()
    ids = np.array([[2, -1], [0, 2], [-1, 1], [7, 1], [0, -5]], dtype=np.int32)
    off, e2p, p2e, _, ws = m.moe_permute(torch.from_numpy(ids).to(dev()), 3)
    assert m.moe_read_device_status(ws) == m.MOE_ERR_BAD_EXPERT_ID
    clean = np.where((ids >= 0) & (ids < 3), ids, -1)
    off_r, e2p_r, p2e_r = oracle.permute(clean, 3)
    assert np.array_equal(off.cpu().numpy(), off_r)
    assert np.array_equal(e2p.cpu().numpy(), e2p_r)
    assert np.array_equal(p2e.cpu().numpy(), p2e_r)


# ----------------------------------------------------------------- forward

FULL_SAMPLE = {"prefill_T4096": list(range(0, 4096, 64)) + [4095]}


@pytest.mark.parametrize("name", workloads.WORKLOAD_ORDER)
def test_forward_workload(name):
    inp = cached_inputs(name)
    res = run_gpu(inp)
    assert res["status"] == 0, res["status_str"]
    check_routing(res, inp)
    tokens = FULL_SAMPLE.get(name)
    ref = oracle.forward_inputs(inp, tokens=tokens)
    got = res["out64"] if tokens is None else res["out64"][tokens]
    rel = assert_output_close(got, ref["out64"], name)
    print(f"{name}: relative Frobenius error {rel:.3e}")


@pytest.mark.parametrize("tile_n", [16, 32, 64, 128, 256])
def test_forward_every_tile_width(tile_n):
    wl = workloads.small_workload("tiles", T=96, H=192, I=136, E=6, top_k=3, num_adapters=3,
                                  rank=16, map_lo=-1, map_hi=2, seed=31)
    inp = workloads.make_inputs(wl)
    res = run_gpu(inp, tile_n=tile_n)
    assert res["status"] == 0, res["status_str"]
    check_routing(res, inp)
    assert_output_close(res["out64"], oracle.forward_inputs(inp)["out64"], f"tile_n={tile_n}")


EDGE = [
    workloads.small_workload("one_token", T=1, H=64, I=64, E=4, top_k=2, rank=8, seed=41),
    workloads.small_workload("one_expert_k1", T=20, H=128, I=64, E=1, top_k=1, num_adapters=2,
                             rank=16, seed=42),
    workloads.small_workload("k_eq_E", T=17, H=64, I=32, E=4, top_k=4, num_adapters=2, rank=8,
                             seed=43),
    workloads.small_workload("ragged_dims", T=33, H=200, I=72, E=5, top_k=2, num_adapters=2,
                             rank=24, seed=44),
    workloads.small_workload("rank128", T=40, H=256, I=128, E=4, top_k=2, num_adapters=2,
                             rank=128, seed=45),
    workloads.small_workload("rank72", T=40, H=256, I=128, E=4, top_k=2, num_adapters=3,
                             rank=72, seed=46),
    workloads.small_workload("many_adapters", T=200, H=128, I=64, E=8, top_k=2, num_adapters=64,
                             rank=8, map_lo=-1, map_hi=63, seed=47),
    workloads.small_workload("shared_outer", T=64, H=256, I=128, E=8, top_k=4, num_adapters=3,
                             rank=32, shared_outer=True, bias_sigma=2.0, map_lo=-1, map_hi=2,
                             seed=48),
    workloads.small_workload("no_lora", T=50, H=128, I=96, E=6, top_k=2, num_adapters=0, rank=0,
                             seed=49),
    workloads.small_workload("hot_expert", T=700, H=128, I=64, E=16, top_k=2, num_adapters=2,
                             rank=16, bias_sigma=4.0, seed=50),
    workloads.small_workload("many_chunks", T=1500, H=64, I=64, E=32, top_k=2, num_adapters=2,
                             rank=8, seed=51),
    # the ABI's maximum expert count and top-k (one-CTA permute, 32-slot finalize)
    workloads.small_workload("max_experts_top32", T=40, H=64, I=64, E=1024, top_k=32,
                             num_adapters=2, rank=8, map_lo=-1, map_hi=1, seed=52),
]


def test_forward_max_experts_many_rows():
    """1024 experts and 24000 rows: the multi-kernel permute with its largest
    counter arrays and the 128-row-tile shrink over 1024 experts; the oracle
    checks every 11th token."""
    wl = workloads.small_workload("max_experts_rows", T=3000, H=64, I=64, E=1024, top_k=8,
                                  num_adapters=3, rank=16, map_lo=-1, map_hi=2, seed=53)
    inp = workloads.make_inputs(wl)
    res = run_gpu(inp)
    assert res["status"] == 0, res["status_str"]
    check_routing(res, inp)
    tokens = np.arange(0, wl.T, 11)
    assert_output_close(res["out64"][tokens], oracle.forward_inputs(inp, tokens=tokens)["out64"],
                        wl.name)


@pytest.mark.parametrize("wl", EDGE, ids=lambda w: w.name)
def test_forward_edge_cases(wl):
    inp = workloads.make_inputs(wl)
    res = run_gpu(inp)
    assert res["status"] == 0, res["status_str"]
    check_routing(res, inp)
    assert_output_close(res["out64"], oracle.forward_inputs(inp)["out64"], wl.name)


def test_intermediates_match_oracle():
    """Activation h and expert output y, row by row, on the tiny layer."""
    import moe_lora_expert_gb300 as m
    torch = torch_mod()
    inp = cached_inputs("tiny_T8")
    wl = inp.wl
    res = run_gpu(inp)
    ref = oracle.forward_inputs(inp, keep_intermediates=True)
    layer = res["layer"]
    plan = layer.plan(wl.T)
    ws = layer._ws
    n = wl.T * wl.top_k

    def view_bf16(off, cols):
        return ws[off:off + n * cols * 2].view(torch.bfloat16).reshape(n, cols).float().cpu().numpy()

    h = view_bf16(plan.act, wl.I)
    y = view_bf16(plan.expert_out, wl.H)
    for t in range(wl.T):
        for j in range(wl.top_k):
            p = res["e2p"][t * wl.top_k + j]
            g_r, h_r, y_r = ref["intermediates"][(t, j)]
            assert_output_close(h[p], h_r, f"h[{t},{j}]")
            assert_output_close(y[p], y_r, f"y[{t},{j}]")


def test_no_adapter_tokens_reproduce_plain_moe_bitwise():
    inp = workloads.make_inputs(workloads.WORKLOADS["tiny_T8"])
    plain = run_gpu(inp, with_lora=False)["out"]
    none = run_gpu(inp, mapping=np.full(inp.wl.T, -1, np.int32))["out"]
    torch = torch_mod()
    assert torch.equal(plain.view(torch.int16), none.view(torch.int16))
    mixed = run_gpu(inp)["out"].float()
    rows = np.where(inp.mapping < 0)[0]
    assert len(rows) > 0
    assert torch.equal(mixed[rows], plain.float()[rows])


def test_zero_scaling_reproduces_plain_moe():
    wl = dataclasses.replace(workloads.WORKLOADS["tiny_T8"], scaling=0.0)
    inp = workloads.make_inputs(wl)
    torch = torch_mod()
    a = run_gpu(inp)["out"].float()
    b = run_gpu(inp, with_lora=False)["out"].float()
    assert torch.equal(a, b)


def test_bad_mapping_is_flagged_and_dropped():
    import moe_lora_expert_gb300 as m
    inp = workloads.make_inputs(workloads.WORKLOADS["tiny_T8"])
    bad = inp.mapping.copy()
    bad[1], bad[5] = 7, -4
    res = run_gpu(inp, mapping=bad)
    assert res["status"] == m.MOE_ERR_BAD_MAPPING
    clean = bad.copy()
    clean[1] = clean[5] = -1
    inp.mapping = clean
    assert_output_close(res["out64"], oracle.forward_inputs(inp)["out64"], "bad mapping")


def test_empty_batch_is_a_noop():
    import moe_lora_expert_gb300 as m
    torch = torch_mod()
    inp = cached_inputs("tiny_T8")
    layer = make_layer(inp)
    hidden = torch.empty((0, inp.wl.H), dtype=torch.bfloat16, device=dev())
    logits = torch.empty((0, inp.wl.E), dtype=torch.float32, device=dev())
    mapping = torch.empty((0,), dtype=torch.int32, device=dev())
    out = layer.forward(hidden, logits, mapping)
    assert out.shape == (0, inp.wl.H)
    assert layer.device_status() == m.MOE_OK


def test_repeated_calls_are_deterministic():
    inp = cached_inputs("decode_T16")
    layer = make_layer(inp)
    torch = torch_mod()
    a = run_gpu(inp, layer=layer)["out"].clone()
    b = run_gpu(inp, layer=layer)["out"]
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("with_lora", [True, False])
@pytest.mark.parametrize("tile_n", [128, 256])
def test_forward_cta_pairs(tile_n, with_lora):
    """Wide token tiles on CTA pairs that share one M = 256 MMA (cta_group::2).
    I=136 gives an odd number of gate_up feature blocks (the last pair's second
    CTA has none); T=700 over 3 experts gives full and partial tiles, some
    with no valid row in the second CTA's half; without LoRA the down GEMM
    follows the gate_up GEMM directly."""
    cases = [
        workloads.small_workload("pair_odd", T=300, H=192, I=136, E=3, top_k=2, num_adapters=3,
                                 rank=16, map_lo=-1, map_hi=2, seed=61),
        workloads.small_workload("pair_tiles", T=700, H=256, I=192, E=3, top_k=2, num_adapters=2,
                                 rank=32, map_lo=-1, map_hi=1, seed=67),
        # tiles of a few rows (the second CTA's half is empty) and a single
        # feature block in both GEMMs (the second CTA has none)
        workloads.small_workload("pair_tiny", T=20, H=128, I=64, E=8, top_k=2, num_adapters=2,
                                 rank=8, map_lo=-1, map_hi=1, seed=71),
    ]
    for wl in cases:
        inp = workloads.make_inputs(wl)
        res = run_gpu(inp, tile_n=tile_n, with_lora=with_lora, tuning={"cta_pairs": 2})
        assert res["status"] == 0, res["status_str"]
        check_routing(res, inp)
        ref = oracle.forward_inputs(inp, with_lora=with_lora)["out64"]
        assert_output_close(res["out64"], ref, f"{wl.name} tile_n={tile_n} lora={with_lora}")


@pytest.mark.parametrize("with_lora", [True, False])
def test_forward_many_rows_row_block_shrink(with_lora):
    """T*k = 4000 rows (more than 16 per SM) takes the 128-row-tile shrink with
    its cp.async pipeline: H=200 and I=72 leave partial 64-column chunks in
    both shrinks, three adapters and unadapted rows share tiles, rank 24."""
    wl = workloads.small_workload("rows", T=1000, H=200, I=72, E=5, top_k=4, num_adapters=3,
                                  rank=24, map_lo=-1, map_hi=2, seed=81)
    inp = workloads.make_inputs(wl)
    res = run_gpu(inp, with_lora=with_lora)
    assert res["status"] == 0, res["status_str"]
    check_routing(res, inp)
    tokens = np.arange(0, wl.T, 7)
    ref = oracle.forward_inputs(inp, tokens=tokens, with_lora=with_lora)["out64"]
    assert_output_close(res["out64"][tokens], ref, f"rows lora={with_lora}")


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("name", ["decode_T16", "decode_T64_mixed8", "tiny_T8"])
def test_forward_shrink_in_gemm_and_separate(name, mode):
    """Decode-sized tiles compute the LoRA shrinks inside the expert GEMMs
    (tile flags between CTAs) after a row-gather kernel (tuning 0);
    tuning.shrink_in_gemm = 1 keeps the separate shrink kernels, 2 moves the
    row gather into the gate_up GEMM too.  Each against the oracle."""
    inp = cached_inputs(name)
    res = run_gpu(inp, tuning={"shrink_in_gemm": mode})
    assert res["status"] == 0, res["status_str"]
    check_routing(res, inp)
    assert_output_close(res["out64"], oracle.forward_inputs(inp)["out64"], f"{name} mode={mode}")


@pytest.mark.parametrize("name", ["decode_T16", "decode_T64_mixed8"])
def test_row_gather_kernel_or_inside_the_gemm_bit_identical(name):
    """The row gather as a kernel of its own or inside the gate_up GEMM
    moves the same rows; the shrinks and GEMMs then compute the same
    products in the same order, so the two outputs agree bit for bit."""
    torch = torch_mod()
    inp = cached_inputs(name)
    a = run_gpu(inp, tuning={"shrink_in_gemm": 0})
    b = run_gpu(inp, tuning={"shrink_in_gemm": 2})
    assert a["status"] == 0 and b["status"] == 0
    assert torch.equal(a["out"].view(torch.int16), b["out"].view(torch.int16))


def test_forward_shrink_in_gemm_full_tiles():
    """Sixteen rows per expert in 16-wide tiles (every tile full, so each
    CTA's in-kernel shrink walks 16 rows), four adapters and unadapted rows
    mixed in the tiles, rank 32 (the largest the in-kernel shrink takes)."""
    wl = workloads.small_workload("fulltiles", T=256, H=320, I=96, E=16, top_k=1, num_adapters=4,
                                  rank=32, map_lo=-1, map_hi=3, seed=91)
    inp = workloads.make_inputs(wl)
    res = run_gpu(inp, tile_n=16)
    assert res["status"] == 0, res["status_str"]
    check_routing(res, inp)
    assert_output_close(res["out64"], oracle.forward_inputs(inp)["out64"], "fulltiles")


@pytest.mark.parametrize("rank", [64, 128])
def test_forward_many_rows_large_rank(rank):
    """The 128-row-tile shrink with ranks above 32 (each thread then copies
    several factor rows per chunk) and shared-outer factors."""
    wl = workloads.small_workload("rows_rank", T=700, H=192, I=64, E=6, top_k=4, num_adapters=2,
                                  rank=rank, map_lo=-1, map_hi=1, shared_outer=(rank == 64),
                                  seed=90 + rank)
    inp = workloads.make_inputs(wl)
    res = run_gpu(inp)
    assert res["status"] == 0, res["status_str"]
    check_routing(res, inp)
    tokens = np.arange(0, wl.T, 5)
    ref = oracle.forward_inputs(inp, tokens=tokens)["out64"]
    assert_output_close(res["out64"][tokens], ref, f"rank {rank}")


def test_forward_replays_from_a_cuda_graph():
    """The forward enqueues only launches and memsets: captured into a CUDA graph
    and replayed it gives the eager result bit for bit, also after the inputs
    are overwritten in place between replays."""
    torch = torch_mod()
    for name in ["decode_T16", "skewed_T256_shared_outer_r64"]:
        inp = cached_inputs(name)
        layer = make_layer(inp)
        hid = bf16_tensor(inp.hidden)
        lg = torch.from_numpy(inp.logits).to(dev())
        mp = torch.from_numpy(inp.mapping).to(dev())
        eager = layer.forward(hid, lg, mp).clone()
        out = torch.empty_like(eager)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            layer.forward(hid, lg, mp, out=out)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16)), name
        lg.copy_(torch.flip(lg, dims=[0]))
        hid.copy_(torch.flip(hid, dims=[0]))
        graph.replay()
        eager2 = layer.forward(hid, lg, mp)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager2.view(torch.int16)), name
        assert layer.device_status() == 0


def test_device_wait_timeout_is_reported_and_recoverable():
    """A pipeline wait that can only run out (test flag: the gate_up GEMM's MMA
    role waits on a barrier nobody signals) ends with MOE_ERR_DEVICE_TIMEOUT
    in the status word; the kernel drains and frees its tensor memory, and the
    next call on the same workspace is correct again."""
    import moe_lora_expert_gb300 as m
    torch = torch_mod()
    inp = cached_inputs("tiny_T8")
    layer = make_layer(inp)
    hid = bf16_tensor(inp.hidden)
    lg = torch.from_numpy(inp.logits).to(dev())
    mp = torch.from_numpy(inp.mapping).to(dev())
    layer.forward(hid, lg, mp, wait_timeout_ms=20, debug_flags=m.MOE_DEBUG_STALL_GATE_UP_MMA)
    assert layer.device_status() == m.MOE_ERR_DEVICE_TIMEOUT
    out = layer.forward(hid, lg, mp)
    assert layer.device_status() == m.MOE_OK
    assert_output_close(to_f64(out), oracle.forward_inputs(inp)["out64"], "after timeout")


@pytest.mark.parametrize("T,A,rank", [(403, 3, 64), (1000, 2, 32)])
def test_forward_shared_outer_multi_phase(T, A, rank):
    """Shared gate_up A factor with more 16-token tiles than one wave of
    single-phase CTAs holds: the per-token shrink splits K (H = 2048) into
    three (T = 403, rank 64 in four slices, a ragged last tile) or two
    (T = 1000, rank 32 in two slices) equal phases so that the grid is
    resident at once; its factor product runs before the permute is known to
    be complete and its row gather is shared by every CTA of a tile."""
    wl = workloads.small_workload("so_phases", T=T, H=2048, I=64, E=8, top_k=2, num_adapters=A,
                                  rank=rank, map_lo=-1, map_hi=A - 1, shared_outer=True, seed=T + rank)
    inp = workloads.make_inputs(wl)
    res = run_gpu(inp)
    assert res["status"] == 0, res["status_str"]
    check_routing(res, inp)
    tokens = list(range(0, T, 7)) + [T - 1]
    ref = oracle.forward_inputs(inp, tokens=tokens)["out64"]
    assert_output_close(res["out64"][tokens], ref, f"shared-outer phases T={T} r={rank}")


@pytest.mark.parametrize("rank", [16, 48, 128])
def test_forward_shared_outer_rank_slices(rank):
    """Shared gate_up A factor (per-token shrink): ranks of 32 or more are
    split into 16-column slices over separate CTAs (3 and 8 slices here);
    rank 16 stays whole.  Partial K chunks (H=200) and unadapted tokens."""
    wl = workloads.small_workload("slices", T=40, H=200, I=72, E=6, top_k=3, num_adapters=3,
                                  rank=rank, map_lo=-1, map_hi=2, shared_outer=True, seed=95)
    inp = workloads.make_inputs(wl)
    res = run_gpu(inp)
    assert res["status"] == 0, res["status_str"]
    check_routing(res, inp)
    assert_output_close(res["out64"], oracle.forward_inputs(inp)["out64"], f"slices r={rank}")


def test_shrink_flag_wait_timeout_is_reported_and_recoverable():
    """The in-GEMM shrink's tile flags: with permuted row 0 never counted
    (test flag), the wait for its tile runs out and reports
    MOE_ERR_DEVICE_TIMEOUT; the kernels drain and exit, and the next call on
    the same workspace (the permute clears the flags) is correct."""
    import moe_lora_expert_gb300 as m
    torch = torch_mod()
    inp = cached_inputs("decode_T16")
    layer = make_layer(inp)
    hid = bf16_tensor(inp.hidden)
    lg = torch.from_numpy(inp.logits).to(dev())
    mp = torch.from_numpy(inp.mapping).to(dev())
    layer.forward(hid, lg, mp, wait_timeout_ms=20, debug_flags=m.MOE_DEBUG_HOLD_SHRINK_ROW)
    assert layer.device_status() == m.MOE_ERR_DEVICE_TIMEOUT
    out = layer.forward(hid, lg, mp)
    assert layer.device_status() == m.MOE_OK
    assert_output_close(to_f64(out), oracle.forward_inputs(inp)["out64"], "after flag timeout")


@pytest.mark.parametrize("shape", ["small", "decode_T16"])
def test_peft_adapters_separate_gate_up_mixed_ranks_and_scales(shape):
    """Separate gate/up pairs, per-adapter ranks and scales, packed into the
    fused layout (block-diagonal, zero-padded) and run through the kernels,
    against the oracle's direct per-projection formulation."""
    import moe_lora_expert_gb300 as m
    from moe_lora_expert_gb300 import adapters as pk
    torch = torch_mod()
    specs = [("separate", 8, 16.0), ("fused", 16, 32.0), ("separate", 16, 8.0), ("fused", 8, 8.0)]
    if shape == "small":
        wl = workloads.small_workload("peft_gpu", T=40, H=128, I=64, E=6, top_k=2, num_adapters=4,
                                      rank=8, map_lo=-1, map_hi=3, seed=81)
    else:
        wl = workloads.WORKLOADS["decode_T16"]
    inp = workloads.make_inputs(wl) if shape == "small" else cached_inputs("decode_T16")
    ads = workloads.make_peft_adapters(wl, specs, seed=82)
    ads_t = [{"scaling": ad["scaling"], **{k: (bf16_tensor(v[0]), bf16_tensor(v[1]))
                                           for k, v in ad.items() if k != "scaling"}} for ad in ads]
    A_gu, B_gu, A_dn, B_dn, scales = pk.pack_adapters(ads_t, wl.E, wl.H, wl.I)
    layer = m.MoeLoraLayer(bf16_tensor(inp.w13), bf16_tensor(inp.w2), wl.top_k, A_gu, B_gu, A_dn,
                           B_dn, scaling=1.0, adapter_scaling=scales)
    mapping = inp.mapping.clip(-1, 3).astype(np.int32)
    out = layer.forward(bf16_tensor(inp.hidden), torch.from_numpy(inp.logits).to(dev()),
                        torch.from_numpy(mapping).to(dev()))
    assert layer.device_status() == 0
    ref, _ = oracle.moe_lora_forward_general(inp.hidden, inp.logits, inp.w13, inp.w2, mapping,
                                             wl.top_k, ads)
    assert_output_close(to_f64(out), ref, f"peft {shape}")


@pytest.mark.parametrize("max_ctas", [152, 5, 1])
@pytest.mark.parametrize("name", ["decode_T16", "decode_T64_mixed8"])
def test_shrink_in_gemm_needs_no_co_resident_grid(name, max_ctas):
    """The in-GEMM shrink hands its rows to running CTAs only (a row counter),
    so a producer never waits on a row that a CTA which has not started owns.
    With the expert GEMMs' persistent grid cut to one CTA per SM, to five
    CTAs, or to one CTA (which then shrinks every row itself), the forward is
    correct and no wait runs out."""
    inp = cached_inputs(name)
    res = run_gpu(inp, tuning={"gemm_max_ctas": max_ctas})
    assert res["status"] == 0, res["status_str"]
    check_routing(res, inp)
    assert_output_close(res["out64"], oracle.forward_inputs(inp)["out64"], f"{name} ctas={max_ctas}")


@pytest.mark.parametrize("name", ["tiny_T8", "decode_T16", "decode_T64_mixed8",
                                  "skewed_T256_shared_outer_r64"])
def test_two_stream_gate_up_shrink(name):
    """The two-stream schedule: the gate_up LoRA shrink on a second stream,
    forked after the permute and joined by an event before the gate_up GEMM,
    while the main stream gathers the rows.  Against the oracle, eager and
    replayed from a CUDA graph captured on the main stream."""
    torch = torch_mod()
    inp = cached_inputs(name)
    side = torch.cuda.Stream()
    evs = [torch.cuda.Event(), torch.cuda.Event()]
    res = run_gpu(inp, side_stream=side, side_events=evs)
    assert res["status"] == 0, res["status_str"]
    check_routing(res, inp)
    ref = oracle.forward_inputs(inp)["out64"]
    assert_output_close(res["out64"], ref, f"{name} two streams")
    layer = res["layer"]
    hid = bf16_tensor(inp.hidden)
    lg = torch.from_numpy(inp.logits).to(dev())
    mp = torch.from_numpy(inp.mapping).to(dev())
    out = torch.empty_like(res["out"])
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.forward(hid, lg, mp, out=out, side_stream=side, side_events=evs)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), res["out"].view(torch.int16)), name
    assert layer.device_status() == 0


@pytest.mark.parametrize("T,k,E,shard", [(2500, 4, 200, None), (5000, 2, 256, None), (3000, 8, 96, (40, 56))])
def test_forward_two_kernel_route_permute(T, k, E, shard):
    """Past the one-CTA permute (more than 8192 slots) routing and the
    permutation run as three chained kernels (routing, count per chunk of
    whole tokens, scan + scatter per chunk): ragged last chunk, E up to 256, top-k 2..8,
    out-of-range mappings (flagged, treated as none), and an expert shard
    (slots of other shards dropped).  Routing and the permutation bit-exact,
    the output against the oracle."""
    import moe_lora_expert_gb300 as m
    wl = workloads.small_workload("rp", T=T, H=64, I=32, E=E, top_k=k, num_adapters=3, rank=8,
                                  map_lo=-1, map_hi=2, seed=T + E)
    inp = workloads.make_inputs(wl)
    mapping = inp.mapping.copy()
    mapping[::97] = 7          # outside [-1, 3): reported, treated as -1
    ref_map = np.where((mapping >= -1) & (mapping < 3), mapping, -1).astype(np.int32)
    if shard is None:
        res = run_gpu(inp, mapping=mapping)
        assert res["status"] == m.MOE_ERR_BAD_MAPPING, res["status_str"]
        check_routing(res, inp)
        ref_inp = workloads.LayerInputs(inp.wl, inp.logits, inp.hidden, inp.w13, inp.w2, inp.A_gu, inp.B_gu,
                                        inp.A_dn, inp.B_dn, ref_map)
        assert_output_close(res["out64"], oracle.forward_inputs(ref_inp)["out64"], f"rp T={T} k={k}")
    else:
        off, cnt = shard
        sub = workloads.shard_experts(inp, off, cnt)
        layer = make_layer(sub, local_expert_offset=off, num_router_experts=E)
        res = run_gpu(sub, layer=layer, mapping=mapping)
        assert res["status"] == m.MOE_ERR_BAD_MAPPING, res["status_str"]
        check_routing(res, inp, shard=(off, cnt))
        ref_sub = workloads.LayerInputs(sub.wl, sub.logits, sub.hidden, sub.w13, sub.w2, sub.A_gu, sub.B_gu,
                                        sub.A_dn, sub.B_dn, ref_map)
        ref = oracle.forward_inputs(ref_sub, local_expert_offset=off)["out64"]
        assert_output_close(res["out64"], ref, f"rp shard {shard}")
