"""Helpers shared by the GPU parity tests: upload seeded inputs, run the CUDA
path through the C ABI, compare with the oracle."""
import functools

import numpy as np

import oracle
import workloads

# Output acceptance: per element |gpu - ref| <= ATOL + RTOL*|ref|, and the
# relative Frobenius error of the whole compared block <= FROB.
ATOL, RTOL, FROB = 3e-2, 2e-2, 1e-2
# Routing weights: float32 exp/sum/divide against the float64 oracle.  With
# unit roundoff u = 2^-24, |l - m| <= 16 and k <= 32 terms, the float32 result
# is within (|l - m| + 2 + 2 + k + 1) u < 3.2e-6 relative; 4e-6 is used.
W_RTOL = 4e-6


def torch_mod():
    import torch
    return torch


def dev():
    return torch_mod().device("cuda:0")


def bf16_tensor(a):
    torch = torch_mod()
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev()).view(torch.bfloat16)


def to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


@functools.lru_cache(maxsize=8)
def cached_inputs(name):
    return workloads.make_inputs(workloads.WORKLOADS[name])


def make_layer(inp, with_lora=True, **shard):
    """``shard``: local_expert_offset / num_router_experts for an expert shard."""
    import moe_lora_expert_gb300 as m
    wl = inp.wl
    if with_lora and inp.A_gu is not None:
        return m.MoeLoraLayer(bf16_tensor(inp.w13), bf16_tensor(inp.w2), wl.top_k,
                              bf16_tensor(inp.A_gu), bf16_tensor(inp.B_gu), bf16_tensor(inp.A_dn),
                              bf16_tensor(inp.B_dn), scaling=wl.scaling, **shard)
    return m.MoeLoraLayer(bf16_tensor(inp.w13), bf16_tensor(inp.w2), wl.top_k, scaling=wl.scaling,
                          **shard)


def run_gpu(inp, layer=None, tile_n=0, with_lora=True, mapping=None, **fwd):
    """Returns dict(out64, ids, w, e2p, status, layer).  ``fwd``: further
    forward arguments (tuning, side_stream, side_events, ...)."""
    import moe_lora_expert_gb300 as m
    torch = torch_mod()
    wl = inp.wl
    T = inp.hidden.shape[0]
    layer = layer or make_layer(inp, with_lora)
    ids = torch.empty((T, wl.top_k), dtype=torch.int32, device=dev())
    w = torch.empty((T, wl.top_k), dtype=torch.float32, device=dev())
    e2p = torch.empty((T * wl.top_k,), dtype=torch.int32, device=dev())
    mp = inp.mapping if mapping is None else mapping
    out = layer.forward(bf16_tensor(inp.hidden), torch.from_numpy(inp.logits).to(dev()),
                        torch.from_numpy(np.ascontiguousarray(mp, dtype=np.int32)).to(dev())
                        if layer.num_adapters else None,
                        topk_ids=ids, topk_w=w, expanded_to_permuted=e2p, tile_n=tile_n, **fwd)
    status = layer.device_status()
    torch.cuda.synchronize()
    return {"out64": to_f64(out), "out": out, "ids": ids.cpu().numpy(), "w": w.cpu().numpy(),
            "e2p": e2p.cpu().numpy(), "status": status, "layer": layer, "status_str": m.status_string(status)}


def assert_output_close(got, ref, label=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), f"{label}: non-finite output"
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{label}: {bad.sum()} elements out of tolerance, worst at "
                           f"{np.unravel_index(np.argmax(err - bound), err.shape)}: "
                           f"got {got.flat[np.argmax(err - bound)]}, ref {ref.flat[np.argmax(err - bound)]}")
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert rel <= FROB, f"{label}: relative Frobenius error {rel:.3e} > {FROB}"
    return rel


def check_routing(res, inp, shard=None):
    """ids and the permutation bit-exact; weights within W_RTOL.  ``shard`` =
    (offset, count) of an expert shard: the ids stay global, the permutation
    is over the shard's experts, other slots dropped (-1)."""
    ids_ref, w_ref = oracle.route_topk(inp.logits, inp.wl.top_k)
    assert np.array_equal(res["ids"], ids_ref), "routing ids differ from the oracle"
    np.testing.assert_allclose(res["w"], w_ref, rtol=W_RTOL, atol=1e-9)
    if shard is None:
        _, e2p_ref, _ = oracle.permute(ids_ref, inp.wl.E)
    else:
        off, cnt = shard
        local = ids_ref - off
        local = np.where((local >= 0) & (local < cnt), local, -1).astype(np.int32)
        _, e2p_ref, _ = oracle.permute(local, cnt)
    assert np.array_equal(res["e2p"], e2p_ref), "expanded_to_permuted differs from the oracle"
    return ids_ref
