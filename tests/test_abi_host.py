"""C ABI checks that need no GPU: the library loads, exports every function
that include/moe_lora.h declares, plans workspaces, and rejects invalid
arguments on the host before launching anything."""
import ctypes
import os
import re

import pytest

import moe_lora_expert_gb300 as m

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_lora.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(m.LIB_PATH):
        from moe_lora_expert_gb300 import _build
        _build.build()
    return m.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(moe_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ["moe_route_topk", "moe_permute", "moe_lora_forward", "moe_lora_workspace_size",
                 "moe_read_device_status", "moe_status_string"]:
        assert must in names
    assert sorted(names) == sorted(m.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_abi_version_and_struct_layout(lib, tmp_path):
    """ctypes field offsets equal the C compiler's offsetof for every field."""
    import shutil
    import subprocess
    assert lib.moe_lora_abi_version() == 1
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    checks = []
    structs = [(m.LoraFactors, "moe_lora_factors_t"), (m.MoeLoraArgs, "moe_lora_args_t"),
               (m.WorkspacePlan, "moe_lora_workspace_plan_t"), (m.Tuning, "moe_lora_tuning_t")]
    for struct, ctype in structs:
        checks.append(f'printf("%s sizeof %zu\\n", "{ctype}", sizeof({ctype}));')
        for fname, _ in struct._fields_:
            checks.append(f'printf("%s %s %zu\\n", "{ctype}", "{fname}", offsetof({ctype}, {fname}));')
    prog = tmp_path / "layout.c"
    prog.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "moe_lora.h"\n'
                    "int main(void) {\n" + "\n".join(checks) + "\nreturn 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)], check=True)
    lines = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = {}
    for ln in lines:
        if ln.strip():
            *key, val = ln.split()
            got[" ".join(key)] = int(val)
    for struct, ctype in structs:
        assert got[f"{ctype} sizeof"] == ctypes.sizeof(struct), ctype
        for fname, _ in struct._fields_:
            assert got[f"{ctype} {fname}"] == getattr(struct, fname).offset, (ctype, fname)


def test_status_strings(lib):
    for code in range(0, -10, -1):
        s = m.status_string(code)
        assert s.startswith("MOE_"), (code, s)
    assert "unknown" in m.status_string(-99)


def test_workspace_plan(lib):
    T, H, I, E, k, A, r = 16, 2048, 768, 128, 8, 4, 16
    plan = m.moe_lora_workspace_plan(T, H, I, E, k, A, r)
    n = T * k
    assert plan.total_bytes == m.moe_lora_workspace_size(T, H, I, E, k, A, r)
    offs = [plan.status, plan.topk_ids, plan.topk_w, plan.expert_offsets, plan.expanded_to_permuted,
            plan.permuted_to_expanded, plan.row_adapter, plan.permute_scratch, plan.permuted_hidden,
            plan.lora_u, plan.act]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert plan.act + n * I * 2 <= plan.total_bytes
    assert plan.lora_u + n * A * r * 2 <= plan.act
    # the down GEMM output reuses the permuted hidden rows, the down operand the gate_up one
    assert plan.expert_out == plan.permuted_hidden and plan.lora_v == plan.lora_u
    # no LoRA -> no LoRA operand
    p0 = m.moe_lora_workspace_plan(T, H, I, E, k, 0, 0)
    assert p0.act == p0.lora_u
    assert m.moe_lora_workspace_size(0, H, I, E, k, A, r) > 0


@pytest.mark.parametrize("args,status", [
    ((16, 2048, 768, 128, 129, 4, 16), m.MOE_ERR_UNSUPPORTED),   # top_k > 32
    ((16, 2048, 768, 8, 9, 4, 16), m.MOE_ERR_SHAPE),             # top_k > E
    ((16, 2044, 768, 128, 8, 4, 16), m.MOE_ERR_ALIGN),           # H % 8
    ((16, 2048, 770, 128, 8, 4, 16), m.MOE_ERR_ALIGN),           # I % 8
    ((16, 2048, 768, 128, 8, 4, 12), m.MOE_ERR_UNSUPPORTED),     # rank % 8
    ((16, 2048, 768, 128, 8, 4, 136), m.MOE_ERR_UNSUPPORTED),    # rank > 128
    ((16, 2048, 768, 128, 8, 65, 16), m.MOE_ERR_UNSUPPORTED),    # adapters > 64
    ((16, 2048, 768, 1025, 8, 4, 16), m.MOE_ERR_UNSUPPORTED),    # E > 1024
    ((-1, 2048, 768, 128, 8, 4, 16), m.MOE_ERR_SHAPE),
])
def test_plan_rejects(lib, args, status):
    plan = m.WorkspacePlan()
    assert lib.moe_lora_workspace_plan(*args, ctypes.byref(plan)) == status
    assert lib.moe_lora_workspace_size(*args) == 0


def _valid_args(**over):
    """Arguments that pass every host check except the ones overridden.  The
    pointers are fake (never dereferenced: each case fails a check first)."""
    a = m.MoeLoraArgs()
    a.struct_size = ctypes.sizeof(m.MoeLoraArgs)
    a.T, a.H, a.I, a.E, a.top_k, a.num_adapters, a.rank = 16, 2048, 768, 128, 8, 4, 16
    a.scaling = 2.0
    fake = 1 << 20
    a.hidden = a.w13 = a.w2 = a.router_logits = a.token_lora_mapping = a.out = fake
    a.gate_up = m.LoraFactors(fake, fake, 128 * 16 * 2048, 16 * 2048, 128 * 1536 * 16, 1536 * 16)
    a.down = m.LoraFactors(fake, fake, 128 * 16 * 768, 16 * 768, 128 * 2048 * 16, 2048 * 16)
    a.workspace = fake
    a.workspace_bytes = m.moe_lora_workspace_size(16, 2048, 768, 128, 8, 4, 16)
    for k, v in over.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("over,status", [
    ({"struct_size": 8}, m.MOE_ERR_UNSUPPORTED),
    ({"hidden": None}, m.MOE_ERR_NULL),
    ({"out": None}, m.MOE_ERR_NULL),
    ({"router_logits": None}, m.MOE_ERR_NULL),
    ({"workspace": None}, m.MOE_ERR_NULL),
    ({"token_lora_mapping": None}, m.MOE_ERR_NULL),
    ({"w13": (1 << 20) + 8}, m.MOE_ERR_ALIGN),
    ({"workspace": (1 << 20) + 128}, m.MOE_ERR_WORKSPACE),
    ({"workspace_bytes": 1024}, m.MOE_ERR_WORKSPACE),
    ({"top_k": 200}, m.MOE_ERR_UNSUPPORTED),
    ({"top_k": 0}, m.MOE_ERR_SHAPE),
    ({"tile_n": 48}, m.MOE_ERR_UNSUPPORTED),
    ({"wait_timeout_ms": -1}, m.MOE_ERR_SHAPE),
    ({"rank": 20}, m.MOE_ERR_UNSUPPORTED),
    ({"gate_up": m.LoraFactors(1 << 20, 1 << 20, 4, 0, 0, 0)}, m.MOE_ERR_ALIGN),
    ({"down": m.LoraFactors(1 << 20, 1 << 20, 8, 8, 24, 0)}, m.MOE_ERR_ALIGN),   # b stride % r
    ({"down": m.LoraFactors(1 << 20, 1 << 20, -8, 0, 0, 0)}, m.MOE_ERR_SHAPE),
    ({"down": m.LoraFactors(1 << 20, None, 8, 8, 16, 0)}, m.MOE_ERR_NULL),
    # expert parallelism: shard outside the router's experts, router too wide
    ({"num_router_experts": 256, "local_expert_offset": 129}, m.MOE_ERR_SHAPE),
    ({"num_router_experts": 256, "local_expert_offset": -1}, m.MOE_ERR_SHAPE),
    ({"num_router_experts": 64}, m.MOE_ERR_SHAPE),                     # fewer than E
    ({"num_router_experts": 2048, "local_expert_offset": 0}, m.MOE_ERR_SHAPE),
    ({"local_expert_offset": 1}, m.MOE_ERR_SHAPE),                     # no room without a router width
    # a valid shard passes the shard checks (then fails on the fake workspace size)
    ({"num_router_experts": 256, "local_expert_offset": 128, "workspace_bytes": 1024},
     m.MOE_ERR_WORKSPACE),
    # structures from before the shard fields, or before the weight-format
    # fields: accepted with the defaults, checks go on
    ({"struct_size": m.MoeLoraArgs.local_expert_offset.offset, "hidden": None}, m.MOE_ERR_NULL),
    ({"struct_size": m.MoeLoraArgs.weight_format.offset, "hidden": None}, m.MOE_ERR_NULL),
    ({"struct_size": m.MoeLoraArgs.local_expert_offset.offset - 4}, m.MOE_ERR_UNSUPPORTED),
    # FP8 block-scaled weights
    ({"weight_format": 2}, m.MOE_ERR_UNSUPPORTED),
    ({"weight_format": m.MOE_WEIGHTS_FP8_E4M3_B128}, m.MOE_ERR_NULL),          # no scales
    ({"weight_format": m.MOE_WEIGHTS_FP8_E4M3_B128, "w13_scale": 1 << 20, "w2_scale": (1 << 20) + 2},
     m.MOE_ERR_ALIGN),
    ({"weight_format": m.MOE_WEIGHTS_FP8_E4M3_B128, "H": 2056}, m.MOE_ERR_ALIGN),  # 1-byte rows
    # kernel-choice overrides outside their sets
    ({"tuning": m.Tuning(cta_pairs=3)}, m.MOE_ERR_UNSUPPORTED),
    ({"tuning": m.Tuning(shrink_kernel=-1)}, m.MOE_ERR_UNSUPPORTED),
    ({"tuning": m.Tuning(shrink_in_gemm=3)}, m.MOE_ERR_UNSUPPORTED),
    ({"tuning": m.Tuning(gemm_max_ctas=-5)}, m.MOE_ERR_UNSUPPORTED),
    # a structure from before the tuning fields ignores them (checks go on)
    ({"struct_size": m.MoeLoraArgs.tuning.offset, "tuning": m.Tuning(cta_pairs=3), "hidden": None},
     m.MOE_ERR_NULL),
    # the two-stream schedule needs both events
    ({"side_stream": 1 << 12}, m.MOE_ERR_NULL),
    # FP8 activations: a known format, FP8 weights, the larger workspace
    ({"activation_format": 2}, m.MOE_ERR_UNSUPPORTED),
    ({"activation_format": m.MOE_ACT_FP8_E4M3_G128}, m.MOE_ERR_UNSUPPORTED),   # bf16 weights
    ({"activation_format": m.MOE_ACT_FP8_E4M3_G128, "weight_format": m.MOE_WEIGHTS_FP8_E4M3_B128,
      "w13_scale": 1 << 20, "w2_scale": 1 << 20}, m.MOE_ERR_WORKSPACE),    # bf16-sized workspace
    # a structure from before activation_format ignores it (checks go on)
    ({"struct_size": m.MoeLoraArgs.activation_format.offset, "activation_format": 2, "hidden": None},
     m.MOE_ERR_NULL),
])
def test_forward_rejects_on_host(lib, over, status):
    a = _valid_args(**over)
    assert lib.moe_lora_forward(ctypes.byref(a), None) == status


def test_forward_null_args(lib):
    assert lib.moe_lora_forward(None, None) == m.MOE_ERR_NULL


def test_route_and_permute_reject_on_host(lib):
    fake = 1 << 20
    assert lib.moe_route_topk(fake, 4, 8, 9, fake, fake, None) == m.MOE_ERR_SHAPE
    assert lib.moe_route_topk(fake, 4, 2048, 8, fake, fake, None) == m.MOE_ERR_UNSUPPORTED
    assert lib.moe_route_topk(None, 4, 8, 2, fake, fake, None) == m.MOE_ERR_NULL
    assert lib.moe_route_topk(None, 0, 8, 2, None, None, None) == m.MOE_OK   # T == 0: nothing to do
    ws = m.lib().moe_permute_workspace_size(4, 2, 8)
    assert ws > 0
    assert lib.moe_permute(fake, 4, 2, 8, None, 0, fake, fake, fake, None, fake + 64, ws, None) == \
        m.MOE_ERR_WORKSPACE
    assert lib.moe_permute(fake, 4, 2, 8, None, 0, fake, fake, fake, None, fake, 16, None) == \
        m.MOE_ERR_WORKSPACE
    assert lib.moe_permute(fake, 4, 2, 8, fake, 12, fake, fake, fake, fake, fake, ws, None) == \
        m.MOE_ERR_ALIGN
    assert lib.moe_permute(fake, 4, 2, 8, None, 0, None, fake, fake, None, fake, ws, None) == \
        m.MOE_ERR_NULL


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(m, "_lib", None)
    monkeypatch.setattr(m, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        m.lib()


def test_fp8_workspace_and_quant_host_checks(lib):
    base = lib.moe_lora_workspace_size(16, 2048, 768, 128, 8, 4, 16)
    assert lib.moe_lora_workspace_size_ex(16, 2048, 768, 128, 8, 4, 16, m.MOE_ACT_BF16) == base
    n = 16 * 8
    extra = lib.moe_lora_workspace_size_ex(16, 2048, 768, 128, 8, 4, 16, m.MOE_ACT_FP8_E4M3_G128) - base
    # quantized rows, their scales, the float32 activation, its codes and scales
    assert extra >= n * 2048 + n * 16 * 4 + n * 768 * 4 + n * 768 + n * 6 * 4
    assert lib.moe_lora_workspace_size_ex(16, 2048, 768, 128, 8, 4, 16, 7) == 0
    fake = 1 << 20
    q = lib.moe_per_token_group_quant_fp8
    assert q(fake, 0, 4, 24, None, 1, fake, fake, None) == m.MOE_ERR_ALIGN       # K % 16
    assert q(fake, 2, 4, 32, None, 1, fake, fake, None) == m.MOE_ERR_SHAPE       # x type flag
    assert q(fake, 0, 4, 32, None, 0, fake, fake, None) == m.MOE_ERR_SHAPE       # map_div
    assert q(None, 0, 4, 32, None, 1, fake, fake, None) == m.MOE_ERR_NULL
    assert q(fake + 8, 0, 4, 32, None, 1, fake, fake, None) == m.MOE_ERR_ALIGN
    assert q(None, 0, 0, 32, None, 1, None, None, None) == m.MOE_OK              # nothing to do
