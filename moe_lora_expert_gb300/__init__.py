"""Python binding of libmoelora, the GB300 (sm_103a) routed MoE-LoRA forward.

Argument marshalling only: every step of the forward runs in the library's
CUDA kernels.  PyTorch supplies device memory and the current stream.  There
is no CPU or PyTorch fallback: if the compiled library is missing, importing
the binding's functions raises.

Functions with the C names (``moe_route_topk``, ``moe_permute``,
``moe_lora_forward``, ...) take torch tensors and call the C ABI of
``include/moe_lora.h`` through ctypes.  ``MoeLoraLayer`` holds one layer's
weights and a workspace and runs the forward on the current stream.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libmoelora.so")

MOE_OK = 0
MOE_ERR_NULL = -1
MOE_ERR_SHAPE = -2
MOE_ERR_ALIGN = -3
MOE_ERR_UNSUPPORTED = -4
MOE_ERR_WORKSPACE = -5
MOE_ERR_CUDA = -6
MOE_ERR_DEVICE_TIMEOUT = -7
MOE_ERR_BAD_MAPPING = -8
MOE_ERR_BAD_EXPERT_ID = -9
MOE_NUM_STAGE_EVENTS = 8
MOE_WEIGHTS_BF16 = 0
MOE_WEIGHTS_FP8_E4M3_B128 = 1
MOE_ACT_BF16 = 0
MOE_ACT_FP8_E4M3_G128 = 1
MOE_ACT_FP8_GROUP = 128
MOE_DEBUG_STALL_GATE_UP_MMA = 1
MOE_DEBUG_HOLD_SHRINK_ROW = 2
STAGE_NAMES = ["route", "permute", "shrink_gate_up", "gemm_gate_up", "shrink_down", "gemm_down",
               "finalize"]

EXPORTED_SYMBOLS = [
    "moe_status_string", "moe_lora_abi_version", "moe_route_topk", "moe_permute_workspace_size",
    "moe_permute", "moe_lora_workspace_plan", "moe_lora_workspace_size", "moe_lora_forward",
    "moe_read_device_status", "moe_permute_noalloc", "moe_per_token_group_quant_fp8",
    "moe_lora_workspace_size_ex",
]


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class LoraFactors(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("B", ctypes.c_void_p),
                ("a_stride_adapter", ctypes.c_int64), ("a_stride_expert", ctypes.c_int64),
                ("b_stride_adapter", ctypes.c_int64), ("b_stride_expert", ctypes.c_int64)]


class Tuning(ctypes.Structure):
    """Kernel-choice overrides (moe_lora_tuning_t); all zero = the library's choices."""
    _fields_ = [("cta_pairs", ctypes.c_int), ("shrink_kernel", ctypes.c_int),
                ("shrink_in_gemm", ctypes.c_int), ("gemm_max_ctas", ctypes.c_int)]


class MoeLoraArgs(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_uint32),
                ("T", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int), ("E", ctypes.c_int),
                ("top_k", ctypes.c_int), ("num_adapters", ctypes.c_int), ("rank", ctypes.c_int),
                ("scaling", ctypes.c_float),
                ("hidden", ctypes.c_void_p), ("w13", ctypes.c_void_p), ("w2", ctypes.c_void_p),
                ("router_logits", ctypes.c_void_p), ("token_lora_mapping", ctypes.c_void_p),
                ("gate_up", LoraFactors), ("down", LoraFactors),
                ("out", ctypes.c_void_p),
                ("topk_ids_out", ctypes.c_void_p), ("topk_w_out", ctypes.c_void_p),
                ("expanded_to_permuted_out", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("tile_n", ctypes.c_int), ("wait_timeout_ms", ctypes.c_int),
                ("debug_flags", ctypes.c_uint32),
                ("stage_events", ctypes.c_void_p),
                ("adapter_scaling", ctypes.c_void_p),
                ("local_expert_offset", ctypes.c_int), ("num_router_experts", ctypes.c_int),
                ("weight_format", ctypes.c_int), ("w13_scale", ctypes.c_void_p),
                ("w2_scale", ctypes.c_void_p),
                ("tuning", Tuning),
                ("side_stream", ctypes.c_void_p), ("side_events", ctypes.c_void_p * 2),
                ("activation_format", ctypes.c_int)]


class WorkspacePlan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "total_bytes", "status", "topk_ids", "topk_w", "expert_offsets", "expanded_to_permuted",
        "permuted_to_expanded", "row_adapter", "permute_scratch", "permuted_hidden", "lora_u",
        "act", "lora_v", "expert_out")]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C library.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_status_string.argtypes = [i32]
        L.moe_lora_abi_version.restype = i32
        L.moe_route_topk.restype = i32
        L.moe_route_topk.argtypes = [vp, i32, i32, i32, vp, vp, vp]
        L.moe_permute_workspace_size.restype = sz
        L.moe_permute_workspace_size.argtypes = [i32, i32, i32]
        L.moe_permute.restype = i32
        L.moe_permute.argtypes = [vp, i32, i32, i32, vp, i32, vp, vp, vp, vp, vp, sz, vp]
        L.moe_lora_workspace_plan.restype = i32
        L.moe_lora_workspace_plan.argtypes = [i32] * 7 + [ctypes.POINTER(WorkspacePlan)]
        L.moe_lora_workspace_size.restype = sz
        L.moe_lora_workspace_size.argtypes = [i32] * 7
        L.moe_lora_forward.restype = i32
        L.moe_lora_forward.argtypes = [ctypes.POINTER(MoeLoraArgs), vp]
        L.moe_read_device_status.restype = i32
        L.moe_read_device_status.argtypes = [vp, vp]
        L.moe_permute_noalloc.restype = i32
        L.moe_permute_noalloc.argtypes = [vp, i32, i32, i32, vp, i32, vp, vp, vp, vp, vp, vp]
        L.moe_per_token_group_quant_fp8.restype = i32
        L.moe_per_token_group_quant_fp8.argtypes = [vp, i32, i32, i32, vp, i32, vp, vp, vp]
        L.moe_lora_workspace_size_ex.restype = sz
        L.moe_lora_workspace_size_ex.argtypes = [i32] * 8
        _lib = L
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().moe_status_string(int(status)).decode()
    except ImportError:
        return "libmoelora not built"


def _check(status: int, what: str):
    if status != MOE_OK:
        raise MoeError(status, what)


# ----------------------------------------------------------------------------
# torch helpers (allocation and stream plumbing only)
# ----------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream=None) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _require(t, dtype, shape, name):
    torch = _torch()
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


# ----------------------------------------------------------------------------
# Entry points with the C names
# ----------------------------------------------------------------------------

def moe_route_topk(logits, top_k: int, topk_ids=None, topk_w=None, stream=None):
    torch = _torch()
    T, E = logits.shape
    _require(logits, torch.float32, (T, E), "logits")
    if topk_ids is None:
        topk_ids = torch.empty((T, top_k), dtype=torch.int32, device=logits.device)
    if topk_w is None:
        topk_w = torch.empty((T, top_k), dtype=torch.float32, device=logits.device)
    _check(lib().moe_route_topk(_ptr(logits), T, E, top_k, _ptr(topk_ids), _ptr(topk_w),
                                _stream_handle(stream)), "moe_route_topk")
    return topk_ids, topk_w


def moe_permute(topk_ids, E: int, hidden=None, gather=True, stream=None):
    """Returns (expert_offsets, expanded_to_permuted, permuted_to_expanded, permuted_hidden, ws)."""
    torch = _torch()
    T, k = topk_ids.shape
    dev = topk_ids.device
    _require(topk_ids, torch.int32, (T, k), "topk_ids")
    H = hidden.shape[1] if hidden is not None else 0
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    e2p = torch.empty(T * k, dtype=torch.int32, device=dev)
    p2e = torch.empty(T * k, dtype=torch.int32, device=dev)
    permuted = None
    if hidden is not None and gather:
        _require(hidden, torch.bfloat16, (T, H), "hidden")
        permuted = torch.empty((T * k, H), dtype=torch.bfloat16, device=dev)
    ws_bytes = lib().moe_permute_workspace_size(T, k, E)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    _check(lib().moe_permute(_ptr(topk_ids), T, k, E, _ptr(hidden), H, _ptr(offsets), _ptr(e2p),
                             _ptr(p2e), _ptr(permuted), _ptr(ws), ws.numel(),
                             _stream_handle(stream)), "moe_permute")
    return offsets, e2p, p2e, permuted, ws


def moe_lora_workspace_plan(T, H, I, E, top_k, num_adapters, rank) -> WorkspacePlan:
    plan = WorkspacePlan()
    _check(lib().moe_lora_workspace_plan(T, H, I, E, top_k, num_adapters, rank, ctypes.byref(plan)),
           "moe_lora_workspace_plan")
    return plan


def moe_lora_workspace_size(T, H, I, E, top_k, num_adapters, rank) -> int:
    return int(lib().moe_lora_workspace_size(T, H, I, E, top_k, num_adapters, rank))


def moe_lora_workspace_size_ex(T, H, I, E, top_k, num_adapters, rank, activation_format) -> int:
    return int(lib().moe_lora_workspace_size_ex(T, H, I, E, top_k, num_adapters, rank,
                                                activation_format))


def moe_per_token_group_quant_fp8(x, row_map=None, map_div=1, rows=None, stream=None):
    """Codes (uint8 [rows, K]) and scales (float32 [rows, ceil(K / 128)]) of
    the rows of ``x`` (bf16 or float32 [*, K]); ``row_map``: int32 [rows],
    output row i reads x row row_map[i] // map_div (negative: a zero row)."""
    torch = _torch()
    if x.dtype not in (torch.bfloat16, torch.float32) or not x.is_contiguous() or x.dim() != 2:
        raise ValueError("x must be a contiguous bf16 or float32 matrix")
    K = x.shape[1]
    if rows is None:
        rows = row_map.shape[0] if row_map is not None else x.shape[0]
    codes = torch.empty((rows, K), dtype=torch.uint8, device=x.device)
    scales = torch.empty((rows, (K + MOE_ACT_FP8_GROUP - 1) // MOE_ACT_FP8_GROUP), dtype=torch.float32,
                         device=x.device)
    _check(lib().moe_per_token_group_quant_fp8(_ptr(x), 1 if x.dtype == torch.float32 else 0, rows, K,
                                               _ptr(row_map), map_div, _ptr(codes), _ptr(scales),
                                               _stream_handle(stream)), "moe_per_token_group_quant_fp8")
    return codes, scales


def moe_lora_forward(args: MoeLoraArgs, stream=None) -> int:
    """Raw call: returns the status code (no raise)."""
    return int(lib().moe_lora_forward(ctypes.byref(args), _stream_handle(stream)))


def moe_read_device_status(workspace, stream=None) -> int:
    return int(lib().moe_read_device_status(_ptr(workspace), _stream_handle(stream)))


# ----------------------------------------------------------------------------
# Layer object
# ----------------------------------------------------------------------------

class MoeLoraLayer:
    """One routed MoE layer with per-(adapter, expert) LoRA, weights on the GPU.

    w13 [E, 2I, H] bf16, w2 [E, H, I] bf16.  LoRA factors (bf16, optional):
    A_gu [A, E, r, H] or shared [A, r, H]; B_gu [A, E, 2I, r];
    A_dn [A, E, r, I]; B_dn [A, E, H, r] or shared [A, H, r].

    FP8 weights: w13 / w2 as uint8 (or float8_e4m3fn) e4m3 codes with
    ``w13_scale`` [E, ceil(2I/128), ceil(H/128)] and ``w2_scale``
    [E, ceil(H/128), ceil(I/128)] float32 block scales (128 x 128 blocks).

    Expert parallelism: ``num_router_experts`` > E makes this layer one shard
    holding experts [local_expert_offset, local_expert_offset + E) of a router
    over num_router_experts experts (router_logits [T, num_router_experts]);
    its forward returns the shard's partial sum (see ``ep``).
    """

    def __init__(self, w13, w2, top_k: int, A_gu=None, B_gu=None, A_dn=None, B_dn=None,
                 scaling: float = 1.0, max_tokens: int = 0, adapter_scaling=None,
                 local_expert_offset: int = 0, num_router_experts: int = 0,
                 w13_scale=None, w2_scale=None, fp8_activations: bool = False):
        torch = _torch()
        self.E, twoI, self.H = w13.shape
        self.local_expert_offset = int(local_expert_offset)
        self.num_router_experts = int(num_router_experts) or self.E
        self.I = twoI // 2
        self.fp8 = w13.dtype != torch.bfloat16
        if self.fp8:
            fp8_types = (torch.uint8,) + ((torch.float8_e4m3fn,) if hasattr(torch, "float8_e4m3fn") else ())
            if w13.dtype not in fp8_types or w2.dtype != w13.dtype:
                raise TypeError("FP8 weights: w13 and w2 as uint8 or float8_e4m3fn")
            _require(w13, w13.dtype, (self.E, 2 * self.I, self.H), "w13")
            _require(w2, w2.dtype, (self.E, self.H, self.I), "w2")
            nb = lambda n: (n + 127) // 128
            _require(w13_scale, torch.float32, (self.E, nb(2 * self.I), nb(self.H)), "w13_scale")
            _require(w2_scale, torch.float32, (self.E, nb(self.H), nb(self.I)), "w2_scale")
        else:
            _require(w13, torch.bfloat16, (self.E, 2 * self.I, self.H), "w13")
            _require(w2, torch.bfloat16, (self.E, self.H, self.I), "w2")
        self.w13_scale, self.w2_scale = w13_scale, w2_scale
        if fp8_activations and not self.fp8:
            raise TypeError("FP8 activations need FP8 weights (W8A8)")
        self.act_format = MOE_ACT_FP8_E4M3_G128 if fp8_activations else MOE_ACT_BF16
        self.w13, self.w2, self.top_k, self.scaling = w13, w2, top_k, float(scaling)
        self.A_gu, self.B_gu, self.A_dn, self.B_dn = A_gu, B_gu, A_dn, B_dn
        if A_gu is not None:
            self.num_adapters = A_gu.shape[0]
            self.rank = A_gu.shape[-2]
            E, H, I, A, r = self.E, self.H, self.I, self.num_adapters, self.rank
            gu_shared = A_gu.dim() == 3
            dn_shared = B_dn.dim() == 3
            _require(A_gu, torch.bfloat16, (A, r, H) if gu_shared else (A, E, r, H), "A_gu")
            _require(B_gu, torch.bfloat16, (A, E, 2 * I, r), "B_gu")
            _require(A_dn, torch.bfloat16, (A, E, r, I), "A_dn")
            _require(B_dn, torch.bfloat16, (A, H, r) if dn_shared else (A, E, H, r), "B_dn")
            self.gu = LoraFactors(A_gu.data_ptr(), B_gu.data_ptr(),
                                  r * H if gu_shared else E * r * H, 0 if gu_shared else r * H,
                                  E * 2 * I * r, 2 * I * r)
            self.dn = LoraFactors(A_dn.data_ptr(), B_dn.data_ptr(), E * r * I, r * I,
                                  H * r if dn_shared else E * H * r, 0 if dn_shared else H * r)
        else:
            self.num_adapters, self.rank = 0, 0
            self.gu = LoraFactors(None, None, 0, 0, 0, 0)
            self.dn = LoraFactors(None, None, 0, 0, 0, 0)
        self._ws = None
        self._ws_T = -1
        self._scales = None
        if adapter_scaling is not None:
            if len(adapter_scaling) != self.num_adapters:
                raise ValueError("adapter_scaling needs one value per adapter")
            self._scales = (ctypes.c_float * max(1, self.num_adapters))(*[float(v) for v in adapter_scaling])
        if max_tokens > 0:
            self.workspace(max_tokens)

    def workspace(self, T: int):
        torch = _torch()
        need = moe_lora_workspace_size_ex(T, self.H, self.I, self.E, self.top_k, self.num_adapters,
                                          self.rank, self.act_format)
        if need == 0:
            raise MoeError(MOE_ERR_SHAPE, "moe_lora_workspace_size")
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=self.w13.device)
        return self._ws

    def plan(self, T: int) -> WorkspacePlan:
        return moe_lora_workspace_plan(T, self.H, self.I, self.E, self.top_k, self.num_adapters,
                                       self.rank)

    def make_args(self, hidden, router_logits, token_lora_mapping, out, topk_ids=None, topk_w=None,
                  expanded_to_permuted=None, tile_n=0, wait_timeout_ms=0, stage_events=None,
                  debug_flags=0, tuning=None, side_stream=None, side_events=None):
        """``tuning``: a Tuning or a dict of its fields.  ``side_stream`` (a
        torch.cuda.Stream) with ``side_events`` (two torch.cuda.Event): the
        two-stream schedule of the gate_up LoRA shrink."""
        T = hidden.shape[0]
        ws = self.workspace(T)
        a = MoeLoraArgs()
        a.struct_size = ctypes.sizeof(MoeLoraArgs)
        a.T, a.H, a.I, a.E, a.top_k = T, self.H, self.I, self.E, self.top_k
        a.num_adapters, a.rank, a.scaling = self.num_adapters, self.rank, self.scaling
        a.hidden, a.w13, a.w2 = hidden.data_ptr(), self.w13.data_ptr(), self.w2.data_ptr()
        a.router_logits = router_logits.data_ptr()
        a.token_lora_mapping = _ptr(token_lora_mapping)
        a.gate_up, a.down = self.gu, self.dn
        a.out = out.data_ptr()
        a.topk_ids_out, a.topk_w_out = _ptr(topk_ids), _ptr(topk_w)
        a.expanded_to_permuted_out = _ptr(expanded_to_permuted)
        a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
        a.tile_n, a.wait_timeout_ms = int(tile_n), int(wait_timeout_ms)
        a.debug_flags = int(debug_flags)
        a.local_expert_offset, a.num_router_experts = self.local_expert_offset, self.num_router_experts
        a.activation_format = self.act_format
        if self.fp8:
            a.weight_format = MOE_WEIGHTS_FP8_E4M3_B128
            a.w13_scale, a.w2_scale = self.w13_scale.data_ptr(), self.w2_scale.data_ptr()
        a.adapter_scaling = ctypes.cast(self._scales, ctypes.c_void_p) if self._scales is not None else None
        if tuning is not None:
            a.tuning = tuning if isinstance(tuning, Tuning) else Tuning(**tuning)
        if side_stream is not None:
            if side_events is None or len(side_events) != 2:
                raise ValueError("side_stream needs two side_events")
            for e in side_events:        # torch creates the CUDA event on first record
                if not e.cuda_event:
                    e.record()
            a.side_stream = side_stream.cuda_stream
            a.side_events[0], a.side_events[1] = side_events[0].cuda_event, side_events[1].cuda_event
        self._events_keepalive = None
        if stage_events is not None:
            if len(stage_events) != MOE_NUM_STAGE_EVENTS:
                raise ValueError(f"stage_events needs {MOE_NUM_STAGE_EVENTS} events")
            for e in stage_events:       # torch creates the CUDA event on first record
                if not e.cuda_event:
                    e.record()
            arr = (ctypes.c_void_p * MOE_NUM_STAGE_EVENTS)(*[e.cuda_event for e in stage_events])
            self._events_keepalive = arr
            a.stage_events = ctypes.cast(arr, ctypes.c_void_p)
        return a

    def forward(self, hidden, router_logits, token_lora_mapping=None, out=None, topk_ids=None,
                topk_w=None, expanded_to_permuted=None, tile_n=0, wait_timeout_ms=0,
                stage_events: Optional[Sequence] = None, stream=None, debug_flags=0, tuning=None,
                side_stream=None, side_events=None):
        torch = _torch()
        T = hidden.shape[0]
        _require(hidden, torch.bfloat16, (T, self.H), "hidden")
        _require(router_logits, torch.float32, (T, self.num_router_experts), "router_logits")
        if token_lora_mapping is not None:
            _require(token_lora_mapping, torch.int32, (T,), "token_lora_mapping")
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.bfloat16, device=hidden.device)
        args = self.make_args(hidden, router_logits, token_lora_mapping, out, topk_ids, topk_w,
                              expanded_to_permuted, tile_n, wait_timeout_ms, stage_events,
                              debug_flags, tuning, side_stream, side_events)
        _check(moe_lora_forward(args, stream), "moe_lora_forward")
        return out

    def device_status(self, stream=None) -> int:
        return moe_read_device_status(self._ws, stream)
