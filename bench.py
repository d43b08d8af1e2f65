#!/usr/bin/env python
"""Benchmark of the routed BF16 MoE-LoRA layer forward (libmoelora, GB300).

One step = one ``moe_lora_forward`` call over one batch: routing, permute,
gate_up LoRA shrink, gate_up GEMM (+ LoRA expand, SwiGLU), down LoRA shrink,
down GEMM (+ LoRA expand), finalize.  Inputs are the seeded synthetic layer of
``workloads.py`` (default: decode_T16, T=16 tokens of a 30B-A3B-shaped layer,
H=2048, I=768, E=128, top-8, 4 adapters of rank 16), resident in HBM when the
timed region starts.  L2 is flushed (256 MiB write) before every step, outside
the step's events.

Prints one JSON line.  ``--impl reference`` times the CPU oracle instead.
Multi-GPU (torchrun): every rank runs an independent replica of the same
workload (the path has no cross-GPU exchange); value = all ranks' tokens /
the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import re
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-LoRA layer tokens/s at T=16/64/4096; % of HBM/tensor roofline"
DEFAULT_WORKLOAD = "decode_T16"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--tile-n", type=int, default=0)
    ap.add_argument("--weights", choices=["bf16", "fp8"], default="bf16",
                    help="expert weight format (fp8: e4m3 with 128x128 block scales)")
    ap.add_argument("--fp8-activations", action="store_true",
                    help="with --weights fp8: FP8 activations too (W8A8, per-token-group quant)")
    ap.add_argument("--only-workload", action="store_true",
                    help="measure --workload alone (default: also the metric's other batch shapes)")
    ap.add_argument("--shrink-in-gemm", choices=["auto", "off", "with-gather"], default="auto",
                    help="off: separate gather/shrink kernels (A/B of the in-GEMM shrink); "
                         "with-gather: the row gather inside the gate_up GEMM too")
    ap.add_argument("--side-stream", action="store_true",
                    help="two-stream schedule: gate_up LoRA shrink on a side stream")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-baseline-child", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help=argparse.SUPPRESS)
    return ap.parse_args()


# ---------------------------------------------------------------------------
# Algorithmic work of one forward (from the actual routing of the inputs)
# ---------------------------------------------------------------------------

def algorithmic_work(wl, ids, mapping, fp8=False, in_gemm_allowed=True, gemm_reads_hidden=False):
    """Bytes and FLOPs the forward must move / compute, intermediates excluded.

    Bytes: every touched expert's w13 and w2 once (fp8: one byte per weight
    plus one float32 scale per 128 x 128 block), every touched LoRA factor
    once (shared factors once per adapter), the hidden input, the output, the
    router logits and the mapping.  FLOPs: 2 per multiply-add of the two expert
    GEMMs for every (token, slot) and of the four LoRA products for adapted
    slots (the shared gate_up shrink once per token).

    Per expert GEMM the same rule: the weights and LoRA factors it reads, plus
    the layer input where it reads that itself (``gemm_reads_hidden``: the
    gate_up GEMM's in-kernel shrink reads the hidden rows, W8A8, or the row
    gather runs inside it); the permuted rows, the LoRA operands, the
    activation and the expert outputs are intermediates and are not charged.
    """
    T, H, I, E, k, A, r = wl.T, wl.H, wl.I, wl.E, wl.top_k, wl.num_adapters, wl.rank
    n = T * k
    experts = sorted(set(int(e) for e in ids.ravel()))
    lora = A > 0 and r > 0
    adapted = [(t, int(mapping[t])) for t in range(T) if lora and mapping[t] >= 0]
    pairs = sorted({(a, int(e)) for t, a in adapted for e in ids[t]})
    adapters = sorted({a for _, a in adapted})
    if fp8:
        nb = lambda x: (x + 127) // 128
        w13_b, w2_b = 2 * I * H + nb(2 * I) * nb(H) * 4, H * I + nb(H) * nb(I) * 4
    else:
        w13_b, w2_b = 2 * I * H * 2, H * I * 2
    gu_A = (len(adapters) if wl.shared_outer else len(pairs)) * r * H * 2
    gu_B = len(pairs) * 2 * I * r * 2
    dn_A = len(pairs) * r * I * 2
    dn_B = (len(adapters) if wl.shared_outer else len(pairs)) * H * r * 2
    io = T * H * 2 * 2 + T * E * 4 + T * 4
    n_ad = len(adapted) * k
    shrink_gu_rows = len(adapted) if wl.shared_outer else n_ad
    flops_gemm = n * 2 * (2 * I * H + H * I)
    flops_lora = 2 * r * (shrink_gu_rows * H + n_ad * 2 * I + n_ad * I + n_ad * H)
    work = {
        "distinct_experts": len(experts), "lora_pairs": len(pairs),
        "bytes": len(experts) * (w13_b + w2_b) + gu_A + gu_B + dn_A + dn_B + io,
        "flops": flops_gemm + flops_lora,
    }
    work["gemm_gate_up"] = {
        "bytes": len(experts) * w13_b + gu_B,
        "flops": n * 2 * 2 * I * H + n_ad * 2 * 2 * I * r,
    }
    work["gemm_down"] = {
        "bytes": len(experts) * w2_b + dn_B,
        "flops": n * 2 * H * I + n_ad * 2 * H * r,
    }
    if shrink_in_gemm(wl, fp8, in_gemm_allowed):
        # the GEMMs also run the LoRA shrinks (A factors; gate_up, where it
        # reads them itself, the hidden rows)
        work["gemm_gate_up"]["bytes"] += gu_A + (T * H * 2 if gemm_reads_hidden else 0)
        work["gemm_gate_up"]["flops"] += n_ad * 2 * r * H
        work["gemm_down"]["bytes"] += dn_A
        work["gemm_down"]["flops"] += n_ad * 2 * r * I
    return work


def auto_tile_n(n_rows, E):
    """The library's default token-tile width (api.cu, auto_tile_n)."""
    touched = max(1, min(E, n_rows))
    avg = -(-n_rows // touched)
    bn = 16
    while bn < 256 and bn < 2 * avg:
        bn *= 2
    while bn < 64 and bn < 4 * avg:
        bn *= 2
    return bn


def shrink_in_gemm(wl, fp8=False, allowed=True):
    """Whether the library runs the LoRA shrinks inside the expert GEMMs
    (api.cu: 16-wide tiles, so at most four rows per expert
    on average and never the row-block shrink; rank <= 32; per-expert gate_up
    A factors; the one-CTA permute; bf16 or FP8 weights alike)."""
    n, E = wl.T * wl.top_k, wl.E
    small = n <= 8192 and (((n + 1) & ~1) * 4 + 32 * E * 4 + (E + 1) * 4) <= 200 * 1024
    lora = wl.num_adapters > 0 and wl.rank > 0
    return (allowed and lora and small and auto_tile_n(n, E) == 16 and wl.rank <= 32 and
            not wl.shared_outer)


def kernels_per_forward(wl, fp8=False, in_gemm_allowed=True, two_streams=False, w8a8=False,
                        gather_in_gemm=False):
    """Kernels one moe_lora_forward launches (mirrors the library's choices):
    routing (unless fused into the one-CTA permute), the permute (one CTA, or
    count + scan + scatter), the gather/gate_up shrink and the down shrink
    (with the shrinks inside the GEMMs: the row gather alone, unless it runs
    inside the gate_up GEMM too; the two-stream schedule splits the first
    into a gather and a shrink), the gate_up GEMM, the down GEMM and the
    finalize."""
    n, E = wl.T * wl.top_k, wl.E
    small = n <= 8192 and (((n + 1) & ~1) * 4 + 32 * E * 4 + (E + 1) * 4) <= 200 * 1024
    fuse_route = small and wl.T <= 128
    # past the one-CTA permute: routing, count, scan + scatter (E <= 256,
    # top_k dividing 1024), else routing, count, scan, scatter
    chained = not small and E <= 256 and 1024 % wl.top_k == 0
    route_permute = 1 if small else (3 if chained else 4)
    lora = wl.num_adapters > 0 and wl.rank > 0
    two = two_streams and lora
    route_permute += 0 if (fuse_route or not small) else 1
    fuse_shrink = shrink_in_gemm(wl, fp8, in_gemm_allowed and not two)
    if w8a8:  # the row quant, the gate_up shrink, the activation quant, the down shrink
        sh = 1 if lora and not fuse_shrink else 0
        return route_permute + 1 + sh + 1 + 1 + sh + 1 + 1
    return (route_permute + (0 if fuse_shrink and gather_in_gemm else 1) + (1 if two else 0) + 1 +
            (1 if lora and not fuse_shrink else 0) + 1 + 1)


def max_over_ranks(value_ms, dist=None, device=None):
    """Largest per-rank time (ms) across the process group (identity without one)."""
    if dist is None:
        return float(value_ms)
    import torch
    t = torch.tensor([float(value_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_step, steps, world, total_ms_per_rank, dist=None, device=None):
    """Whole-job tokens/s of ``world`` replicas: every rank processes
    ``tokens_per_step`` tokens per step; the job takes as long as its slowest
    rank.  Returns (tokens_per_s, slowest_rank_total_ms)."""
    slowest = max_over_ranks(total_ms_per_rank, dist, device)
    return world * tokens_per_step * steps / (slowest / 1e3), slowest


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {k: float(pk[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def _code_only(text):
    """C++ source without its comments and blank lines (string literals in
    these files hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash(fp8_activations=False):
    """Hash of the code (comments left out) of the expert GEMM kernels: the
    bf16 / FP8-weight kernel (expert_gemm.cu), or with FP8 activations the
    W8A8 kernel (fp8_gemm.cu), with the headers both include."""
    h = hashlib.sha256()
    main = "fp8_gemm.cu" if fp8_activations else "expert_gemm.cu"
    for name in [main, "gemm_common.cuh", "ptx.cuh", "kernels.cuh"]:
        with open(os.path.join(ROOT, "moe_lora_expert_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def committed_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current source of that kernel; else None.  Workload tags ending in
    _w8a8 are the W8A8 kernels."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            doc = json.load(f)
    except Exception:
        return None
    ent = doc.get(kernel, {}).get(workload)
    if not ent or ent.get("kernel_source_sha") != kernel_source_hash(workload.endswith("_w8a8")):
        return None
    return ent.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# CPU oracle baseline (run in a fresh single-threaded interpreter)
# ---------------------------------------------------------------------------

def cpu_baseline_child(workload, seconds):
    import numpy as np
    import oracle
    import workloads
    wl = workloads.WORKLOADS[workload]
    inp = workloads.make_inputs(wl)
    tokens_done, elapsed, calls = 0, 0.0, 0
    stride = max(1, wl.T // 4)
    start_tok = 0
    while elapsed < seconds:
        toks = [(start_tok + i * stride) % wl.T for i in range(4)]
        t0 = time.perf_counter()
        oracle.forward_inputs(inp, tokens=toks)
        elapsed += time.perf_counter() - t0
        tokens_done += len(toks)
        calls += 1
        start_tok += 1
    print(json.dumps({"value": tokens_done / elapsed, "tokens": tokens_done, "seconds": elapsed,
                      "calls": calls}))


def run_cpu_baseline(workload, seconds):
    env = dict(os.environ)
    for v in ["OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"]:
        env[v] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    res = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-baseline-child",
                          "--workload", workload, "--cpu-seconds", str(seconds)],
                         capture_output=True, text=True, env=env, timeout=600)
    if res.returncode != 0:
        return {"error": res.stderr.strip().splitlines()[-1:] or ["failed"]}
    d = json.loads(res.stdout.strip().splitlines()[-1])
    return {"value": d["value"], "unit": "tokens/s", "cores": 1, "host_cores": os.cpu_count(),
            "kind": "oracle",
            "sample": (f"{d['tokens']} tokens of {workload} in {d['calls']} oracle calls of 4 tokens "
                       f"({d['seconds']:.1f} s, float64 numpy, 1 BLAS thread)")}


# ---------------------------------------------------------------------------
# Clock sampling
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi clocks polled every ``period_ms`` from before the first warm-up
    to after the last pass, each sample stamped with the host clock so that
    the samples inside a given window (the timed region) can be picked out."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index, period_ms=50):
        self.index = index
        self.period_ms = period_ms
        self.proc = None
        self.samples = []   # (host time, sm MHz, max MHz, power W, reasons)
        self._thread = None

    def start(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
        except Exception:
            self.proc = None
            return
        self._thread = threading.Thread(target=self._read, daemon=True)
        self._thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm, mx = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            try:
                pw = float(parts[2])
            except ValueError:
                pw = None
            reasons = {nm for nm, v in zip(self.NAMES, parts[4:8]) if v.lower().startswith("active")}
            self.samples.append((time.perf_counter(), sm, mx, pw, reasons))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=5)

    @staticmethod
    def summary(samples):
        if not samples:
            return {"samples": 0}
        sm = [x[1] for x in samples]
        pw = [x[3] for x in samples if x[3] is not None]
        reasons = set().union(*[x[4] for x in samples])
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(x[2] for x in samples),
                "sm_mhz_min": min(sm), "power_w_max": max(pw) if pw else None,
                "reasons": sorted(reasons), "samples": len(samples)}

    def window(self, t0, t1):
        return [x for x in self.samples if t0 <= x[0] <= t1]


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

# The metric's three batch shapes: T=16 (the headline), T=64 and T=4096.
METRIC_WORKLOADS = ["decode_T16", "decode_T64_mixed8", "prefill_T4096"]


def workload_config(wl, args, world):
    """The ``config`` object of both arms' JSON lines for workload ``wl``."""
    return {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E,
            "top_k": wl.top_k, "num_adapters": wl.num_adapters, "rank": wl.rank,
            "lora_scaling": wl.scaling, "shared_outer": wl.shared_outer,
            "tile_n": args.tile_n or "auto", "weights": args.weights,
            "activations": "fp8" if (args.fp8_activations and args.weights == "fp8") else "bf16",
            "l2": "GPU arm: flushed before every step (256 MiB write, outside the step events)",
            "parallelism": "replicas" if world > 1 else "single"}


def tuning_from_args(args):
    t = {}
    if args.shrink_in_gemm == "off":
        t["shrink_in_gemm"] = 1
    elif args.shrink_in_gemm == "with-gather":
        t["shrink_in_gemm"] = 2
    return t or None


class Layer:
    """One workload's layer on the GPU: weights, inputs, output buffers."""

    def __init__(self, name, args, dev):
        import numpy as np
        import torch

        import moe_lora_expert_gb300 as m
        import workloads
        self.wl = wl = workloads.WORKLOADS[name]
        self.inp = inp = workloads.make_inputs(wl)

        def bf16(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

        self.lora = inp.A_gu is not None
        self.fp8 = args.weights == "fp8"
        if self.fp8:
            q13, s13, q2, s2 = workloads.fp8_weights(inp)
            w13_d, w2_d = torch.from_numpy(q13).to(dev), torch.from_numpy(q2).to(dev)
            scales = dict(w13_scale=torch.from_numpy(s13).to(dev), w2_scale=torch.from_numpy(s2).to(dev))
        else:
            w13_d, w2_d, scales = bf16(inp.w13), bf16(inp.w2), {}
        lora = self.lora
        self.layer = m.MoeLoraLayer(w13_d, w2_d, wl.top_k,
                                    bf16(inp.A_gu) if lora else None, bf16(inp.B_gu) if lora else None,
                                    bf16(inp.A_dn) if lora else None, bf16(inp.B_dn) if lora else None,
                                    scaling=wl.scaling, max_tokens=wl.T,
                                    fp8_activations=bool(args.fp8_activations and self.fp8), **scales)
        self.hidden = bf16(inp.hidden)
        self.logits = torch.from_numpy(inp.logits).to(dev)
        self.mapping = torch.from_numpy(inp.mapping).to(dev) if lora else None
        self.out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=dev)
        self.ids = torch.empty((wl.T, wl.top_k), dtype=torch.int32, device=dev)
        self.tile_n = args.tile_n
        self.tuning = tuning_from_args(args)
        self.side = None
        self.in_gemm_allowed = args.shrink_in_gemm != "off" and not args.side_stream
        self.a8 = bool(args.fp8_activations and self.fp8)
        # the gate_up GEMM reads the hidden rows itself: W8A8's in-kernel
        # shrink, or the row gather inside the GEMM
        self.gemm_reads_hidden = self.a8 or args.shrink_in_gemm == "with-gather"
        if args.side_stream:
            self.side = (torch.cuda.Stream(device=dev), [torch.cuda.Event(), torch.cuda.Event()])

    def step(self, evs=None, hidden=None, logits=None, mapping=None):
        side = {} if self.side is None else {"side_stream": self.side[0], "side_events": self.side[1]}
        self.layer.forward(self.hidden if hidden is None else hidden,
                           self.logits if logits is None else logits,
                           self.mapping if mapping is None else mapping,
                           out=self.out, topk_ids=self.ids, tile_n=self.tile_n, stage_events=evs,
                           tuning=self.tuning, **side)


def time_steps(L, flush, steps, warmup, pg):
    """W untimed warm-ups, then ``steps`` forwards, each bracketed by one
    CUDA event pair on the launching stream (L2 flushed before each, outside
    the events), a barrier and a synchronize on both sides.  Returns
    (per-step ms, host start, host end)."""
    import torch
    import moe_lora_expert_gb300 as m
    for _ in range(warmup):
        flush.zero_()
        L.step()
    torch.cuda.synchronize()
    st = L.layer.device_status()
    if st != m.MOE_OK:
        raise SystemExit(f"{L.wl.name}: device status after warm-up: {m.status_string(st)}")
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    h0 = time.perf_counter()
    for i in range(steps):
        flush.zero_()
        ev0[i].record()
        L.step()
        ev1[i].record()
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    h1 = time.perf_counter()
    return [a.elapsed_time(b) for a, b in zip(ev0, ev1)], h0, h1


def stage_breakdown(L, flush, n):
    """A separate pass with events between the stages (they break the
    programmatic overlap of consecutive kernels, so it is not the timed
    pass): per-stage CUDA-event times, one list per forward."""
    import torch
    import moe_lora_expert_gb300 as m
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(m.MOE_NUM_STAGE_EVENTS)]
              for _ in range(n)]
    for i in range(n):
        flush.zero_()
        L.step(events[i])
    torch.cuda.synchronize()
    return [[ev[j].elapsed_time(ev[j + 1]) for j in range(m.MOE_NUM_STAGE_EVENTS - 1)] for ev in events]


def rooflines(L, ms_per_step, stage_ms, peaks, peak_src, workload_tag):
    """The dominant expert GEMM's roofline (its CUDA-event time in the stage
    pass) and the whole forward's (max of bytes / HBM and FLOPs / bf16 peak)."""
    import moe_lora_expert_gb300 as m
    wl = L.wl
    ids_np = L.ids.cpu().numpy()
    work = algorithmic_work(wl, ids_np, L.inp.mapping, fp8=L.fp8, in_gemm_allowed=L.in_gemm_allowed,
                            gemm_reads_hidden=L.gemm_reads_hidden)
    med = [statistics.median(s[j] for s in stage_ms) for j in range(len(m.STAGE_NAMES))]
    stages_us = {nm: round(v * 1e3, 2) for nm, v in zip(m.STAGE_NAMES, med)}
    top = "gemm_gate_up" if med[3] >= med[5] else "gemm_down"
    kt_ms = statistics.mean(s[3 if top == "gemm_gate_up" else 5] for s in stage_ms)
    kw = work[top]
    t_bytes = kw["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_flops = kw["flops"] / (peaks["bf16_tflops"] * 1e12)
    if t_bytes >= t_flops:
        achieved = kw["bytes"] / (kt_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4)}
    else:
        achieved = kw["flops"] / (kt_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4)}
    roof.update({"traffic": committed_traffic(top, workload_tag), "kernel": top,
                 "kernel_us": round(kt_ms * 1e3, 2), "algorithmic_bytes": kw["bytes"],
                 "algorithmic_flops": kw["flops"],
                 "frac_of_max_roof": round(max(t_bytes, t_flops) / (kt_ms / 1e3), 4),
                 "peak_source": "of measured (MEASURED_PEAKS.json)" if peak_src == "measured"
                 else "of fallback"})
    tb = work["bytes"] / (peaks["hbm_gbs"] * 1e9)
    tf = work["flops"] / (peaks["bf16_tflops"] * 1e12)
    t_roof = max(tb, tf)
    fwd = {"bound": "hbm" if tb >= tf else "tensor", "t_roof_us": round(t_roof * 1e6, 2),
           "t_us": round(ms_per_step * 1e3, 2), "frac": round(t_roof / (ms_per_step / 1e3), 4),
           "bytes": work["bytes"], "flops": work["flops"],
           "distinct_experts": work["distinct_experts"], "lora_pairs": work["lora_pairs"]}
    return roof, fwd, stages_us


def run_ours(args):
    import torch

    import moe_lora_expert_gb300 as m

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = run_cpu_baseline(args.workload, args.cpu_seconds)

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    visible = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids_vis = [v.strip() for v in visible.split(",") if v.strip()]
    clocks = ClockSampler(ids_vis[local] if local < len(ids_vis) else local)
    clocks.start()

    L = Layer(args.workload, args, dev)
    wl = L.wl
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    peaks, peak_src = load_peaks()
    fp8 = L.fp8
    tag = lambda name: name + ("_w8a8" if fp8 and args.fp8_activations else "_fp8" if fp8 else "")
    run0 = time.perf_counter()

    step_ms, h0, h1 = time_steps(L, flush, args.steps, args.warmup, pg)
    stage_ms = stage_breakdown(L, flush, max(3, min(args.steps, 30)))
    value, total_ms = job_throughput(wl.T, args.steps, world, sum(step_ms), pg, dev)
    ms_per_step = total_ms / args.steps

    # ---------------- e2e: host buffers, copies inside the timed region
    lora = L.lora
    h_hidden = L.hidden.cpu().pin_memory()
    h_logits = L.logits.cpu().pin_memory()
    h_mapping = L.mapping.cpu().pin_memory() if lora else None
    h_out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16).pin_memory()
    d_hidden, d_logits = torch.empty_like(L.hidden), torch.empty_like(L.logits)
    d_mapping = torch.empty_like(L.mapping) if lora else None

    def e2e_step():
        d_hidden.copy_(h_hidden, non_blocking=True)
        d_logits.copy_(h_logits, non_blocking=True)
        if lora:
            d_mapping.copy_(h_mapping, non_blocking=True)
        L.step(hidden=d_hidden, logits=d_logits, mapping=d_mapping)
        h_out.copy_(L.out, non_blocking=True)

    e2e_steps = max(1, min(args.steps, 200))
    e_ms = 0.0
    for i in range(args.warmup + e2e_steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        e2e_step()
        e1.record()
        e1.synchronize()
        if i >= args.warmup:
            e_ms += e0.elapsed_time(e1)
    e_ms = max_over_ranks(e_ms, pg, dev)
    h2d = wl.T * wl.H * 2 + wl.T * wl.E * 4 + (wl.T * 4 if lora else 0)
    e2e = {"value": world * wl.T * e2e_steps / (e_ms / 1e3), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": wl.T * wl.H * 2}

    # ---------------- the same steps replayed from CUDA graphs: the forward
    # alone, and the whole host-to-host step (copies + forward + copy back)
    def replay_ms(g, n):
        total = 0.0
        for i in range(args.warmup + n):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            e1.synchronize()
            if i >= args.warmup:
                total += e0.elapsed_time(e1)
        return total

    g_fwd, g_e2e = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g_fwd):
        L.step()
    with torch.cuda.graph(g_e2e):
        e2e_step()
    torch.cuda.synchronize()
    gf_ms = max_over_ranks(replay_ms(g_fwd, e2e_steps), pg, dev)
    ge_ms = max_over_ranks(replay_ms(g_e2e, e2e_steps), pg, dev)
    st = L.layer.device_status()
    if st != m.MOE_OK:
        raise SystemExit(f"device status after graph replays: {m.status_string(st)}")
    graph = {"forward_us_per_step": round(gf_ms / e2e_steps * 1e3, 2),
             "forward_value": round(world * wl.T * e2e_steps / (gf_ms / 1e3), 1),
             "e2e_value": round(world * wl.T * e2e_steps / (ge_ms / 1e3), 1), "unit": "tokens/s",
             "note": "one CUDA graph per step, replayed; e2e_value includes the host copies"}
    roof, fwd, stages_us = rooflines(L, ms_per_step, stage_ms, peaks, peak_src, tag(wl.name))
    n_kernels = kernels_per_forward(wl, fp8, args.shrink_in_gemm != "off", args.side_stream,
                                    bool(fp8 and args.fp8_activations), args.shrink_in_gemm == "with-gather")
    del L, h_hidden, h_logits, h_mapping, d_hidden, d_logits, d_mapping, g_fwd, g_e2e

    # ---------------- the metric's other batch shapes (T=64, T=4096): the
    # same timing (steps, warm-ups, L2 flush), rooflines from their own routing
    others = {}
    if not args.only_workload:
        for name in METRIC_WORKLOADS:
            if name == wl.name:
                continue
            Lo = Layer(name, args, dev)
            o_ms, _, _ = time_steps(Lo, flush, args.steps, args.warmup, pg)
            o_stage = stage_breakdown(Lo, flush, max(3, min(args.steps, 30)))
            o_value, o_total = job_throughput(Lo.wl.T, args.steps, world, sum(o_ms), pg, dev)
            o_roof, o_fwd, o_stages = rooflines(Lo, o_total / args.steps, o_stage, peaks, peak_src,
                                                tag(name))
            others[name] = {"value": round(o_value, 1), "unit": "tokens/s",
                            "ms_per_step": round(o_total / args.steps, 5),
                            "config": workload_config(Lo.wl, args, world),
                            "roofline": o_roof, "forward_roofline": o_fwd, "stages_us": o_stages}
            del Lo
            torch.cuda.empty_cache()
    run1 = time.perf_counter()
    clocks.stop()

    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return

    timed = ClockSampler.summary(clocks.window(h0, h1))
    clk = ClockSampler.summary(clocks.window(run0, run1))
    clk["timed_region_samples"] = timed.get("samples", 0)
    clk["window"] = ("nvidia-smi every 50 ms from the first warm-up of the headline workload to the "
                     "end of the last workload's passes (timed regions, stage passes, e2e, graphs)")
    if "sm_mhz" in clk:
        clk["us_x_mhz"] = round(ms_per_step * 1e3 * clk["sm_mhz"], 1)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("fp8 e4m3 x e4m3 (W8A8; bf16 LoRA, fp32 accumulate)" if fp8 and args.fp8_activations
                  else "bf16 (fp8 e4m3 expert weights, dequantized to bf16)" if fp8 else "bf16"),
        "data": "synthetic (seeded normal inputs and weights; no trained weights)",
        "config": workload_config(wl, args, world),
        "roofline": roof, "forward_roofline": fwd, "stages_us": stages_us,
        "cpu_baseline": cpu, "e2e": e2e, "graph": graph, "gpu_launches": n_kernels * args.steps,
        "clocks": clk, "wall_s_timed_region": round(h1 - h0, 4),
        "workloads": others,
    }
    if args.side_stream:
        line["schedule"] = "two streams: gate_up LoRA shrink on a side stream, joined before the gate_up GEMM"
    print(json.dumps(line))
    if pg:
        pg.destroy_process_group()


# ---------------------------------------------------------------------------
# Reference arm: the CPU oracle as it stands
# ---------------------------------------------------------------------------

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import oracle
    import workloads
    wl = workloads.WORKLOADS[args.workload]
    inp = workloads.make_inputs(wl)
    threads = 1
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        threads = max([d.get("num_threads", 1) for d in info] + [1])
    except Exception:
        threads = os.cpu_count() or 1
    t = 0.0
    tokens = 0
    for i in range(args.warmup + args.steps):
        tok = [i % wl.T]
        t0 = time.perf_counter()
        oracle.forward_inputs(inp, tokens=tok)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            t += dt
            tokens += len(tok)
    value = tokens / t
    sample = (f"1 token of {wl.name} per step (float64 numpy oracle, BLAS pool of {threads} "
              f"threads on a host with {os.cpu_count()} cores)")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded normal inputs and weights; no trained weights)",
            "config": workload_config(wl, args, world),
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": threads,
                             "host_cores": os.cpu_count(), "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    args = parse_args()
    if args.cpu_baseline_child:
        cpu_baseline_child(args.workload, args.cpu_seconds)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
