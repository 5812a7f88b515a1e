#!/usr/bin/env python
"""Throughput of the dropless MoE layer (forward + backward) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config pangu_bf16] [--no-cpu-baseline]

One step = the whole hot path over one batch: router scores, fused top-k, permutation,
grouped SwiGLU forward, combine, and the backward (dY permutation, expert dX chain, score
gradient, dX combine, expert dW products, router dW), through moe_layer_fwd/moe_layer_bwd.
The default workload is the Pangu-Ultra-MoE-shaped layer (T=8192, d=7680, 256 routed
experts, top-8, f=2048, 1 shared expert, Zipf(0.8) routing skew), synthetic and seeded.

N > 1 (torchrun, one process per GPU): every rank runs its own replica of the step
(weak scaling, no data-path collective); value = tokens processed by all ranks / the
slowest rank's time.  Rank 0 prints one JSON line.

--impl reference times the fp64 CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s fwd+bwd"
UNIT = "tokens/s"

# DRAM traffic per launch from an ncu capture of the dominant kernel, keyed by the phase
# name; valid only while the kernel source still hashes to src_sha256.
NCU_TRAFFIC = {
    # ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum on the small case T=1024, E=32
    # (33 gradient groups, 9216 token-copy rows), one launch after warm-up, scaled to the full
    # workload by the units each term grows with: reads by the token-copy rows (73728 / 9216),
    # writes by the gradient groups (257 / 33). Small case: 217.6 MB read, 2018.9 MB
    # written; scaled: 1741.0 MB + 15723.2 MB. See profiles/gemm_dw13_pangu_bf16.md.
    # Applies only while the kernel's source file is unchanged since the capture.
    "gemm_dw13": {"src": "gemm_tc_pair.cu", "workload": "pangu_bf16",
                  "bytes_per_launch": 1741023232 + 15723167542,
                  "src_sha256": "d4145c7d9898e288cc3eb2b62baa12a1b453960ea9c48e6a6abb6d93bee45e33"},
}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def _sha(path):
    return hashlib.sha256(open(path, "rb").read()).hexdigest()


# --------------------------------------------------------------------------- accounting
def algorithmic_work(cfg):
    """Per-launch algorithmic FLOPs (tensor phases) or bytes (memory phases) of each phase."""
    T, d, E, k, f, S, fs = (cfg[n] for n in ("T", "d", "E", "k", "f", "S", "f_s"))
    es = 4 if cfg["dtype"] == "f32" else 2
    Tk = T * k
    rows_f = Tk * f + S * T * fs          # sum over groups of rows x width
    flops = {
        "gemm_fwd1": 4.0 * d * rows_f, "gemm_fwd2": 2.0 * d * rows_f,
        "gemm_bwd2t": 2.0 * d * rows_f, "gemm_bwd1t": 4.0 * d * rows_f,
        "gemm_dw2": 2.0 * d * rows_f, "gemm_dw13": 4.0 * d * rows_f,
        "router_gemm": 2.0 * T * d * E,
    }
    bytes_ = {
        "route_topk": 4.0 * T * E + 4.0 * E + 8.0 * Tk,
        "permute_hist": 4.0 * Tk + 4.0 * Tk + 8.0 * E * ((T + 63) // 64),
        "permute_scatter": (1 + k) * T * d * es + 24.0 * Tk,
        "permute_rows": (1 + k) * T * d * es + 4.0 * Tk,
        "combine": (k + 2 if S else k + 1) * T * d * es + 8.0 * Tk,
        "combine_bwd": (k + 2 if S else k + 1) * T * d * es + 8.0 * Tk + 8.0 * Tk,
        "route_bwd": 16.0 * Tk + 4.0 * T * E,
        "dwr": Tk * d * es + 8.0 * Tk + 4.0 * 8 * E * d,
    }
    return flops, bytes_


def executed_rows(c):
    """Rows the token-row products multiply for a group of c rows: 128-row M tiles, the last
    one a 64-row tile when at most 64 rows are left."""
    q, r = divmod(int(c), 128)
    return q * 128 + (0 if r == 0 else 64 if r <= 64 else 128)


def group_roofline(cfg, counts, peaks):
    """Per-group roofline of each grouped product: the sum over groups (the routed experts
    with their n_e token copies, then the shared experts over all T tokens) of
    max(flops_g / P, bytes_g / BW), in ms. A group below the ridge (n_e < P / BW in
    flop per weight byte) is bound by streaming its weight (or, for the dW products,
    writing its gradient) once; a group above it by the tensor cores. bytes_g counts the
    weight (or gradient) of the group once plus its activation rows read and written."""
    d, f, fs, S, T = cfg["d"], cfg["f"], cfg["f_s"], cfg["S"], cfg["T"]
    es = 4 if cfg["dtype"] == "f32" else 2
    P = peaks["bf16_tflops_sustained"] * 1e12
    BW = peaks["hbm_gbs"] * 1e9
    groups = [(n, f) for n in counts] + [(T, fs)] * S

    def work(phase, n, w):
        wgt = d * w * es                       # one of the three d x w matrices
        if phase == "gemm_fwd1":               # x rows -> Z [n, 2w], h [n, w]
            return 4.0 * d * w * n, 2 * wgt + es * n * (d + 3 * w)
        if phase == "gemm_fwd2":               # h -> y_perm
            return 2.0 * d * w * n, wgt + es * n * (w + d)
        if phase == "gemm_bwd2t":              # dY rows, Z -> dz [n, 2w], hw [n, w], dgate
            return 2.0 * d * w * n, wgt + es * n * (d + 5 * w) + 4 * n
        if phase == "gemm_bwd1t":              # dz -> dx_perm
            return 4.0 * d * w * n, 2 * wgt + es * n * (2 * w + d)
        if phase == "gemm_dw2":                # dY rows, hw -> dW2 written
            return 2.0 * d * w * n, wgt + es * n * (d + w)
        if phase == "gemm_dw13":               # dz, x rows -> dW13 written
            return 4.0 * d * w * n, 2 * wgt + es * n * (2 * w + d)
        raise KeyError(phase)

    out = {}
    for phase in ("gemm_fwd1", "gemm_fwd2", "gemm_bwd2t", "gemm_bwd1t", "gemm_dw2", "gemm_dw13"):
        per_group = 0.0
        fl = by = 0.0
        for n, w in groups:
            a, b = work(phase, n, w)
            per_group += max(a / P, b / BW)
            fl += a
            by += b
        # the looser bound of the whole launch, every group overlapped with every other
        out[phase] = {"per_group_ms": per_group * 1e3, "whole_launch_ms": max(fl / P, by / BW) * 1e3,
                      "bytes": by}
    return out


def dw_write_bytes(cfg):
    """Bytes of dW written per launch by the two dW products (bf16 or fp32 gradients)."""
    es = 4 if cfg["dtype"] == "f32" else 2
    w13 = 2 * cfg["f"] * cfg["d"] * cfg["E"] + 2 * cfg["f_s"] * cfg["d"] * cfg["S"]
    return {"gemm_dw13": es * w13, "gemm_dw2": es * w13 // 2}


# --------------------------------------------------------------------------- multi-rank
def reduce_max(value: float, device=None) -> float:
    """Max of a float over all ranks (identity without an initialised process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput(world: int, steps: int, tokens_per_step: int, t_max_ms: float) -> float:
    """Whole-job tokens/s: every rank processes its own batch (weak scaling)."""
    return world * steps * tokens_per_step / (t_max_ms / 1e3)


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.th.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- oracle arm
def oracle_scale(cfg):
    """Scale-down factor of the oracle's sample: T / s tokens routed among E / s experts (every
    s-th expert), so that every expert keeps the workload's mean segment of T*k/E copies and
    every token the workload's work (k routed copies at the full d and f, plus the shared
    experts). s is the largest power of two up to 16 that leaves at least 2k experts."""
    s = 16
    while s > 1 and cfg["E"] // s < 2 * cfg["k"]:
        s //= 2
    return s


def oracle_sample(w, logits32, scale):
    """Time the fp64 oracle's forward + backward (layer_forward + layer_backward, as they stand)
    on a sub-layer of the workload: its first T/scale tokens routed (top-k, renormalised) among
    every scale-th expert, with the full d, f and shared experts. The routing is taken from the
    device's fp32 scores restricted to those experts. Returns (seconds, tokens, experts)."""
    import numpy as np
    import torch
    import oracle as O
    c = w.cfg
    Ts, cols = c["T"] // scale, np.arange(0, c["E"], scale)
    bias = None if w.bias is None else w.bias.cpu().numpy()[cols]
    idx, gate = O.route_topk(O.selection_scores(np.ascontiguousarray(logits32[:Ts][:, cols]), bias), c["k"])
    sel = torch.as_tensor(cols).to(w.w13.device)

    def f64(t):     # exact upcast on the tensor's own device, then to host memory
        return None if t is None else t.double().cpu().numpy()
    x, dy = f64(w.x[:Ts]), f64(w.dy[:Ts])
    w13, w2 = f64(w.w13[sel]), f64(w.w2[sel])
    ws13, ws2 = f64(w.ws13), f64(w.ws2)
    w_r = None if w.w_r is None else f64(w.w_r[:, sel])
    t0 = time.perf_counter()
    fwd = O.layer_forward(x, idx, gate, w13, w2, ws13, ws2)
    O.layer_backward(x, idx, gate, fwd, dy, w13, w2, ws13, ws2, w_r=w_r)
    return time.perf_counter() - t0, Ts, len(cols)


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count()


def sample_text(cfg, scale, Ts, Es):
    return (f"fp64 oracle (layer_forward + layer_backward) on a 1/{scale} sub-layer of the workload: "
            f"its first {Ts} tokens routed top-{cfg['k']} among {Es} of its {cfg['E']} experts "
            f"(every {scale}th), {Ts * cfg['k'] // Es} copies per expert on average as in the full "
            f"layer, full d={cfg['d']}, f={cfg['f']} and {cfg['S']} shared expert(s); the per-token "
            f"work equals the full layer's, so tokens/s is the oracle's rate on this workload")


def cpu_baseline(w, logits32, min_seconds=10.0):
    """The oracle's tokens/s: the sub-layer sample repeated until about min_seconds of CPU work."""
    scale = oracle_scale(w.cfg)
    tot, toks, runs = 0.0, 0, 0
    while tot < min_seconds or runs == 0:
        dt, Ts, Es = oracle_sample(w, logits32, scale)
        tot, toks, runs = tot + dt, toks + Ts, runs + 1
    return {"value": toks / tot, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "sample": sample_text(w.cfg, scale, Ts, Es) + f"; {runs} run(s), {tot:.1f} s"}


# --------------------------------------------------------------------------- layer variants
def time_variant(params, cfg, w, args, stream, **kw):
    """ms per fwd+bwd step of a layer variant (MoELayer keyword arguments), timed like the
    main step on the same workload, this rank only."""
    import torch
    from dropless_token_routing_gb300.api import MoELayer, get_device_error
    T, k, E = cfg["T"], cfg["k"], cfg["E"]
    lay = MoELayer(params, T, cfg["d"], E, k, cfg["f"], cfg["S"], cfg["f_s"], w.torch_dtype,
                   device=w.x.device, logits_input=w.logits_in is not None, **kw)
    lay.alloc_grads()

    def step():
        lay.forward(w.x, w.logits_in)
        lay.backward(w.dy)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    if get_device_error(lay.ws) != 0:
        raise RuntimeError(f"device error in the {kw} run")
    ms = a.elapsed_time(b) / args.steps
    del lay
    torch.cuda.empty_cache()
    return ms


def drop_and_pad(factors, params, cfg, w, counts, args, stream):
    """The comparison the pages draw: the same layer step in the drop-and-pad variant, every
    expert given C = ceil(cf * T * k / E) rows (overflow copies dropped, short experts
    padded)."""
    import math
    T, k, E = cfg["T"], cfg["k"], cfg["E"]
    out = []
    for cf in factors:
        C = max(1, math.ceil(cf * T * k / E))
        ms = time_variant(params, cfg, w, args, stream, capacity=C)
        kept = sum(min(c, C) for c in counts)
        out.append({"capacity_factor": cf, "capacity": C, "value": round(T / (ms / 1e3), 1),
                    "unit": UNIT, "ms_per_step": round(ms, 3),
                    "dropped_copy_fraction": round(1 - kept / (T * k), 4),
                    "padding_row_fraction": round(1 - kept / (E * C), 4)})
    return out


def fused_rearrange(params, cfg, w, args, stream):
    """The rearrangement fused into the expert GEMMs' operand loads (row gathers from x and
    dy, no rearranged copies) instead of the copies the default step makes; and the
    un-rearrangement fused into the second expert GEMM's stores (token-major rows, so the
    combine reads each token's rows as one block), alone and with the gathers."""
    out = {}
    for key, r in (("gather", 1), ("scatter", 2), ("gather_and_scatter", 3)):
        ms = time_variant(params, cfg, w, args, stream, rearrange=r, recompute=bool(r & 1))
        out[key] = {"value": round(cfg["T"] / (ms / 1e3), 1), "unit": UNIT, "ms_per_step": round(ms, 3)}
    # the gather variant's figures stay at the top level, as before
    return dict(out["gather"], variants=out)


def balance_statistics(cfg, w, logits, ws, stream, peaks, reps=50):
    """Routing with the micro-batch balance statistics: the top-k call and the statistics call
    one after the other, against the single call that takes both from one read of the scores.
    Each variant's `reps` calls are captured in a CUDA graph and replayed, so that the device
    time is measured rather than the host's call rate; the scores stay in L2 between
    repetitions, as in the step, where the router writes them just before."""
    import torch
    from dropless_token_routing_gb300 import api as A
    T, E, k = cfg["T"], cfg["E"], cfg["k"]
    dev = logits.device
    idx = torch.empty(T, k, dtype=torch.int32, device=dev)
    gw = torch.empty(T, k, device=dev)
    cnt = torch.empty(E, dtype=torch.int32, device=dev)
    P = torch.empty(E, device=dev)
    aux = torch.empty(1, device=dev)
    alpha = 1e-2
    runs = {
        "topk_only": lambda: A.route_topk(logits, w.bias, k, idx, gw, cnt, ws),
        "topk_then_balance": lambda: (A.route_topk(logits, w.bias, k, idx, gw, cnt, ws),
                                      A.route_balance(logits, w.bias, cnt, k, alpha, P, aux, ws)),
        "fused": lambda: A.route_topk_balance(logits, w.bias, k, alpha, idx, gw, cnt, P, aux, ws),
    }
    out = {}
    for name, fn in runs.items():
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(reps):
                fn()
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        out[name] = {"us": round(a.elapsed_time(b) / reps * 1e3, 2)}
        del g
    # bytes of the fused call: the scores once, gates and indices out, the partial rows
    nbytes = T * E * 4 + T * k * 8 + min(512, (T + 7) // 8) * E * 4 * 2
    us = out["fused"]["us"]
    out["fused"].update({"bytes": nbytes, "GB/s": round(nbytes / (us * 1e-6) / 1e9, 1),
                         "frac_hbm": round(nbytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 3)})
    return out


# --------------------------------------------------------------------------- summaries
def summarize(cfg, trace, steps, counts, peaks):
    """Per-kernel table, grouped-GEMM totals and routing statistics of a traced run of
    `steps` layer steps (trace: phase -> (launches, total ms))."""
    flops, bytes_ = algorithmic_work(cfg)
    total_ms = sum(v[1] for v in trace.values())
    kernels = {}
    for name, (launches, ms) in sorted(trace.items(), key=lambda kv: -kv[1][1]):
        # every phase is one operation per step, possibly of several launches (the dW_r
        # partial sums and their reduction; the router's weight split and its GEMM), so
        # the operation's work is divided by the phase's time per step
        per = ms / launches
        per_step = ms / steps
        ent = {"launches_per_step": launches / steps, "ms_per_launch": round(per, 4),
               "ms_per_step": round(per_step, 4),
               "share": round(ms / total_ms, 4) if total_ms else None}
        if name in flops and name != "router_gemm":
            ach = flops[name] / (per_step / 1e3) / 1e12
            ent.update(achieved=round(ach, 1), unit="TFLOP/s",
                       frac=round(ach / peaks["bf16_tflops_sustained"], 3))
        elif name in bytes_:
            ach = bytes_[name] / (per_step / 1e3) / 1e9
            ent.update(achieved=round(ach, 1), unit="GB/s", frac=round(ach / peaks["hbm_gbs"], 3))
        elif name == "router_gemm":
            if cfg["dtype"] == "f32":
                ent.update(achieved=round(flops[name] / (per_step / 1e3) / 1e12, 2),
                           unit="TFLOP/s (fp32 FMA)")
            else:   # three bf16 parts of the fp32 weight, each a full product on the tensor cores
                ent.update(achieved=round(3 * flops[name] / (per_step / 1e3) / 1e12, 1),
                           unit="TFLOP/s (bf16, 3-part weight split, executed)")
        kernels[name] = ent
    groof = group_roofline(cfg, counts, peaks)
    for name, g in groof.items():
        if name in kernels:
            ms = kernels[name]["ms_per_step"]
            kernels[name]["group_roofline"] = {
                "per_group_ms": round(g["per_group_ms"], 4), "frac": round(g["per_group_ms"] / ms, 3),
                "whole_launch_ms": round(g["whole_launch_ms"], 4),
                "frac_whole_launch": round(g["whole_launch_ms"] / ms, 3)}
    # the dominant kernel: the phase with the most time among those with algorithmic work
    # (the router GEMM aside, whose executed FLOPs are three times its algorithmic ones)
    ranked = [kv for kv in trace.items() if (kv[0] in flops and kv[0] != "router_gemm") or kv[0] in bytes_]
    dom = max(ranked or trace.items(), key=lambda kv: kv[1][1])[0]
    gemm_names = [k_ for k_ in trace if k_.startswith("gemm")]
    gemm_flops = sum(flops[k_] for k_ in gemm_names)
    gemm_ms = sum(trace[k_][1] for k_ in gemm_names) / steps
    groof_ms = sum(g["per_group_ms"] for n_, g in groof.items() if n_ in trace)
    tf = gemm_flops / (gemm_ms / 1e3) / 1e12 if gemm_ms else 0.0
    T = cfg["T"]
    rows = sum(counts) + cfg["S"] * T
    padded = sum(-(-c // 128) * 128 for c in counts) + cfg["S"] * (-(-T // 128) * 128)
    executed = sum(executed_rows(c) for c in counts) + cfg["S"] * executed_rows(T)
    return {
        "kernels": kernels, "dominant": dom, "launches": sum(v[0] for v in trace.values()),
        "grouped_gemm": {"tflops": round(tf, 1),
                         "frac_of_dense_peak": round(tf / peaks["bf16_tflops_sustained"], 3),
                         "frac_of_burst_peak": round(tf / peaks["bf16_tflops"], 3),
                         "peak_kind": f"useful FLOPs; dense bf16 sustained / burst ({peaks['source']})",
                         "per_group_roofline_ms": round(groof_ms, 3),
                         "frac_of_per_group_roofline": round(groof_ms / gemm_ms, 3) if gemm_ms else None},
        "routing": {"max_expert_rows": max(counts), "empty_experts": sum(1 for c in counts if c == 0),
                    "m_tile_fill": round(rows / executed, 4) if executed else None,
                    "m_tile_fill_128": round(rows / padded, 4) if padded else None}}


def other_workload(name, args, dev, peaks, steps=10):
    """Time another workload the same way as the main one (fwd + bwd on device-resident
    inputs, `steps` steps after the warm-up, per-kernel CUDA-event trace). A workload whose
    recipe is forward-only (the mid-size one) is also timed forward-only."""
    import torch
    from dropless_token_routing_gb300 import _native as N
    from dropless_token_routing_gb300.api import LayerParams, MoELayer, get_device_error
    from synth import CONFIGS, make_workload
    cfg = dict(CONFIGS[name], name=name)
    T = cfg["T"]
    w = make_workload(cfg, device=dev)
    params = LayerParams(w13=w.w13, w2=w.w2, w_r=w.w_r, bias=w.bias, ws13=w.ws13, ws2=w.ws2)
    layer = MoELayer(params, T, cfg["d"], cfg["E"], cfg["k"], cfg["f"], cfg["S"], cfg["f_s"],
                     w.torch_dtype, device=dev, logits_input=w.logits_in is not None)
    layer.alloc_grads()
    stream = torch.cuda.current_stream()

    def run(n, bwd=True):
        for _ in range(n):
            layer.forward(w.x, w.logits_in)
            if bwd:
                layer.backward(w.dy)

    run(args.warmup)
    torch.cuda.synchronize()
    N.trace_enable(True)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    run(steps)
    b.record(stream)
    torch.cuda.synchronize()
    trace = N.trace_read()
    N.trace_enable(False)
    ms = a.elapsed_time(b) / steps
    out = {"workload": f"T={T} d={cfg['d']} E={cfg['E']} top-{cfg['k']} f={cfg['f']} S={cfg['S']} "
                       f"f_s={cfg['f_s']} routing={cfg['routing']}"
                       + (f"(s={cfg['zipf_s']})" if cfg["routing"] == "zipf" else ""),
           "steps": steps, "ms_per_step": round(ms, 3), "value": round(T / (ms / 1e3), 1), "unit": UNIT}
    if not cfg["bwd"]:     # the recipe itself is forward-only
        c, d_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c.record(stream)
        run(steps, bwd=False)
        d_.record(stream)
        torch.cuda.synchronize()
        fms = c.elapsed_time(d_) / steps
        out["forward_only"] = {"ms_per_step": round(fms, 3), "value": round(T / (fms / 1e3), 1),
                               "unit": "tokens/s forward"}
    if get_device_error(layer.ws) != 0:
        raise RuntimeError(f"device error in the {name} run")
    summ = summarize(cfg, trace, steps, layer.saved["counts"].cpu().tolist(), peaks)
    out.update(grouped_gemm=summ["grouped_gemm"], routing=summ["routing"])
    keep = ("permute_scatter", "permute_rows", "combine", "combine_bwd")
    out["hbm_frac"] = {k_: summ["kernels"][k_]["frac"] for k_ in keep if k_ in summ["kernels"]}
    out["gemm_frac"] = {k_: summ["kernels"][k_]["frac"] for k_ in summ["kernels"] if k_.startswith("gemm")}
    del layer, params, w
    torch.cuda.empty_cache()
    return out


# --------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="pangu_bf16")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--shrink", default="", help="smaller case of the same recipe, e.g. T=512,E=16 "
                                                  "(for profiler captures; not a bench line)")
    ap.add_argument("--rearrange", default="copy", choices=["copy", "gather", "scatter", "both"],
                    help="the timed step's rearrangement: rearranged copies (default), row gathers "
                         "fused into the expert GEMMs (with selective recompute), the second GEMM "
                         "writing token-major rows for the combine, or both")
    ap.add_argument("--no-balance-statistics", dest="balance_statistics", action="store_false",
                    help="skip the timing of the routing forms with balance statistics")
    ap.add_argument("--no-fused-rearrange", dest="fused_rearrange", action="store_false",
                    help="skip the timing of the fused-rearrangement variant (rank 0, after the "
                         "main measurement)")
    ap.add_argument("--other-workloads", default="dsv3_bf16,adversarial_bf16,mid_bf16",
                    help="further workloads timed after the main one (rank 0, 10 steps each; empty "
                         "to skip); each gets its own entry in the line's other_workloads")
    ap.add_argument("--drop-pad", default="1.0,1.25",
                    help="capacity factors of the drop-and-pad comparison runs (rank 0, after the "
                         "dropless measurement; empty to skip)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    from synth import CONFIGS, make_workload, shrink
    cfg = dict(CONFIGS[args.config], name=args.config)
    if args.shrink:
        over = {kv.split("=")[0]: int(kv.split("=")[1]) for kv in args.shrink.split(",")}
        cfg = shrink(args.config, **over)
    T = cfg["T"]
    dtype_name = "bf16" if cfg["dtype"] == "bf16" else "f32"
    workload_cfg = {"workload": f"{args.config}: T={T} d={cfg['d']} E={cfg['E']} top-{cfg['k']} "
                                f"f={cfg['f']} S={cfg['S']} f_s={cfg['f_s']} routing={cfg['routing']}"
                                + (f"(s={cfg['zipf_s']})" if cfg['routing'] == 'zipf' else ""),
                    "tokens_per_step": T, "l2": "inputs larger than L2 (expert weights > 20 GB)",
                    "parallelism": f"replicas x{world}"}
    if world > 1:
        workload_cfg["replicas"] = "data parallel: the same weights, each rank its own seeded tokens"

    if args.impl == "reference":
        if rank != 0:
            return
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        w = make_workload(cfg, device=dev)
        if w.logits_in is not None:
            logits32 = w.logits_in.cpu().numpy()
        else:       # fp32 scores of the sampled tokens (the oracle's own router, rounded to fp32)
            import oracle as O
            scale = oracle_scale(cfg)
            logits32 = O.router_logits(w.x[:T // scale].double().cpu().numpy(),
                                       w.w_r.double().cpu().numpy()).astype("float32")
        scale = oracle_scale(cfg)
        for _ in range(args.warmup):
            oracle_sample(w, logits32, scale)
        times = []
        for _ in range(args.steps):
            dt, Ts, Es = oracle_sample(w, logits32, scale)
            times.append(dt)
        tot = sum(times)
        value = args.steps * Ts / tot
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": workload_cfg,
                "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                                 "sample": "each step: " + sample_text(cfg, scale, Ts, Es)},
                "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    from dropless_token_routing_gb300 import _native as N
    from dropless_token_routing_gb300.api import LayerParams, MoELayer, get_device_error

    dev = torch.device("cuda", torch.cuda.current_device())
    w = make_workload(cfg, device=dev, replica=rank)   # data parallel: each rank its own tokens
    params = LayerParams(w13=w.w13, w2=w.w2, w_r=w.w_r, bias=w.bias, ws13=w.ws13, ws2=w.ws2)
    rflag = {"copy": 0, "gather": 1, "scatter": 2, "both": 3}[args.rearrange]
    gather = bool(rflag & 1)
    layer = MoELayer(params, T, cfg["d"], cfg["E"], cfg["k"], cfg["f"], cfg["S"], cfg["f_s"],
                     w.torch_dtype, device=dev, logits_input=w.logits_in is not None,
                     rearrange=rflag, recompute=gather)
    layer.alloc_grads()
    x, dy, li = w.x, w.dy, w.logits_in
    if rflag:
        workload_cfg["rearrange"] = {1: "row gathers fused into the expert GEMMs",
                                     2: "token-major rows written by the second expert GEMM",
                                     3: "row gathers and token-major rows fused into the GEMMs"}[rflag]
    stream = torch.cuda.current_stream()

    def step():
        layer.forward(x, li)
        layer.backward(dy)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    err = get_device_error(layer.ws)
    if err != 0:
        raise RuntimeError(f"device error {N.STATUS.get(err, err)} during warm-up")

    # ---------------------------------------------------------------- timed region
    sampler = ClockSampler(local if "CUDA_VISIBLE_DEVICES" not in os.environ else
                           os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local]) if rank == 0 else None
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        t_wait = time.time()
        while not sampler.lines and time.time() - t_wait < 5.0:   # nvidia-smi has started
            time.sleep(0.05)
        time.sleep(0.2)
    N.trace_enable(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    trace = N.trace_read()
    N.trace_enable(False)
    clocks = sampler.stop() if sampler else None
    t_ms = reduce_max(e0.elapsed_time(e1), dev)
    err = get_device_error(layer.ws)
    if err != 0:
        raise RuntimeError(f"device error {N.STATUS.get(err, err)} in the timed region")
    value = throughput(world, args.steps, T, t_ms)

    # ---------------------------------------------------------------- end to end
    # Every step copies its inputs from pinned host memory and reads y and dx back. The copies
    # run on two more streams (host-to-device and device-to-host, so the two directions
    # overlap), double-buffered: step i+2's inputs land while step i computes, y is read back
    # during the backward and dx during the next forward.
    h_x = x.cpu().pin_memory()
    h_dy = dy.cpu().pin_memory()
    h_li = li.cpu().pin_memory() if li is not None else None
    h_y = torch.empty_like(h_x).pin_memory()
    h_dx = torch.empty_like(h_x).pin_memory()
    up = torch.cuda.Stream(device=dev)
    down = torch.cuda.Stream(device=dev)
    d_in = [(torch.empty_like(x), torch.empty_like(dy), torch.empty_like(li) if li is not None else None)
            for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]     # the slot's inputs have landed
    ev_used = [torch.cuda.Event() for _ in range(2)]   # the compute is done with the slot
    ev_y, ev_yd, ev_dx, ev_dxd = (torch.cuda.Event() for _ in range(4))

    def h2d(slot):
        with torch.cuda.stream(up):
            up.wait_event(ev_used[slot])
            bx, bdy, bli = d_in[slot]
            bx.copy_(h_x, non_blocking=True)
            bdy.copy_(h_dy, non_blocking=True)
            if bli is not None:
                bli.copy_(h_li, non_blocking=True)
            ev_in[slot].record(up)

    def e2e_run(n):
        up.wait_stream(stream)
        down.wait_stream(stream)
        for s_ in range(min(2, n)):
            h2d(s_)
        for i in range(n):
            s_ = i % 2
            bx, bdy, bli = d_in[s_]
            stream.wait_event(ev_in[s_])
            stream.wait_event(ev_yd)          # the previous y has been read back
            y = layer.forward(bx, bli)
            ev_y.record(stream)
            with torch.cuda.stream(down):
                down.wait_event(ev_y)
                h_y.copy_(y, non_blocking=True)
                ev_yd.record(down)
            stream.wait_event(ev_dxd)         # the previous dx has been read back
            g = layer.backward(bdy)
            ev_used[s_].record(stream)
            ev_dx.record(stream)
            with torch.cuda.stream(down):
                down.wait_event(ev_dx)
                h_dx.copy_(g["dx"], non_blocking=True)
                ev_dxd.record(down)
            if i + 2 < n:
                h2d(s_)                       # the inputs of step i + 2
        stream.wait_stream(up)
        stream.wait_stream(down)

    e2e_run(2)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    k_e2e = max(3, args.steps)
    e2.record(stream)
    e2e_run(k_e2e)
    e3.record(stream)
    torch.cuda.synchronize()
    t_e2e = reduce_max(e2.elapsed_time(e3), dev)
    es = 2 if cfg["dtype"] == "bf16" else 4
    h2d = 2 * T * cfg["d"] * es + (T * cfg["E"] * 4 if li is not None else 0)
    d2h = 2 * T * cfg["d"] * es
    e2e = {"value": throughput(world, k_e2e, T, t_e2e), "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h}

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    # ---------------------------------------------------------------- roofline
    peaks = _peaks()
    cnt = layer.saved["counts"].cpu().tolist()
    summ = summarize(cfg, trace, args.steps, cnt, peaks)
    kernels, launches = summ["kernels"], summ["launches"]
    dom = summ["dominant"]
    dl, dms = trace[dom]
    per = dms / dl
    flops, bytes_ = algorithmic_work(cfg)
    traffic = None
    tr = NCU_TRAFFIC.get(dom)
    # the captured bytes hold only for the workload they were captured on
    if tr and tr.get("bytes_per_launch") and tr.get("workload") == cfg["name"]:
        src = os.path.join(ROOT, "dropless_token_routing_gb300", "csrc", tr["src"])
        if tr.get("src_sha256") == _sha(src):
            traffic = tr["bytes_per_launch"]
    if dom in flops:
        ach = flops[dom] / (per / 1e3) / 1e12
        peak = peaks["bf16_tflops_sustained"]
        roof = {"bound": "tensor", "achieved": round(ach, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(ach / peak, 3), "traffic": traffic, "kernel": dom,
                "peak_kind": f"bf16 dense, sustained ({peaks['source']})",
                "frac_of_burst_peak": round(ach / peaks["bf16_tflops"], 3)}
    else:
        ach = bytes_[dom] / (per / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / peaks["hbm_gbs"], 3), "traffic": traffic, "kernel": dom,
                "peak_kind": f"HBM copy ({peaks['source']})"}
    wb = dw_write_bytes(cfg).get(dom)
    if wb:
        # the dW products write their whole output and read little: their writes alone
        # against the HBM bandwidth (a fill by TMA bulk stores from shared memory reaches the
        # copy figure on this part)
        wach = wb / (per / 1e3) / 1e9
        roof["write_stream"] = {"bytes": wb, "achieved": round(wach, 1), "peak": peaks["hbm_gbs"],
                                "unit": "GB/s", "frac": round(wach / peaks["hbm_gbs"], 3),
                                "peak_kind": f"HBM copy ({peaks['source']})"}
    line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_ms / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype_name,
            "data": "synthetic (seeded, device-generated)", "config": workload_cfg,
            "roofline": roof, "gpu_launches": launches, "e2e": e2e, "clocks": clocks,
            "grouped_gemm": summ["grouped_gemm"], "routing": summ["routing"], "kernels": kernels}
    if not args.no_cpu_baseline and world == 1:
        logits32 = (li if li is not None else layer.saved["logits"]).cpu().numpy()
        line["cpu_baseline"] = cpu_baseline(w, logits32)
    factors = [float(v) for v in args.drop_pad.split(",") if v.strip()]
    if factors:
        line["drop_and_pad"] = drop_and_pad(factors, params, cfg, w, cnt, args, stream)
    if args.fused_rearrange and cfg["dtype"] == "bf16":
        line["fused_rearrange"] = fused_rearrange(params, cfg, w, args, stream)
    if args.balance_statistics:
        line["balance_statistics"] = balance_statistics(
            cfg, w, (li if li is not None else layer.saved["logits"]), layer.ws, stream, peaks)
    others = [n for n in args.other_workloads.split(",") if n.strip() and n.strip() != args.config]
    if others and not args.shrink:
        del layer, params, w, x, dy, li, d_in, h_x, h_dy, h_li, h_y, h_dx
        torch.cuda.empty_cache()
        line["other_workloads"] = {n: other_workload(n.strip(), args, dev, peaks) for n in others}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
