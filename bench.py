#!/usr/bin/env python
"""Benchmark of causal GQA + RoPE attention, forward + backward, on GB300.

Workload: the attention of one full training step of the NanoEuler 116M model
("NanoEuler: a GPT-2-scale LLM built from scratch in C and CUDA", model
configuration table: dim 768, 12/4 heads, 16 layers, context 512), batch 64:
16 independent layers, each B=64 T=512 Hq=12 Hkv=4 d=64, forward then
backward on one stream, every layer with its own buffers (4.3 GB in all, so
each layer's inputs are cold in the 129 MB L2).  Synthetic seeded N(0, 1)
inputs (see ne_inputs.py).

A step = 16 x (ne_attn_fwd_save, then the three backward steps of
ne_attn_bwd_saved) through the C ABI: the training pair, in which the forward
leaves the rotated Q', K' in the workspace for the backward.
The step is captured in a CUDA graph so Python call overhead does not leave
the GPU idle; CUDA events inside the graph time every kernel.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the float64 CPU oracle (the only reference this
subject has) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import ne_inputs  # noqa: E402

W = ne_inputs.STEP_116M
METRIC = "causal GQA attn fwd+bwd TFLOP/s and tokens/s at T=512 12/4 heads; % BF16 peak"
UNIT = "TFLOP/s"
CONFIG = {
    "workload": W.name,
    "layers": W.layers, "B": W.B, "T": W.T, "Hq": W.Hq, "Hkv": W.Hkv, "d": W.d,
    "causal": True, "rope_theta": W.theta,
    "l2": "inputs larger than L2: 16 layers x 270 MB of separate buffers",
}
FLOP_PER_LAYER = W.flops_fwd() + W.flops_bwd()
FLOP_PER_STEP = FLOP_PER_LAYER * W.layers
TOKENS_PER_STEP = W.tokens()          # B*T tokens go through all 16 layers per step


# ------------------------------------------------------------ roofline ---

def _mb(n_elem, bytes_per):
    return n_elem * bytes_per


def kernel_work(w=W):
    """Algorithmic flops and compulsory HBM bytes of ONE launch of each kernel
    for one layer (per-unit figures x the units one launch processes).

    "bytes" follows the compulsory-traffic convention: the forward reads Q, K,
    V and writes O and lse.  Traffic a kernel makes by choice goes to
    "extra_bytes" and is not counted in the roofline: the training-path
    forward also stores the fp16 rotated Q' and K' for the backward.  The dq
    and dk/dv kernels read those fp16 Q', K' in place of the bf16 q, k (the
    same number of bytes)."""
    B, T, Hq, Hkv, d = w.B, w.T, w.Hq, w.Hkv, w.d
    pairs = w.pairs * B * Hq                       # causal (t, s) pairs x heads
    q = B * T * Hq * d * 2
    kv = B * T * Hkv * d * 2
    row = B * Hq * T * 4                           # lse or D
    return {
        # QK^T and PV: 2 GEMMs of 2d flops per pair; reads Q K V, writes O lse
        "fwd": {"flops": 4.0 * d * pairs, "bytes": q + 2 * kv + q + row, "extra_bytes": q + kv},
        # D = rowsum(dO * O): reads O, dO; writes D
        "bwd_pre": {"flops": 2.0 * B * T * Hq * d, "bytes": 2 * q + row, "extra_bytes": 0},
        # dQ = dS K' (one GEMM; the S and dP recompute is not algorithmic work);
        # reads Q' K' V dO lse D, writes dQ
        "bwd_dq": {"flops": 2.0 * d * pairs, "bytes": q + 2 * kv + q + 2 * row + q,
                   "extra_bytes": 0},
        # S, dP, dV, dK (four GEMMs); reads Q' K' V dO lse D, writes dK dV
        "bwd_dkdv": {"flops": 8.0 * d * pairs, "bytes": q + 2 * kv + q + 2 * row + 2 * kv,
                     "extra_bytes": 0},
    }


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def csrc_hash() -> str:
    h = hashlib.sha256()
    d = os.path.join(ROOT, "causal_gqa_attention_ne_gb300", "csrc")
    for name in sorted(os.listdir(d)):
        with open(os.path.join(d, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic_gpt116m_step.txt")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"csrc_sha256_16:\s*([0-9a-f]+)", text)
    if not m or m.group(1) != csrc_hash():
        return None
    m = re.search(rf"^{kernel}\s+([0-9.eE+]+)\s*$", text, re.M)
    return float(m.group(1)) if m else None


# -------------------------------------------------------------- clocks ---

class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t_start = self.t_end = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, start: bool):
        if start:
            self.t_start = time.time()
        else:
            self.t_end = time.time()

    def stop(self):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        win = [l for (t, l) in self.lines if self.t_start and self.t_start - 0.06 <= t <= (
            self.t_end or t) + 0.06]
        if len(win) < 3:
            win = [l for (_, l) in self.lines]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in win:
            parts = [p.strip() for p in l.split(",")]
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(win)}


# ---------------------------------------------------------- our arm ---

def make_event(torch, external):
    if external:
        try:
            return torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:
            pass
    return torch.cuda.Event(enable_timing=True)


def max_over_ranks(ms: float, device, world: int) -> float:
    """The slowest rank's time: every rank passes its own, every rank gets the max
    (one all-reduce; a no-op for a single process)."""
    if world <= 1:
        return ms
    import torch
    tt = torch.tensor([ms], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
    return float(tt.item())


def job_rate(world: int, units_per_step: float, steps: int, elapsed_ms: float) -> float:
    """Whole-job throughput of weak-scaled replicas: the units all ranks processed
    over the slowest rank's time."""
    return world * units_per_step * steps / (elapsed_ms * 1e-3)


def run_ours(args, rank, world, local_rank):
    import torch

    import causal_gqa_attention_ne_gb300 as ne
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    ne.load_library()

    layers = []
    for layer in range(W.layers):
        x = ne_inputs.make_inputs(W, layer)
        host = {n: t.pin_memory() for n, t in x.items()}
        d = {n: t.to(dev) for n, t in x.items()}
        d["o"] = torch.empty_like(d["q"])
        d["lse"] = torch.empty(W.B, W.Hq, W.T, dtype=torch.float32, device=dev)
        d["dq"] = torch.empty_like(d["q"])
        d["dk"] = torch.empty_like(d["k"])
        d["dv"] = torch.empty_like(d["v"])
        d["ws"] = torch.empty(ne.ne_attn_bwd_workspace_size(W.B, W.T, W.Hq, W.Hkv, W.d),
                              dtype=torch.uint8, device=dev)
        out_host = {n: torch.empty(d[n].shape, dtype=d[n].dtype, pin_memory=True)
                    for n in ("o", "lse", "dq", "dk", "dv")}
        layers.append((host, d, out_host))
    theta = W.theta
    names = ("fwd", "bwd_pre", "bwd_dq", "bwd_dkdv")

    def step(evs=None):
        for li, (_, d, _) in enumerate(layers):
            if evs is not None:
                evs[li][0].record()
            ne.ne_attn_fwd_save(d["q"], d["k"], d["v"], d["o"], d["lse"], d["ws"], theta)
            if evs is not None:
                evs[li][1].record()
            ne.ne_attn_bwd_preprocess_d(d["o"], d["do"], d["ws"], W.Hkv)
            if evs is not None:
                evs[li][2].record()
            ne.ne_attn_bwd_dq(d["q"], d["k"], d["v"], d["lse"], d["do"], d["dq"], d["ws"], theta)
            if evs is not None:
                evs[li][3].record()
            ne.ne_attn_bwd_dkdv(d["q"], d["k"], d["v"], d["lse"], d["do"], d["dk"], d["dv"],
                                d["ws"], theta)
            if evs is not None:
                evs[li][4].record()

    # eager warm-up call (sets kernel attributes, checks status)
    step()
    torch.cuda.synchronize()
    st = ne.ne_attn_get_error()
    if st != 0:
        raise RuntimeError(f"device status {ne.NE_STATUS.get(st, st)} after warm-up")

    # The timed step is one CUDA graph of the 4 x 16 kernels alone.  The
    # kernels are launched with programmatic dependent launch, so in the graph
    # each one is scheduled while its predecessor drains; a timing event
    # between two kernels would cut that edge, so the per-kernel durations
    # come from a second capture of the same step with an event between
    # consecutive kernels, replayed right after the timed region.
    K, Wm = args.steps, args.warmup
    cap_stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap_stream):
        step()
    KI = min(K, 8)
    igraphs, events = [], []
    for k in range(KI):
        evs = [[make_event(torch, True) for _ in range(5)] for _ in range(W.layers)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap_stream):
            step(evs)
        igraphs.append(g)
        events.append(evs)
    torch.cuda.synchronize()

    warm = max(Wm, 1)
    for i in range(warm):
        graph.replay()
    for g in igraphs:
        g.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    sampler.mark(True)
    t0.record()
    for _ in range(K):
        graph.replay()
    t1.record()
    torch.cuda.synchronize()
    sampler.mark(False)
    if world > 1:
        torch.distributed.barrier()
    sampler.stop()
    elapsed_ms = t0.elapsed_time(t1)
    st = ne.ne_attn_get_error()
    if st != 0:
        raise RuntimeError(f"device status {ne.NE_STATUS.get(st, st)} after timed region")

    # per-kernel durations: the instrumented step graphs, each replayed once
    for g in igraphs:
        g.replay()
    torch.cuda.synchronize()
    per = {n: [] for n in names}
    for evs in events:
        for le in evs:
            for i, n in enumerate(names):
                per[n].append(le[i].elapsed_time(le[i + 1]))
    avg_ms = {n: statistics.mean(v) for n, v in per.items()}

    elapsed_ms = max_over_ranks(elapsed_ms, dev, world)
    ms_per_step = elapsed_ms / K
    value = job_rate(world, FLOP_PER_STEP, K, elapsed_ms) / 1e12
    tokens_per_s = job_rate(world, TOKENS_PER_STEP, K, elapsed_ms)

    # end to end: host buffers in, host buffers out, through the eager C-ABI
    # calls.  The layers are pipelined over three streams: the uploads of
    # every layer's inputs (h2d), the kernels (s, each layer after its
    # inputs have landed), the downloads of every layer's outputs (d2h, each
    # after its layer's kernels), so layer i+1's inputs and layer i-1's
    # outputs travel while layer i computes.  A step's uploads wait for the
    # previous step's kernels, and its kernels for the previous step's
    # downloads (the buffers are reused).
    e2e_steps = max(1, min(args.e2e_steps, K))
    h2d = sum(sum(t.numel() * t.element_size() for t in host.values()) for host, _, _ in layers)
    d2h = sum(sum(t.numel() * t.element_size() for t in oh.values()) for _, _, oh in layers)
    s = torch.cuda.current_stream()
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    for rep in range(e2e_steps + 1):          # first pass warms the copy path
        if rep == 1:
            torch.cuda.synchronize()
            if world > 1:
                torch.distributed.barrier()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(s)
            h0 = time.perf_counter()
        ev_in = [torch.cuda.Event() for _ in layers]
        ev_done = [torch.cuda.Event() for _ in layers]
        h2d_s.wait_stream(s)
        with torch.cuda.stream(h2d_s):
            for li, (host, d, _) in enumerate(layers):
                for n in ("q", "k", "v", "do"):
                    d[n].copy_(host[n], non_blocking=True)
                ev_in[li].record(h2d_s)
        s.wait_stream(d2h_s)
        for li, (host, d, oh) in enumerate(layers):
            s.wait_event(ev_in[li])
            ne.ne_attn_fwd_save(d["q"], d["k"], d["v"], d["o"], d["lse"], d["ws"], theta)
            ne.ne_attn_bwd_saved(d["q"], d["k"], d["v"], d["o"], d["lse"], d["do"], d["dq"],
                                 d["dk"], d["dv"], d["ws"], theta)
            ev_done[li].record(s)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(ev_done[li])
                for n in ("o", "lse", "dq", "dk", "dv"):
                    oh[n].copy_(d[n], non_blocking=True)
        s.wait_stream(d2h_s)
    e1.record(s)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    host_ms = (time.perf_counter() - h0) * 1e3 / e2e_steps
    e2e_ms = max_over_ranks(max(e2e_ms, host_ms), dev, world)
    st = ne.ne_attn_get_error()
    if st != 0:
        raise RuntimeError(f"device status {ne.NE_STATUS.get(st, st)} after e2e")

    # roofline of the dominant kernel (largest share of the step)
    peaks = load_peaks()
    work = kernel_work()
    dom = max(names, key=lambda n: avg_ms[n])
    wk = work[dom]
    t_tensor = wk["flops"] / (peaks["bf16_tflops"] * 1e12)
    t_hbm = wk["bytes"] / (peaks["hbm_gbs"] * 1e9)
    dur_s = avg_ms[dom] * 1e-3
    if t_tensor >= t_hbm:
        roof = {"bound": "tensor", "achieved": wk["flops"] / dur_s / 1e12,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": wk["bytes"] / dur_s / 1e9,
                "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = measured_traffic(dom)
    roof["kernel"] = dom
    roof["peak_source"] = f"{peaks['source']} (burst: kernels timed inside a short step)"
    roof["algorithmic"] = {"flops": wk["flops"], "bytes": wk["bytes"],
                           "extra_bytes": wk["extra_bytes"]}

    kernels = {n: {"avg_us": avg_ms[n] * 1e3, "launches": len(per[n]),
                   "share": avg_ms[n] / sum(avg_ms.values()),
                   "tflops": work[n]["flops"] / (avg_ms[n] * 1e-3) / 1e12,
                   "gbs": work[n]["bytes"] / (avg_ms[n] * 1e-3) / 1e9} for n in names}

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": warm, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "operand_dtypes": {"qk_scores_and_dS": "fp16", "p_v_dO": "bf16", "accumulate": "fp32"},
        "data": "synthetic (seeded N(0,1), see ne_inputs.py)",
        "config": CONFIG,
        "tokens_per_s": tokens_per_s,
        "pct_bf16_peak": value / (peaks["bf16_tflops"] * world) * 100.0,
        "e2e": {"value": job_rate(world, FLOP_PER_STEP, 1, e2e_ms) / 1e12, "unit": UNIT,
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps,
                "overlap": "per layer: uploads, kernels and downloads on three streams"},
        "gpu_launches": 4 * W.layers * K,
        "roofline": roof,
        "kernels": kernels,
        "clocks": sampler.summary(),
    }
    return result


def run_decode(args):
    """Decode against a KV cache: 16 layers (own caches, 537 MB in all, so each
    layer's cache is cold in L2) x ne_attn_decode of B=64 new tokens over 512
    cached positions, 12/4 heads, d=64; one CUDA graph per step.  HBM-bound:
    the metric is the algorithmic bytes (K and V caches, q, o, lse) per second."""
    import torch

    import causal_gqa_attention_ne_gb300 as ne
    w = ne_inputs.DECODE_116M
    ne.load_library()
    dev = torch.device("cuda", 0)
    layers = []
    for layer in range(w.layers):
        x = ne_inputs.make_inputs(w, layer)
        q1 = x["q"][:, -1].contiguous().to(dev)
        k, v = x["k"].to(dev), x["v"].to(dev)
        o = torch.empty_like(q1)
        lse = torch.empty(w.B, w.Hq, dtype=torch.float32, device=dev)
        ws = torch.empty(ne.ne_attn_decode_workspace_size(w.B, w.T, w.Hq, w.Hkv, w.d),
                         dtype=torch.uint8, device=dev)
        layers.append((q1, k, v, o, lse, ws))

    def step():
        for q1, k, v, o, lse, ws in layers:
            ne.ne_attn_decode(q1, k, v, o, lse, ws, w.theta)

    step()
    torch.cuda.synchronize()
    st = ne.ne_attn_get_error()
    if st != 0:
        raise RuntimeError(f"device status {ne.NE_STATUS.get(st, st)}")
    cap = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        step()
    for _ in range(max(args.warmup, 3)):
        graph.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.mark(True)
    e0.record()
    for _ in range(args.steps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    sampler.mark(False)
    sampler.stop()
    ms = e0.elapsed_time(e1) / args.steps
    kv = 2 * w.B * w.T * w.Hkv * w.d * 2
    small = w.B * w.Hq * w.d * 2 * 2 + w.B * w.Hq * 4
    nbytes = (kv + small) * w.layers
    gbs = nbytes / (ms * 1e-3) / 1e9
    peaks = load_peaks()
    return {
        "metric": "decode attention against a KV cache: GB/s of algorithmic HBM traffic "
                  "(K, V caches, q, o, lse) at Tk=512, 12/4 heads, d=64",
        "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True,
        "dtype": "bf16 in, fp32 math", "data": "synthetic (seeded N(0,1), see ne_inputs.py)",
        "config": {"workload": w.name, "layers": w.layers, "B": w.B, "Tk": w.T, "Hq": w.Hq,
                   "Hkv": w.Hkv, "d": w.d,
                   "l2": "16 layers x 33.6 MB of separate caches (537 MB > L2)"},
        "tokens_per_s": w.B * args.steps / (e0.elapsed_time(e1) * 1e-3),
        "gpu_launches": 2 * w.layers * args.steps,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                     "peak_source": peaks["source"]},
        "clocks": sampler.summary(),
    }


def run_window(args):
    """The training step's workload (16 layers x B64 T512 12/4 d64, own buffers)
    with a sliding window of args.window keys: the training pair
    (ne_attn_fwd_save, ne_attn_bwd_saved) with `window`, one CUDA graph per step.  Algorithmic flops
    count the pairs inside the window only (t - W < s <= t)."""
    import torch

    import causal_gqa_attention_ne_gb300 as ne
    Wn = args.window
    ne.load_library()
    dev = torch.device("cuda", 0)
    layers = []
    for layer in range(W.layers):
        x = {n: t.to(dev) for n, t in ne_inputs.make_inputs(W, layer).items()}
        x["o"] = torch.empty_like(x["q"])
        x["lse"] = torch.empty(W.B, W.Hq, W.T, dtype=torch.float32, device=dev)
        x["dq"], x["dk"], x["dv"] = (torch.empty_like(x["q"]), torch.empty_like(x["k"]),
                                     torch.empty_like(x["v"]))
        x["ws"] = torch.empty(ne.ne_attn_bwd_workspace_size(W.B, W.T, W.Hq, W.Hkv, W.d),
                              dtype=torch.uint8, device=dev)
        layers.append(x)

    def step():
        for d in layers:
            ne.ne_attn_fwd_save(d["q"], d["k"], d["v"], d["o"], d["lse"], d["ws"], W.theta,
                                window=Wn)
            ne.ne_attn_bwd_saved(d["q"], d["k"], d["v"], d["o"], d["lse"], d["do"], d["dq"],
                                 d["dk"], d["dv"], d["ws"], W.theta, window=Wn)

    step()
    torch.cuda.synchronize()
    st = ne.ne_attn_get_error()
    if st != 0:
        raise RuntimeError(f"device status {ne.NE_STATUS.get(st, st)}")
    cap = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        step()
    for _ in range(max(args.warmup, 3)):
        graph.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.mark(True)
    e0.record()
    for _ in range(args.steps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    sampler.mark(False)
    sampler.stop()
    ms = e0.elapsed_time(e1) / args.steps
    pairs = sum(min(t + 1, Wn) for t in range(W.T))
    flops = 14.0 * W.d * pairs * W.B * W.Hq * W.layers
    peaks = load_peaks()
    value = flops / (ms * 1e-3) / 1e12
    return {
        "metric": f"sliding-window (W={Wn}) GQA attn fwd+bwd TFLOP/s at T=512 12/4 heads",
        "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1), see ne_inputs.py)",
        "config": {"workload": W.name, "window": Wn, "pairs_per_head": pairs,
                   "causal_pairs_per_head": W.pairs,
                   "path": "ne_attn_fwd_save + ne_attn_bwd_saved with window"},
        "tokens_per_s": W.tokens() * args.steps / (e0.elapsed_time(e1) * 1e-3),
        "pct_bf16_peak": value / peaks["bf16_tflops"] * 100.0,
        "gpu_launches": 4 * W.layers * args.steps,
        "clocks": sampler.summary(),
    }


def run_varlen(args):
    """The 116M SFT step: 16 layers of B64 sequences padded to T=512 (12/4
    heads, d64), each sequence with its own seeded valid length (ne_inputs:
    uniform on [16, 512]); per layer ne_attn_fwd_varlen_dev then
    ne_attn_bwd_varlen_dev with the lengths in device memory, the 16 layers
    captured as one CUDA graph (the unit tables are planned on the GPU).
    Algorithmic flops count the causal pairs of the valid rows only.  Timed
    beside it: the padded causal step (ne_attn_fwd + ne_attn_bwd on the same
    buffers, also one graph) and the host-length entry points launched
    eagerly (their tables are copied from host memory, which a graph cannot
    capture)."""
    import numpy as np
    import torch

    import causal_gqa_attention_ne_gb300 as ne
    w = ne_inputs.SFT_116M
    lens = w.seqlens()
    ne.load_library()
    dev = torch.device("cuda", 0)
    layers = []
    for layer in range(w.layers):
        x = {n: t.to(dev) for n, t in ne_inputs.make_inputs(w, layer).items()}
        x["o"] = torch.empty_like(x["q"])
        x["lse"] = torch.empty(w.B, w.Hq, w.T, dtype=torch.float32, device=dev)
        x["dq"], x["dk"], x["dv"] = (torch.empty_like(x["q"]), torch.empty_like(x["k"]),
                                     torch.empty_like(x["v"]))
        x["ws"] = torch.empty(ne.ne_attn_varlen_workspace_size(w.B, w.T, w.Hq, w.Hkv, w.d),
                              dtype=torch.uint8, device=dev)
        layers.append(x)
    sl = np.asarray(lens, dtype=np.int32)
    sl_dev = torch.from_numpy(sl).to(dev)

    def step_varlen_dev():
        for d in layers:
            ne.ne_attn_fwd_varlen_dev(d["q"], d["k"], d["v"], d["o"], d["lse"], sl_dev, d["ws"],
                                      w.theta)
            ne.ne_attn_bwd_varlen_dev(d["q"], d["k"], d["v"], d["o"], d["lse"], d["do"],
                                      d["dq"], d["dk"], d["dv"], sl_dev, d["ws"], w.theta)

    def step_varlen():
        for d in layers:
            ne.ne_attn_fwd_varlen(d["q"], d["k"], d["v"], d["o"], d["lse"], sl, d["ws"], w.theta)
            ne.ne_attn_bwd_varlen(d["q"], d["k"], d["v"], d["o"], d["lse"], d["do"], d["dq"],
                                  d["dk"], d["dv"], sl, d["ws"], w.theta)

    def step_padded():
        for d in layers:
            ne.ne_attn_fwd(d["q"], d["k"], d["v"], d["o"], d["lse"], w.theta)
            ne.ne_attn_bwd(d["q"], d["k"], d["v"], d["o"], d["lse"], d["do"], d["dq"], d["dk"],
                           d["dv"], d["ws"], w.theta)

    def as_graph(step):
        step()                                  # eager once: kernel attributes, checks
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=torch.cuda.Stream()):
            step()
        return g.replay

    def timed(step, sampler=None):
        for _ in range(max(args.warmup, 3)):
            step()
        torch.cuda.synchronize()
        st = ne.ne_attn_get_error()
        if st != 0:
            raise RuntimeError(f"device status {ne.NE_STATUS.get(st, st)}")
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if sampler:
            sampler.mark(True)
        e0.record()
        for _ in range(args.steps):
            step()
        e1.record()
        torch.cuda.synchronize()
        if sampler:
            sampler.mark(False)
        return e0.elapsed_time(e1) / args.steps

    ms_pad = timed(as_graph(step_padded))
    ms_eager = timed(step_varlen)
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.3)
    ms = timed(as_graph(step_varlen_dev), sampler)
    sampler.stop()
    pairs = w.valid_pairs()
    flops = 14.0 * w.d * pairs * w.Hq * w.layers
    peaks = load_peaks()
    value = flops / (ms * 1e-3) / 1e12
    counts, _ = ne.ne_attn_varlen_plan(lens, w.T, w.Hq, w.Hkv, w.d, with_tables=False)
    return {
        "metric": "padded variable-length GQA attn fwd+bwd TFLOP/s (valid causal pairs) at "
                  "T=512 12/4 heads",
        "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) and lengths, see ne_inputs.py)",
        "config": {"workload": w.name, "valid_tokens": int(sum(lens)),
                   "padded_tokens": w.B * w.T, "valid_pair_fraction": pairs / (w.B * w.pairs),
                   "live_units": counts,
                   "path": "ne_attn_fwd_varlen_dev + ne_attn_bwd_varlen_dev (lengths in device "
                           "memory), one CUDA graph per step"},
        "valid_tokens_per_s": sum(lens) * w.layers / (ms * 1e-3),
        "padded_causal_ms_per_step": ms_pad,
        "speedup_vs_padded": ms_pad / ms,
        "host_lengths_eager_ms_per_step": ms_eager,
        "pct_bf16_peak": value / peaks["bf16_tflops"] * 100.0,
        "gpu_launches": 8 * w.layers * args.steps,
        "clocks": sampler.summary(),
    }


def run_config(args):
    """One workload of the parity set timed on its own (SURVEY measurement
    plan): c3 = gpt116m_b16_t512_h12x4_d64 (one 116M layer, B16), c5 =
    stress_b4_t4096_h16x4_d128.  Per call, CUDA events on the stream, 10
    warm-up calls then the median of `--reps`: the forward (ne_attn_fwd), the
    backward (ne_attn_bwd, preprocess included), the two back to back, and
    the training pair (ne_attn_fwd_save + ne_attn_bwd_saved).  Inputs of c3
    fit in L2, so c3 is timed warm (back to back) and with L2 flushed (a
    write of a buffer twice the L2 size before every timed call)."""
    import torch

    import causal_gqa_attention_ne_gb300 as ne
    w = {"c3": ne_inputs.LAYER_116M, "c5": ne_inputs.STRESS}[args.config]
    ne.load_library()
    dev = torch.device("cuda", 0)
    x = {n: t.to(dev) for n, t in ne_inputs.make_inputs(w, 0).items()}
    o = torch.empty_like(x["q"])
    lse = torch.empty(w.B, w.Hq, w.T, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["v"])
    ws = torch.empty(ne.ne_attn_bwd_workspace_size(w.B, w.T, w.Hq, w.Hkv, w.d),
                     dtype=torch.uint8, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)

    def fwd():
        ne.ne_attn_fwd(x["q"], x["k"], x["v"], o, lse, w.theta)

    def bwd():
        ne.ne_attn_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], dq, dk, dv, ws, w.theta)

    def both():
        fwd()
        bwd()

    def pair():
        ne.ne_attn_fwd_save(x["q"], x["k"], x["v"], o, lse, ws, w.theta)
        ne.ne_attn_bwd_saved(x["q"], x["k"], x["v"], o, lse, x["do"], dq, dk, dv, ws, w.theta)

    def median_ms(fn, flush_l2):
        for _ in range(10):
            fn()
        torch.cuda.synchronize()
        times = []
        for _ in range(args.reps):
            if flush_l2:
                flush.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        st = ne.ne_attn_get_error()
        if st != 0:
            raise RuntimeError(f"device status {ne.NE_STATUS.get(st, st)}")
        return statistics.median(times)

    peaks = load_peaks()
    flops = {"fwd": w.flops_fwd(), "bwd": w.flops_bwd()}
    flops["fwd_bwd"] = flops["fwd"] + flops["bwd"]
    flops["train_pair"] = flops["fwd_bwd"]
    modes = [False, True] if args.config == "c3" else [False]
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.3)
    sampler.mark(True)
    out = {}
    for fl in modes:
        key = "l2_flushed" if fl else "warm"
        res = {}
        for name, fn in (("fwd", fwd), ("bwd", bwd), ("fwd_bwd", both), ("train_pair", pair)):
            ms = median_ms(fn, fl)
            tf = flops[name] / (ms * 1e-3) / 1e12
            res[name] = {"median_ms": ms, "tflops": tf,
                         "pct_bf16_peak": tf / peaks["bf16_tflops"] * 100.0}
        out[key] = res
    sampler.mark(False)
    sampler.stop()
    head = out["warm"]["fwd_bwd"]
    return {
        "metric": f"causal GQA attn fwd+bwd TFLOP/s, {w.name}",
        "value": head["tflops"], "unit": "TFLOP/s", "n_gpus": 1, "steps": args.reps,
        "warmup": 10, "ms_per_step": head["median_ms"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded, see ne_inputs.py)",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d,
                   "timing": "median of per-call CUDA events",
                   "l2": "warm and L2-flushed (c3 fits in L2)" if args.config == "c3"
                   else "inputs larger than L2"},
        "tokens_per_s": w.tokens() / (head["median_ms"] * 1e-3),
        "results": out,
        "gpu_launches": None,
        "clocks": sampler.summary(),
    }


def run_one_layer_for_profiler():
    """One layer (B64 T512 12/4 d64, 270 MB of buffers), fwd then bwd, twice.
    The first pass warms up; a profiler captures the second (-s 4 -c 4)."""
    import torch

    import causal_gqa_attention_ne_gb300 as ne
    x = {n: t.cuda() for n, t in ne_inputs.make_inputs(W, 0).items()}
    ws = torch.empty(ne.ne_attn_bwd_workspace_size(W.B, W.T, W.Hq, W.Hkv, W.d),
                     dtype=torch.uint8, device="cuda")
    o, lse = torch.empty_like(x["q"]), torch.empty(W.B, W.Hq, W.T, device="cuda")
    dq, dk, dv = torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["v"])
    for _ in range(2):
        ne.ne_attn_fwd_save(x["q"], x["k"], x["v"], o, lse, ws, W.theta)
        ne.ne_attn_bwd_saved(x["q"], x["k"], x["v"], o, lse, x["do"], dq, dk, dv, ws, W.theta)
    torch.cuda.synchronize()
    st = ne.ne_attn_get_error()
    if st != 0:
        raise RuntimeError(f"device status {ne.NE_STATUS.get(st, st)}")


# --------------------------------------------------------- CPU oracle ---

def oracle_sample(batch_rows: int, threads: int = 0, layer: int = 0):
    """Time the float64 oracle (fwd + bwd) on the first `batch_rows` rows of one layer."""
    import oracle
    x = ne_inputs.make_inputs(W, layer)
    q, k, v, do = (ne_inputs.as_f64(x[n][:batch_rows]) for n in ("q", "k", "v", "do"))
    t0 = time.perf_counter()
    oracle.attn_fwd(q, k, v, W.theta, threads=threads)
    oracle.attn_bwd(q, k, v, do, W.theta, threads=threads)
    dt = time.perf_counter() - t0
    flops = FLOP_PER_LAYER * batch_rows / W.B
    used = threads if threads > 0 else oracle.max_threads()
    return flops / dt / 1e12, dt, used


def cpu_baseline(n_layers: int, single_rows: int = 2):
    """The oracle on the first `n_layers` full layers of the workload (fwd + bwd)
    on all host cores, and on the first `single_rows` batch rows of layer 0
    with one thread."""
    total, used = 0.0, 1
    for layer in range(n_layers):
        _, dt, used = oracle_sample(W.B, layer=layer)
        total += dt
    val = FLOP_PER_LAYER * n_layers / total / 1e12
    v1, dt1, _ = oracle_sample(single_rows, threads=1)
    return {"value": val, "unit": UNIT, "cores": used, "kind": "oracle", "seconds": total,
            "sample": f"layers 0-{n_layers - 1} of the {W.layers} of {W.name} (all {W.B} batch "
                      f"rows), fwd + bwd in float64 (OpenMP over heads / kv groups)",
            "single_thread": {"value": v1, "unit": UNIT, "cores": 1, "seconds": dt1,
                              "sample": f"layer 0, first {single_rows} of {W.B} batch rows, "
                                        f"fwd + bwd in float64, one thread"}}


def run_reference(args):
    """The reference arm: the float64 CPU oracle, timed on the host cores."""
    rows = args.ref_batch_rows
    for _ in range(args.warmup):
        oracle_sample(rows)
    times = []
    used = 1
    for _ in range(args.steps):
        _, dt, used = oracle_sample(rows)
        times.append(dt)
    flops = FLOP_PER_LAYER * rows / W.B
    total = sum(times)
    value = flops * len(times) / total / 1e12
    sample = (f"each step: layer 0 of {W.name}, first {rows} of {W.B} batch rows, "
              f"fwd + bwd in float64")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / len(times) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1), see ne_inputs.py)", "config": CONFIG,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--e2e-steps", type=int, default=2)
    ap.add_argument("--cpu-layers", type=int, default=6,
                    help="full layers of the workload the CPU-baseline oracle sample covers")
    ap.add_argument("--ref-batch-rows", type=int, default=4,
                    help="batch rows per step of the reference (oracle) arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ncu-layer", action="store_true",
                    help="profiler mode: run one layer of the workload (fwd, then the three "
                         "backward steps) twice, eagerly, and exit; no timing, no JSON")
    ap.add_argument("--decode", action="store_true",
                    help="time decode against a KV cache (16 layers of B64, Tk 512) instead "
                         "of the training step; prints its own JSON line")
    ap.add_argument("--window", type=int, default=0,
                    help="time the training step with a sliding window of this many keys "
                         "(the window entry points) instead; prints its own JSON line")
    ap.add_argument("--config", choices=("c3", "c5"), default=None,
                    help="time one parity workload on its own (fwd, bwd, fwd+bwd and the "
                         "training pair; medians of per-call events); own JSON line")
    ap.add_argument("--reps", type=int, default=50)
    ap.add_argument("--varlen", action="store_true",
                    help="time the padded variable-length SFT step (16 layers of B64 padded "
                         "to 512, seeded lengths) instead; prints its own JSON line")
    args = ap.parse_args()
    if args.config:
        print(json.dumps(run_config(args)), flush=True)
        return
    if args.varlen:
        print(json.dumps(run_varlen(args)), flush=True)
        return
    if args.window > 0:
        print(json.dumps(run_window(args)), flush=True)
        return
    if args.ncu_layer:
        run_one_layer_for_profiler()
        return
    if args.decode:
        print(json.dumps(run_decode(args)), flush=True)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    # CPU baseline first (before any CUDA work; the oracle uses OpenMP threads)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.cpu_layers)

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    result = run_ours(args, rank, world, local_rank)
    if rank == 0:
        result["cpu_baseline"] = cpu
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
