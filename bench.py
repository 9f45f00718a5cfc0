#!/usr/bin/env python3
"""Benchmark of the quantized MoE expert layer on GB300.

Metric: routed tokens/s per MoE layer (T / time per layer forward).  The
headline line is the largest configuration, the prefill chunk: H=2048, I=512,
E=512, top-10 + 1 shared expert, NVFP4 experts, T=4096 tokens per step.  A
step passes the tokens through a stack of L distinct layer instances (each its
own weights, so a step touches more than 4x the 129 MB L2), captured once as a
CUDA graph and replayed.  Inputs are resident in HBM before the timed region.

`per_config` times the other layer configurations in the same run, each the
same way: decode (T=1, NVFP4), decode of the larger expert shape (T=1, FP6
e2m3) and the batched decode step (T=64, NVFP4).

Also reported: the dominant kernel's (gate/up + SwiGLU) achieved FLOP rate
(prefill) or HBM bandwidth (the others) against the measured peak, the same
metric end to end through the host-buffer C-ABI call (moe_forward_host: copies
inside the timed region), SM clocks sampled during the timed region, and the
CPU oracle timed on the host cores on a bounded sample (one thread, and every
core).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs its own replicas (weak scaling: no
collective on the data path); the slowest rank's time counts.
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
sys.path.insert(0, ROOT)

METRIC = "routed tokens/s per MoE layer on 1 GB300; HBM GB/s as % of ~8 TB/s roofline"
UNIT = "tokens/s"
WORKLOAD = 4  # prefill-h2048-i512-e512-k10-s1-t4096-nvfp4: the largest config
PER_CONFIG = [1, 2, 3]  # decode NVFP4, decode FP6, batched T=64: timed in the same run
                        # (and the prefill with W4A4 activations)
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FP4_OVER_BF16 = 6.0  # nominal dense FP4 / bf16 tensor rate (13.5 / 2.25 PFLOP/s)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=None,
                    help="layer instances per step (default: enough that a step's weights are "
                         "more than 4x L2)")
    ap.add_argument("--workload", type=int, default=WORKLOAD,
                    help="workload index of the headline line (default: the prefill config)")
    ap.add_argument("--per-config", dest="per_config", action="store_true", default=True,
                    help="also time the decode, FP6 decode and batched configs (default)")
    ap.add_argument("--no-per-config", dest="per_config", action="store_false")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--act", choices=["bf16", "nvfp4"], default="bf16",
                    help="activations of the timed workload: bf16 (W4A16), or NVFP4 per row (W4A4)")
    ap.add_argument("--host-mirror", type=float, default=0.0,
                    help="fraction of each layer's experts placed in the pinned host mirror "
                         "(the coldest by router bias; the kernels read them over the CPU-GPU link)")
    return ap.parse_args()


def max_over_ranks(x, world):
    """The largest of the ranks' values of x (x itself on one rank): the job's
    time is its slowest rank's."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, tokens, layers, steps, seconds):
    """Whole-job throughput: every rank processes `steps` steps of `tokens`
    tokens through `layers` layer instances in (at most) `seconds`."""
    return world * tokens * layers * steps / seconds


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def peaks(kind="hbm"):
    """Roofline denominator: HBM copy GB/s, or dense bf16 TFLOP/s (burst: the
    kernel is timed alone; f16 runs at the bf16 rate on this tensor core)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        if kind == "tensor":
            return float(d["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst cuBLAS; f16 = bf16 rate)"
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, burst copy)"
    except Exception:
        if kind == "tensor":
            return FALLBACK_BF16_TFLOPS, "fallback 1.9 PFLOP/s (no MEASURED_PEAKS.json)"
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (no MEASURED_PEAKS.json)"


def packed_gateup_bytes(w):
    """Bytes of one expert's packed gate + up tiles (layout.cuh; MXFP4 is packed as NVFP4)."""
    if w.fmt in (1, 3):
        units = w.H // 64
        tile = 512 * ((units + 7) // 8 + units)
    else:
        units = w.H // 128
        tile = 128 * ((units + 7) // 8) + 1536 * units
    return (w.I // 16) * 2 * tile


def packed_down_bytes(w):
    """Bytes of one expert's packed down tiles (layout.cuh; MXFP4 is packed as NVFP4)."""
    if w.fmt in (1, 3):
        units = w.I // 64
        tile = 512 * ((units + 7) // 8 + units)
    else:
        units = w.I // 128
        tile = 128 * ((units + 7) // 8) + 1536 * units
    return (w.H // 16) * tile


def tc_path(w, T):
    """The forward takes the tcgen05 grouped GEMMs (NVFP4, >= 16 routed slots per expert)."""
    return w.fmt in (1, 3) and T * w.k >= 16 * w.E and w.H % 128 == 0 and (2 * w.I) % 128 == 0


FORMAT_NAMES = {1: "nvfp4 (e2m1, e4m3 per 16, fp32 tensor scale)",
                2: "fp6 e2m3 (power-of-two scale per 128)",
                3: "mxfp4 (e2m1, power-of-two scale per 32)"}
SHORT_NAMES = {1: "nvfp4", 2: "fp6 e2m3", 3: "mxfp4"}


def placement_mask(w, frac, seed):
    """HBM flags per expert (routed, then shared) with round(frac * n) experts in
    the host mirror: the coldest first by router bias (the routing-heat proxy a
    fresh layer has), ties by index; the always-used shared expert last."""
    import dataclasses

    import numpy as np

    import gen
    n = w.n_experts_total
    n_host = int(round(frac * n))
    if n_host <= 0:
        return None
    b = gen.router_bias(dataclasses.replace(w, seed=seed))
    heat = np.zeros(w.E) if b is None else b.astype(np.float64)
    order = list(np.argsort(heat, kind="stable")) + ([w.E] if w.shared else [])
    mask = np.ones(n, bool)
    mask[order[:n_host]] = False
    return mask


def link_peak_gbs(stream):
    """Host -> device bandwidth of the CPU-GPU link, measured here: a copy of a
    256 MiB pinned host buffer, best of 10 (CUDA events)."""
    import torch
    src = torch.empty(256 << 20, dtype=torch.uint8).pin_memory()
    dst = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    best = None
    with torch.cuda.stream(stream):
        for _ in range(12):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            dst.copy_(src, non_blocking=True)
            b.record(stream)
            b.synchronize()
            ms = a.elapsed_time(b)
            best = ms if best is None else min(best, ms)
    return src.numel() / (best * 1e-3) / 1e9


def config_block(w, L, extra=None):
    c = {"workload": w.name, "H": w.H, "I": w.I, "E": w.E, "k": w.k, "shared_experts": w.shared,
         "tokens_per_step": w.T,
         "format": FORMAT_NAMES[w.fmt],
         "layer_instances_per_step": L, "l2": "inputs larger than L2 (distinct weights per layer)"}
    if extra:
        c.update(extra)
    return c


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ["clocks.sm", "clocks.max.sm", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        self.rows = []

    def _one(self, loop):
        cmd = ["nvidia-smi", f"--query-gpu={','.join(self.FIELDS)}", "--format=csv,noheader,nounits"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        if loop:
            cmd += ["-lms", "100"]
        return cmd

    def start(self):
        try:
            self.rows += self._snap()
            self.proc = subprocess.Popen(self._one(True), stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def _snap(self):
        try:
            out = subprocess.run(self._one(False), capture_output=True, text=True, timeout=10).stdout
            return [l for l in out.splitlines() if l.strip()]
        except Exception:
            return []

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
                self.rows += [l for l in out.splitlines() if l.strip()]
            except Exception:
                self.proc.kill()
        self.rows += self._snap()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle baseline
def _oracle_setup(w, n_tok=4):
    import gen
    import oracle
    oracle.build()
    gen.build(device=False)
    x = gen.x_tokens(w, n_tok)
    base = oracle.Layer(w.fmt, w.H, w.I, w.E, w.k, w.shared, gen.router_weights(w),
                        gen.router_bias(w))
    idx, _ = base.topk(base.logits(x))
    need = sorted(set(idx.ravel().tolist()) | ({w.E} if w.shared else set()))
    return x, idx, oracle.layer_for_workload(w, need)


def oracle_baseline(w, seconds):
    """The oracle as it stands, on a bounded sample of the workload: whole-layer
    forwards (router, top-k, the k + shared expert FFNs, combine) of the
    workload's first tokens, its weights quantised by the oracle beforehand
    (not timed).  Timed twice for about seconds/2 each: one token per call on
    one thread, and one token per host core per call, the oracle threading
    over tokens on every core."""
    cores = os.cpu_count() or 1
    x, _, L = _oracle_setup(w, n_tok=max(4, cores))

    def rate(n, threads, budget):
        t0 = time.perf_counter()
        calls = 0
        while True:
            i = (calls * n) % len(x)
            xs = x[i:i + n] if i + n <= len(x) else x[:n]
            L.forward(xs, threads=threads)
            calls += 1
            if time.perf_counter() - t0 >= budget:
                break
        dt = time.perf_counter() - t0
        return calls * n / dt, calls, dt

    v1, c1, d1 = rate(1, 1, seconds / 2)
    va, ca, da = rate(cores, cores, seconds / 2)
    return {"value": va, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{ca} whole-layer forwards of {cores} tokens of {w.name} ({da:.1f} s, fp64, "
                      f"threaded over tokens on {cores} host cores)",
            "single_thread": {"value": v1, "unit": UNIT, "cores": 1,
                              "sample": f"{c1} single-token forwards ({d1:.1f} s, fp64, 1 thread)"}}


def run_reference(args, w):
    """Reference arm: the CPU oracle (there is no other implementation of this
    path).  A step is one bounded slice of the workload: one (token, expert)
    SwiGLU FFN; a token-layer costs (k + shared) slices plus one router pass,
    which is timed during warm-up and folded into the rate."""
    rank, _, world = dist_env()
    if rank != 0:
        return
    x, idx, L = _oracle_setup(w)
    n_slices = w.k + w.shared
    experts = [(t, int(idx[t, j]) if j < w.k else w.E) for t in range(len(x)) for j in range(n_slices)]
    tr = []
    for i in range(max(3, args.warmup)):
        t0 = time.perf_counter()
        L.logits(x[i % len(x): i % len(x) + 1])
        tr.append(time.perf_counter() - t0)
    t_router = statistics.median(tr)
    for i in range(args.warmup):
        t, e = experts[i % len(experts)]
        L.expert_ffn(e, x[t:t + 1])
    t0 = time.perf_counter()
    for i in range(args.steps):
        t, e = experts[i % len(experts)]
        L.expert_ffn(e, x[t:t + 1])
    dt = time.perf_counter() - t0
    t_step = dt / args.steps
    value = 1.0 / (n_slices * t_step + t_router)
    sample = (f"{args.steps} (token, expert) SwiGLU slices of {w.name}; token-layer = "
              f"{n_slices} slices + router ({t_router * 1e3:.2f} ms); fp64, 1 thread")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded generator)",
            "config": config_block(w, 1, {"reference": "CPU oracle (the pages hold no runnable "
                                                       "implementation of this path)"}),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def traffic_from_profile(kernel, workload, csrc):
    """dram bytes per launch of `kernel` on `workload` from its committed ncu
    summary, or None when the kernel's sources changed since the capture (the
    summary records the translation unit that defines the kernel and a hash of
    it and every header it includes)."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        txt = open(p).read()
        sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", txt).group(1)
        unit = re.search(r"source_unit:\s*(\S+)", txt).group(1)
        b = float(re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt).group(1))
    except Exception:
        return None
    return b if sources_sha256(csrc, unit) == sha else None


def prefill_flops(w, counts):
    """FLOPs of the tensor-core gate/up GEMM for per-expert token counts: the
    routed (token, expert) pairs and the shared experts' T tokens, 2 n 2I H
    each; and the FLOPs as the MMA runs them (each work item of at most 128
    tokens padded to a multiple of 16)."""
    n = [int(v) for v in counts if v > 0] + [w.T] * w.shared
    algo = 2.0 * sum(n) * 2 * w.I * w.H
    cols = sum(((min(128, v - 128 * j) + 15) // 16) * 16 for v in n for j in range((v + 127) // 128))
    return algo, 2.0 * cols * 2 * w.I * w.H


def sources_sha256(csrc, unit):
    """Hash of the translation unit `unit` and the local headers it includes,
    followed recursively, in sorted file-name order."""
    seen, todo = set(), [unit]
    while todo:
        f = todo.pop()
        if f in seen:
            continue
        seen.add(f)
        txt = open(os.path.join(csrc, f)).read()
        todo += re.findall(r'^#include "([^"/]+)"', txt, re.M)
    h = hashlib.sha256()
    for f in sorted(seen):
        h.update(f.encode())
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()


# ---------------------------------------------------------------- our arm
def no_launch_phases(L, T):
    """Phases of moe_debug_run_phase that launch nothing at T tokens: for the
    self-routed path (3 kernels) top-k/dispatch and combine live inside the
    expert kernels; for the other T <= 8 paths the combine is fused."""
    n = L.launches(T)
    if n == 3:
        return {1, 4}
    if T <= 8:
        return {4}
    return set()


def graph_time_us(s, fn, reps, warm=3):
    """Average time of one fn() call: fn captured once into a CUDA graph,
    replayed warm + reps times, CUDA events on the capture stream."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        for _ in range(warm):
            g.replay()
        e0.record(s)
        for _ in range(reps):
            g.replay()
        e1.record(s)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / reps


def measure(w, Ln, steps, warmup, rank, world, host_mirror=0.0, headline=False, act=0):
    """Builds Ln layer instances of workload w, captures one step (the T
    tokens through the Ln layers) as a CUDA graph and times `steps` replays
    after `warmup` (CUDA events, max over ranks).  Also times the dominant
    kernel alone, each phase alone, and (headline) the host-buffer call."""
    import numpy as np
    import torch

    import gen
    from quantized_moe_expert_layer_gb300.synthetic import build_layer

    T = w.T
    masks = [placement_mask(w, host_mirror, 1000 * rank + i) for i in range(Ln)]
    layers = [build_layer(w, T_max=T, seed=1000 * rank + i, in_hbm=masks[i]) for i in range(Ln)]
    for L in layers:
        L.set_act_format(act)
    x_np = gen.x_tokens(w, T, first=rank * T)
    x = torch.from_numpy(x_np.view(np.int16)).cuda()
    outs = [torch.empty((T, w.H), dtype=torch.float32, device="cuda") for _ in range(Ln)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for L, o in zip(layers, outs):
            L.forward(x, o, stream=s)
    s.synchronize()
    for L in layers:
        if L.status() != 0:
            raise RuntimeError("device status word set after warm-up forward")

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for L, o in zip(layers, outs):
            L.forward(x, o, stream=s)
    ref_outs = [o.clone() for o in outs]
    with torch.cuda.stream(s):
        for o in outs:
            o.zero_()
        g.replay()
    s.synchronize()
    for o, r in zip(outs, ref_outs):
        if not torch.equal(o, r):
            raise RuntimeError("graph replay differs from the eager forward")
    with torch.cuda.stream(s):
        for _ in range(warmup):
            g.replay()
    s.synchronize()

    clocks = None
    if headline:
        uuid = None
        try:
            uuid = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
            if not uuid.startswith("GPU-"):
                uuid = "GPU-" + uuid
        except Exception:
            uuid = None
        clocks = ClockSampler(uuid)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):  # replay() launches on the current stream
        ev0.record(s)
        for _ in range(steps):
            g.replay()
        ev1.record(s)
    torch.cuda.synchronize()
    if clocks:
        clocks.stop()
    if world > 1:
        dist.barrier()
    ms = max_over_ranks(ev0.elapsed_time(ev1), world)
    res = {"value": job_rate(world, T, Ln, steps, ms / 1e3), "ms": ms,
           "us_per_layer": ms * 1e3 / (steps * Ln), "launches_per_layer": layers[0].launches(T)}
    if clocks:
        res["clocks"] = clocks.summary()

    # dominant kernel (gate/up + SwiGLU) alone over the L layers (graph of
    # back-to-back launches, launch gaps included): the tcgen05 GEMM for
    # prefill (tensor-bound) or the streaming kernel otherwise (HBM-bound)
    counts = torch.empty(w.E, dtype=torch.int32, device="cuda")
    tc = tc_path(w, T)
    gu = packed_gateup_bytes(w)
    dn = packed_down_bytes(w)
    per_launch, padded, host_per_launch, fq_bytes = [], [], [], []
    # for T <= 8 (NVFP4) gate/up also asks L2 for the touched experts' down
    # matrices, which the down kernel then reads from L2
    prefetch_down = T <= 8 and w.fmt in (1, 3)
    with torch.cuda.stream(s):
        for L, o, m in zip(layers, outs, masks):
            L.forward(x, o, stream=s)
            L.debug_routing(counts=counts, stream=s)
            s.synchronize()
            c = counts.cpu().numpy()
            D = int((c > 0).sum()) + w.shared
            if m is not None:  # weight bytes of the touched experts in the host mirror
                used = np.concatenate([c > 0, [True] * w.shared])
                host_per_launch.append(int((used & ~m).sum()) * (gu + (dn if prefetch_down else 0)))
            if tc:  # FLOPs of the contraction: the routed (token, expert) pairs as computed,
                # and as the MMA runs them (N padded to 16 per work item of <= 128 tokens)
                n = [int(v) for v in c if v > 0] + [T] * w.shared
                algo, as_run = prefill_flops(w, c)
                per_launch.append(algo)
                padded.append(as_run)
                # bytes of the block-scaled (W4A4) launch: the touched experts' packed gate/up
                # tiles, x's NVFP4 codes and scales, a written in fp32
                fq_bytes.append(D * gu + T * w.H * 9 // 16 + sum(n) * w.I * 4)
            else:  # unique weight bytes, x, and a (+ the down matrices it pulls into L2)
                per_launch.append(D * (gu + 8 + (dn if prefetch_down else 0)) + T * w.H * 2
                                  + (T * w.k + T * w.shared) * w.I * 2)

    def run_gateup():
        for L, o in zip(layers, outs):
            L.run_phase(2, x, o, stream=s)
    # (the token rows in slot order again: on the W4A16 tensor-core path they
    # share their buffer with y, which the last forward's down phase wrote)
    with torch.cuda.stream(s):
        for L, o in zip(layers, outs):
            L.run_phase(1, x, o, stream=s)
    # (30 replays, as the per-phase times: a seconds-long loop of the dense
    # GEMM drops the SM clock under the power cap, which the sustained peak covers)
    k_us = graph_time_us(s, run_gateup, 30) / Ln
    work = sum(per_launch) / len(per_launch)
    if tc and act:
        # the block-scaled FP4 GEMM: HBM-bound at these token counts (its FLOPs
        # at the FP4 rate take a fraction of the time its weight bytes take)
        kname = "tc_fp4_kernel"
        peak, peak_kind = peaks("hbm")
        tpeak, tpeak_kind = peaks("tensor")
        fp4_peak = tpeak * FP4_OVER_BF16
        fb = sum(fq_bytes) / len(fq_bytes)
        achieved = fb / (k_us * 1e-6) / 1e9
        t_flops = work / (k_us * 1e-6) / 1e12
        roofline = {"bound": "hbm", "kernel": kname + "<0> (gate/up + SwiGLU, kind::mxf4nvf4)",
                    "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                    "algorithmic_bytes_per_launch": fb,
                    "tensor": {"achieved": t_flops, "peak": fp4_peak, "unit": "TFLOP/s",
                               "frac": t_flops / fp4_peak, "algorithmic_flops_per_launch": work,
                               "peak_source": tpeak_kind + " x 6 (nominal dense FP4 / bf16: "
                                                           "13.5 / 2.25 PFLOP/s)"},
                    "note": "bytes: the touched experts' packed gate/up tiles, x's NVFP4 codes "
                            "and scales, a written in fp32 for its quantiser"}
    elif tc:
        kname = "tc_tmem_kernel" if w.H % 128 == 0 and w.I % 128 == 0 else "tc_expert_kernel"
        peak, peak_kind = peaks("tensor")
        achieved = work / (k_us * 1e-6) / 1e12
        pw = sum(padded) / len(padded)
        roofline = {"bound": "tensor", "kernel": kname + "<0> (gate/up + SwiGLU)",
                    "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                    "algorithmic_flops_per_launch": work,
                    "flops_as_run_per_launch": pw,
                    "note": "algorithmic FLOPs count the routed (token, expert) pairs; the MMA "
                            "also runs the padding of each work item to a multiple of 16 tokens "
                            "(flops_as_run_per_launch)"}
    else:
        kname = ("gateup_routed_kernel" if T <= 8 else
                 "stream_kernel<0>" if w.fmt in (1, 3) else "gateup_kernel")
        peak, peak_kind = peaks("hbm")
        achieved = work / (k_us * 1e-6) / 1e9
        roofline = {"bound": "hbm", "kernel": kname + " (gate/up + SwiGLU)", "achieved": achieved,
                    "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                    "algorithmic_bytes_per_launch": work}
    if host_per_launch:  # the CPU-GPU link bounds the mirrored experts' share
        hb = sum(host_per_launch) / len(host_per_launch)
        lp = link_peak_gbs(s)
        achieved = hb / (k_us * 1e-6) / 1e9
        roofline = {"bound": "link", "kernel": kname + " (gate/up + SwiGLU)", "achieved": achieved,
                    "peak": lp, "unit": "GB/s", "frac": achieved / lp,
                    "algorithmic_bytes_per_launch": hb,
                    "hbm_bytes_per_launch": work - hb,
                    "note": "bytes read from the pinned host mirror over the CPU-GPU link"}
        peak_kind = "measured here: 256 MiB pinned host -> device copy, best of 10"
    roofline.update({"traffic": None if host_per_launch else traffic_from_profile(
                         kname.split("<")[0], w.name + ("-w4a4" if act else ""),
                         os.path.join(ROOT, "quantized_moe_expert_layer_gb300", "csrc")),
                     "avg_launch_us": k_us, "peak_source": peak_kind,
                     "timing": "CUDA events over a graph of back-to-back launches, gaps included"})
    res["roofline"] = roofline
    res["hbm_gbs_layer"] = None if tc else (
        (work + (D * dn if not prefetch_down else 0)) / (res["us_per_layer"] * 1e-6) / 1e9)

    # steady-state time of each phase alone (graphs of L back-to-back launches);
    # phases that launch nothing at this T are null
    skip = no_launch_phases(layers[0], T)
    phase_us = {}
    for ph, name in [(0, "routing"), (1, "topk_dispatch"), (2, "gate_up"), (3, "down"), (4, "combine")]:
        if ph in skip:
            phase_us[name] = None
            continue

        def run_ph(ph=ph):
            for L, o in zip(layers, outs):
                L.run_phase(ph, x, o, stream=s)
        phase_us[name] = graph_time_us(s, run_ph, 30) / Ln
    res["phase_us_alone"] = phase_us

    if headline:
        # e2e: the host-buffer C-ABI call, copies inside the timed region
        xh = torch.from_numpy(x_np.view(np.int16)).pin_memory()
        ohs = [torch.empty((T, w.H), dtype=torch.float32).pin_memory() for _ in range(Ln)]
        for L, oh in zip(layers, ohs):
            L.forward_host(xh, oh, stream=s)
        k_e2e = max(3, min(steps, 20 if T > 8 else 100))
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(k_e2e):
            for L, oh in zip(layers, ohs):
                L.forward_host(xh, oh, stream=s)
        e2e_dt = max_over_ranks(time.perf_counter() - t0, world)
        res["e2e"] = {"value": job_rate(world, T, Ln, k_e2e, e2e_dt), "unit": UNIT,
                      "h2d_bytes_per_step": Ln * T * w.H * 2, "d2h_bytes_per_step": Ln * T * w.H * 4,
                      "call": "moe_forward_host per layer (pinned host buffers, read and written in "
                              "place by the kernels over the CPU-GPU link; synchronous)"}
    for L in layers:
        L.close()
    del layers, outs
    torch.cuda.empty_cache()
    return res


def default_layers(w, host_mirror=0.0):
    """Layer instances per step: enough distinct weights that a step touches
    more than 4x the 129 MB L2 (each instance its own arena)."""
    if w.T <= 8:
        if w.fmt == 2:
            return 4           # 4 x 260 MB touched
        return 16 if host_mirror > 0 else 32   # 32 x 21.6 MB (decode), 32 x 44 MB (DeepSeek shape)
    return 4 if w.T <= 64 else 8   # batched: 4 x 650 MB; prefill: 8 x 960 MB


def run_ours(args, w):
    import torch

    import gen
    import quantized_moe_expert_layer_gb300 as moe

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    gen.build(device=True)
    moe.build()
    Ln = args.layers or default_layers(w, args.host_mirror)
    act = 1 if args.act == "nvfp4" else 0
    r = measure(w, Ln, args.steps, args.warmup, rank, world, args.host_mirror, headline=True, act=act)
    per_config = {}
    if args.per_config:
        # the other configurations, then the headline's shape with W4A4 activations
        for idx, act_c in [(i, 0) for i in PER_CONFIG] + [(WORKLOAD, 1)]:
            wc = gen.get_workload(idx)
            if wc.name == w.name and act_c == act:
                continue
            Lc = default_layers(wc)
            # each config's timed region: about a second of replays
            one = measure(wc, Lc, max(20, args.warmup), 3, rank, world, act=act_c)
            steps_c = max(20, min(5000, int(1.0 / max(one["ms"] * 1e-3 / max(20, args.warmup), 1e-6))))
            rc = measure(wc, Lc, steps_c, 3, rank, world, act=act_c)
            per_config[wc.name + ("-w4a4" if act_c else "")] = {
                "activations": "nvfp4 per row (W4A4)" if act_c else "bf16 x, fp32 a (W4A16)",
                "tokens_per_step": wc.T, "layer_instances_per_step": Lc, "steps": steps_c,
                "value": rc["value"], "unit": UNIT, "us_per_layer": rc["us_per_layer"],
                "format": SHORT_NAMES[wc.fmt], "gpu_launches_per_layer": rc["launches_per_layer"],
                "roofline": rc["roofline"], "hbm_gbs_whole_layer": rc["hbm_gbs_layer"],
                "phase_us_alone": rc["phase_us_alone"]}

    line = {"metric": METRIC, "value": r["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": r["ms"] / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": ("e2m1 x e2m1 -> f32 with e4m3 block scales (W4A4: x and a quantised to "
                      "NVFP4 per row; kind::mxf4nvf4 where the tensor-core path runs)") if act else
                     ("f16 x f16 -> f32 (" + SHORT_NAMES[w.fmt] + " weights dequantised exactly to "
                      "f16; bf16 x copied exactly to f16)"),
            "data": "synthetic (seeded generator; random-init weights quantised on the device)",
            "config": config_block(w, Ln, {"us_per_layer": r["us_per_layer"],
                                           "host_mirror_fraction": args.host_mirror,
                                           "activations": "nvfp4 per row (W4A4)" if act else
                                                          "bf16 x, fp32 a (W4A16)",
                                           "phase_us_alone": r["phase_us_alone"],
                                           "parallelism": f"replicas x{world}"}),
            "roofline": r["roofline"], "e2e": r["e2e"],
            "gpu_launches": r["launches_per_layer"] * Ln * args.steps,
            "clocks": r["clocks"]}
    if per_config:
        line["per_config"] = per_config
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_baseline(w, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    import gen
    w = gen.get_workload(args.workload)
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
