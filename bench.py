#!/usr/bin/env python3
"""Benchmark of the quantized MoE expert layer on GB300.

Metric: routed tokens/s per MoE layer (T / time per layer forward), on the
decode workload H=2048, I=512, E=512, top-10 + 1 shared expert, NVFP4
experts, T=1 token per step.  A step passes the token through a stack of L
distinct layer instances (default 32; each its own weights, so the 32 x 21.6
MB touched per step are far larger than the 129 MB L2), captured once as a
CUDA graph and replayed.  Inputs are resident in HBM before the timed region.

Also reported: the dominant kernel's (gate/up + SwiGLU) achieved HBM bandwidth
against the measured copy bandwidth, the same metric end to end through the
host-buffer C-ABI call (moe_forward_host: copies inside the timed region), SM
clocks sampled during the timed region, and the CPU oracle timed on the host
cores on a bounded sample.

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
WORKLOAD = 1  # decode-h2048-i512-e512-k10-s1-t1-nvfp4
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=None,
                    help="layer instances per step (default 32 for decode, 8 for larger T)")
    ap.add_argument("--workload", type=int, default=WORKLOAD,
                    help="workload index (default: the decode workload the metric is quoted on)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
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
    """The oracle as it stands: whole-layer forwards of single decode tokens (its
    weights quantised by the oracle beforehand, not timed), for ~`seconds`.
    A T=1 forward runs on one thread (the oracle threads over tokens)."""
    x, _, L = _oracle_setup(w)
    t0 = time.perf_counter()
    reps = 0
    while True:
        L.forward(x[reps % len(x): reps % len(x) + 1], threads=1)
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": reps / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{reps} single-token forwards of {w.name} ({dt:.1f} s, fp64, 1 thread)"}



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
def run_ours(args, w):
    import numpy as np
    import torch

    import gen
    import quantized_moe_expert_layer_gb300 as moe
    from quantized_moe_expert_layer_gb300.synthetic import build_layer

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    gen.build(device=True)
    moe.build()
    Ln = args.layers
    T = w.T
    masks = [placement_mask(w, args.host_mirror, 1000 * rank + i) for i in range(Ln)]
    layers = [build_layer(w, T_max=T, seed=1000 * rank + i, in_hbm=masks[i]) for i in range(Ln)]
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

    # one step = the token through the L layer instances, as one CUDA graph
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
        for _ in range(args.warmup):
            g.replay()
    s.synchronize()

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(local_rank).uuid)
        if not uuid.startswith("GPU-"):
            uuid = "GPU-" + uuid
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):  # replay() launches on the current stream
        ev0.record(s)
        for _ in range(args.steps):
            g.replay()
        ev1.record(s)
    torch.cuda.synchronize()
    clocks.stop()
    if world > 1:
        dist.barrier()
    ms = max_over_ranks(ev0.elapsed_time(ev1), world)
    value = job_rate(world, T, Ln, args.steps, ms / 1e3)

    # dominant kernel, timed alone over the L layers (graph of back-to-back
    # launches, launch gaps included): gate/up + SwiGLU, the tcgen05 GEMM for
    # prefill (tensor-bound) or the streaming kernel otherwise (HBM-bound)
    counts = torch.empty(w.E, dtype=torch.int32, device="cuda")
    tc = tc_path(w, T)
    gu = packed_gateup_bytes(w)
    per_launch = []
    host_per_launch = []
    # for T <= 8 (NVFP4) gate/up also asks L2 for the touched experts' down
    # matrices, which the down kernel then reads from L2
    prefetch_down = T <= 8 and w.fmt in (1, 3)
    dn = packed_down_bytes(w)
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
            if tc:  # FLOPs of the contraction (N padded to 16 per work item as the MMA runs it)
                n = [int(v) for v in c if v > 0] + [T] * w.shared
                cols = sum(((min(128, v - 128 * j) + 15) // 16) * 16
                           for v in n for j in range((v + 127) // 128))
                per_launch.append(2.0 * cols * 2 * w.I * w.H)
            else:  # unique weight bytes, x, and a (+ the down matrices it pulls into L2)
                per_launch.append(D * (gu + 8 + (dn if prefetch_down else 0)) + T * w.H * 2
                                  + (T * w.k + T * w.shared) * w.I * 2)
    gk = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gk, stream=s):
        for L, o in zip(layers, outs):
            L.run_phase(2, x, o, stream=s)
    reps = max(20, min(500, args.steps))
    k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        for _ in range(5):
            gk.replay()
        k0.record(s)
        for _ in range(reps):
            gk.replay()
        k1.record(s)
    torch.cuda.synchronize()
    k_us = k0.elapsed_time(k1) * 1e3 / (reps * Ln)
    work = sum(per_launch) / len(per_launch)
    if tc:
        kname = "tc_expert_kernel"
        peak, peak_kind = peaks("tensor")
        achieved = work / (k_us * 1e-6) / 1e12
        roofline = {"bound": "tensor", "kernel": kname + "<0> (gate/up + SwiGLU)", "achieved": achieved,
                    "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                    "algorithmic_flops_per_launch": work}
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
                         kname.split("<")[0], w.name, os.path.join(ROOT, "quantized_moe_expert_layer_gb300", "csrc")),
                     "avg_launch_us": k_us, "peak_source": peak_kind,
                     "timing": "CUDA events over a graph of back-to-back launches, gaps included"})

    # steady-state time of each phase alone (graphs of L back-to-back launches)
    phase_us = {}
    for ph, name in [(0, "routing"), (1, "topk_dispatch"), (2, "gate_up"), (3, "down"), (4, "combine")]:
        gp = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gp, stream=s):
            for L, o in zip(layers, outs):
                L.run_phase(ph, x, o, stream=s)
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            for _ in range(3):
                gp.replay()
            p0.record(s)
            for _ in range(50):
                gp.replay()
            p1.record(s)
        torch.cuda.synchronize()
        phase_us[name] = p0.elapsed_time(p1) * 1e3 / (50 * Ln)

    # e2e: the host-buffer C-ABI call, copies inside the timed region
    xh = torch.from_numpy(x_np.view(np.int16)).pin_memory()
    ohs = [torch.empty((T, w.H), dtype=torch.float32).pin_memory() for _ in range(Ln)]
    for L, oh in zip(layers, ohs):
        L.forward_host(xh, oh, stream=s)
    k_e2e = max(5, min(args.steps, 100))
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(k_e2e):
        for L, oh in zip(layers, ohs):
            L.forward_host(xh, oh, stream=s)
    e2e_dt = max_over_ranks(time.perf_counter() - t0, world)
    e2e = {"value": job_rate(world, T, Ln, k_e2e, e2e_dt), "unit": UNIT,
           "h2d_bytes_per_step": Ln * T * w.H * 2, "d2h_bytes_per_step": Ln * T * w.H * 4,
           "call": "moe_forward_host per layer (pinned host buffers, read and written in place "
                   "by the kernels over the CPU-GPU link; synchronous)"}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16 x f16 -> f32 (" + SHORT_NAMES[w.fmt] + " weights)",
            "data": "synthetic (seeded generator; random-init weights quantised on the device)",
            "config": config_block(w, Ln, {"us_per_layer": ms * 1e3 / (args.steps * Ln),
                                           "host_mirror_fraction": args.host_mirror,
                                           "phase_us_alone": phase_us,
                                           "parallelism": f"replicas x{world}"}),
            "roofline": roofline, "e2e": e2e, "gpu_launches": layers[0].launches(T) * Ln * args.steps,
            "clocks": clocks.summary()}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_baseline(w, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    for L in layers:
        L.close()
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    import gen
    w = gen.get_workload(args.workload)
    if args.layers is None:
        # (16 decode instances with a host mirror: 14.5 GB pinned at most)
        args.layers = (16 if args.host_mirror > 0 else 32) if w.T <= 8 else 8
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
