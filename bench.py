#!/usr/bin/env python3
"""Benchmark of the NVFP4 weight-only linear with LoRA and AQN on GB300.

One step = one rollout decode pass of a Qwen2.5-7B-shaped decoder layer's
seven LoRA linears (q, k, v, o, gate, up, down; r = 32, alpha = 64) at each
decode batch M in {1, 8, 32, 128}: per M, the AQN noise of the four groups
(qkv, o, gate_up, down; one sampler launch; sigma from the exponential-decay
schedule, stage = step mod 10) and the seven linears as four grouped launches
({q,k,v}, {o}, {gate,up}, {down}; --ungrouped: seven single calls).  Inputs are synthetic and seeded; the
weights are NVFP4-quantized by the library from fp32 N(0, 0.02^2) with 0.5% of
input channels scaled x10.  Weights rotate over 8 distinct layer copies
(1.05 GB, far above the 129 MB L2), so every linear streams its weights from
HBM.  Each (stage, M) sub-step is one CUDA graph replay.

`value` is decode throughput in GB/s of NVFP4 weight bytes (0.5625 B per
weight: E2M1 code + E4M3 scale share) over the timed steps.  Also reported:
prefill TFLOP/s (Qwen2.5-14B-shaped layer, M = 4096), quantizer GB/s, an
end-to-end figure through the public API with host buffers, the roofline of
the decode path's largest launch, the oracle timed on host cores, and SM
clocks sampled during the timed region.  Unless --skip-extra: a single
Qwen2.5-3B q_proj at M = 4 (weights hot and cold in L2), 8192 sustained
decode steps through a 28-layer 7B-shaped stack at M in {8, 64, 128} (z
resampled every step, sigma decaying over the run),
and the Qwen2.5-32B-shaped 64-layer weight stream (one M = 16 step through all
448 linears, whose quantization from heavy-tailed bf16 is timed too).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun with N > 1 every rank runs the same workload on its own GPU
(independent replicas, weak scaling); the timed region is bracketed by a
barrier, and the max over ranks is reported.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "NVFP4+LoRA linear: decode HBM GB/s (% of peak); prefill TFLOP/s (% of peak)"
UNIT = "GB/s"
DECODE_MS = (1, 8, 32, 128)
RANK_R = 32
ALPHA = 64.0
NUM_STAGES = 10
SIGMA_START, SIGMA_END = 1e-2, 5e-4
N_COPIES = 8
BYTES_PER_WEIGHT = 0.5625
WORKLOAD = ("Qwen2.5-7B decoder-layer linears q,k,v,o,gate,up,down (N x K: 3584x3584, 512x3584 x2, "
            "3584x3584, 18944x3584 x2, 3584x18944), decode M in {1,8,32,128}, LoRA r=32 alpha=64, "
            "AQN sigma by exponential decay 1e-2 -> 5e-4 over 10 stages (stage = step mod 10)")


# ---------------------------------------------------------------- environment

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# Arm CPU identification: (implementer, part) from /proc/cpuinfo -> core name
# (Arm's published MIDR part numbers).
ARM_PARTS = {(0x41, 0xD0C): "Neoverse-N1", (0x41, 0xD40): "Neoverse-V1", (0x41, 0xD49): "Neoverse-N2",
             (0x41, 0xD4F): "Neoverse-V2", (0x41, 0xD8E): "Neoverse-N3", (0x41, 0xD84): "Neoverse-V3"}


EXTRAS = ("prefill", "quantize", "qproj", "sustained", "32b", "mxfp4", "nf4", "backward")


def host_cpu_model():
    """The host CPU's model name: /proc/cpuinfo's "model name" (x86), else the Arm core named
    from its "CPU implementer" / "CPU part" fields (raw values kept), else the platform string."""
    impl = part = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key, _, val = line.partition(":")
                key, val = key.strip().lower(), val.strip()
                if key in ("model name", "cpu model"):
                    return val
                if key == "cpu implementer" and impl is None:
                    impl = int(val, 0)
                elif key == "cpu part" and part is None:
                    part = int(val, 0)
    except (OSError, ValueError):
        pass
    if impl is not None and part is not None:
        name = ARM_PARTS.get((impl, part), "Arm core")
        return f"{name} (CPU implementer {impl:#x}, part {part:#05x})"
    import platform
    return platform.processor() or platform.machine()


def max_over_ranks(x, world, device):
    """The largest of every rank's x, returned on every rank (x itself for one process):
    the job's time is its slowest replica's."""
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item()


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi sampled every 100 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) >= 9:
                    rows.append(p)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(power) if power else None, "samples": len(rows), "reasons": reasons}


# ---------------------------------------------------------------- workload

class QLinear:
    """One NVFP4-quantized linear with its LoRA adapters (device)."""

    def __init__(self, q, lin, seed, *path, r=RANK_R, w_dtype=torch.float32, fmt="nvfp4"):
        W = wl.weight_f32_device(lin.n, lin.k, seed, *path)
        if w_dtype == torch.bfloat16:
            W = W.to(torch.bfloat16)
        self.lin = lin
        self.w_format = q.QERL_W_NF4 if fmt == "nf4" else q.QERL_W_NVFP4
        if fmt == "mxfp4":
            codes, scales = q.mxfp4_quantize(W)
            self.wp, self.S = q.mxfp4_pack(codes, scales)
        elif fmt == "nf4":
            codes, scales, self.S = q.nf4_quantize(W)
            self.wp = q.pack(codes, scales)
        else:
            codes, scales, self.S = q.quantize(W)
            self.wp = q.pack(codes, scales)
        del codes, scales
        del W
        self.A = wl.normal_bf16_device((r, lin.k), 1.0 / math.sqrt(lin.k), seed, *path, 2)
        self.B = wl.normal_bf16_device((lin.n, r), 0.01, seed, *path, 3)

    @property
    def weight_bytes(self):
        return self.lin.n * self.lin.k * BYTES_PER_WEIGHT


def layer_weights(q, shapes, seed, copy):
    return [QLinear(q, lin, seed, copy, li) for li, lin in enumerate(shapes)]


class Activations:
    """Per-M inputs (one x and one z per AQN group), outputs and a workspace.  The
    inputs are views of one buffer and the outputs views of another, so a step's
    host copies are one transfer each way."""

    def __init__(self, q, shapes, m, seed):
        self.m = m
        ks = {}
        for lin in shapes:
            ks[lin.group] = lin.k
        self.x_all = torch.empty(m * sum(ks.values()), dtype=torch.bfloat16, device="cuda")
        self.x, off = {}, 0
        for gi, (g, k) in enumerate(ks.items()):
            self.x[g] = self.x_all[off:off + m * k].view(m, k)
            self.x[g].copy_(wl.normal_bf16_device((m, k), 1.0, seed, m, gi, 11))
            off += m * k
        # one noise buffer for the layer; each AQN group is a 16-byte aligned slice of it
        self.z_all = torch.zeros(sum(ks.values()), dtype=torch.float32, device="cuda")
        self.z, off = {}, 0
        for g, k in ks.items():
            self.z[g] = self.z_all[off:off + k]
            off += k
        self.y_all = torch.empty(m * sum(lin.n for lin in shapes), dtype=torch.bfloat16, device="cuda")
        self.y, off = [], 0
        for lin in shapes:
            self.y.append(self.y_all[off:off + m * lin.n].view(m, lin.n))
            off += m * lin.n
        need = max(q.qerl_lora_linear_workspace_size(m, lin.n, lin.k, RANK_R) for lin in shapes)
        # a group of up to three rank-RANK_R linears needs room for three LoRA partial sums
        need += 2 * q.qerl_lora_linear_workspace_size(m, 0, max(lin.k for lin in shapes), RANK_R)
        self.ws = q.workspace(need)

    def io_bytes(self):
        return self.x_all.numel() * self.x_all.element_size(), self.y_all.numel() * self.y_all.element_size()

    def group_descs(self, q, layer):
        """Per AQN group: (x, z, descriptor array) of its grouped launch on this layer."""
        out = []
        for g in wl.NOISE_GROUPS:
            members = [(ql.wp, ql.S, ql.A, ql.B, ALPHA, y) for ql, y in zip(layer, self.y) if ql.lin.group == g]
            out.append((self.x[g], self.z[g], q.linear_descs(members)))
        return out


# Linears of one input run as one grouped launch: {q,k,v}, {o}, {gate,up}, {down}.
GROUPED = True


def run_substep(q, layer, act, sigma, counter):
    """One decode batch through the layer: the AQN noise of all four groups (one sampler
    launch over the concatenated channels) + the 7 linears (4 grouped launches, or 7
    single calls), all on the current stream."""
    q.check(q.qerl_aqn_sample(act.z_all, sigma, 0, 0, counter), "qerl_aqn_sample")
    if not GROUPED:
        for ql, y in zip(layer, act.y):
            g = ql.lin.group
            q.check(q.qerl_lora_linear(act.x[g], ql.wp, ql.S, act.z[g], ql.A, ql.B, ALPHA, y, act.ws),
                    "qerl_lora_linear")
        return
    for g in wl.NOISE_GROUPS:
        members = [(ql.wp, ql.S, ql.A, ql.B, ALPHA, y, ql.w_format) for ql, y in zip(layer, act.y)
                   if ql.lin.group == g]
        q.check(q.qerl_lora_linear_group(act.x[g], act.z[g], members, act.ws), "qerl_lora_linear_group")


def linear_algorithmic_bytes(lin, m, r=RANK_R):
    """Minimum HBM/L2 bytes of one linear call: weights + x + z + y + LoRA adapters."""
    return (lin.n * lin.k * BYTES_PER_WEIGHT + m * lin.k * 2 + lin.k * 4 + m * lin.n * 2
            + lin.k * r * 2 + r * lin.n * 2)


def linear_flops(lin, m, r=RANK_R):
    return 2.0 * m * lin.n * lin.k + 2.0 * m * lin.k * r + 2.0 * m * r * lin.n


def group_algorithmic_bytes(lins, m, r=RANK_R):
    """Minimum HBM/L2 bytes of one grouped launch: every member's weights, output and
    LoRA adapters, plus the shared input x and noise z once."""
    k = lins[0].k
    return (sum(l.n * l.k * BYTES_PER_WEIGHT + m * l.n * 2 + l.k * r * 2 + r * l.n * 2 for l in lins)
            + m * k * 2 + k * 4)


# Dominant launch of the decode step: the grouped gate + up launch (two
# 18944 x 3584 linears sharing x; the largest of the step's four launches) at
# M = 8.  DRAM traffic of one such launch (prep_kernel + mma_kernel):
# dram__bytes_read.sum + dram__bytes_write.sum from a 1-pass ncu capture of
# `bench.py --case 8,18944+18944,3584,32` (taken on the build with four MMA
# issuers up to 64 tokens, the compact epilogue and the early weight stages
# that complete without the activations).
DOMINANT = ("gate_up", 8)
DOMINANT_TRAFFIC_BYTES = 79674624  # prep 596,480 + mma 79,022,592 read + 55,552 written (ncu, 1 pass)


def dominant_call(q, layers, acts, hbm_peak, reps=64):
    """Average per-launch time of the dominant grouped launch: a graph of
    back-to-back launches timed with CUDA events on the replaying stream,
    weights rotating over the layer copies (cold in L2)."""
    g, m = DOMINANT
    idx = [i for i, lin in enumerate(wl.QWEN_7B) if lin.group == g]
    lins = [wl.QWEN_7B[i] for i in idx]
    a = acts[DECODE_MS.index(m)]

    def call(i):
        layer = layers[i % len(layers)]
        members = [(layer[j].wp, layer[j].S, layer[j].A, layer[j].B, ALPHA, a.y[j]) for j in idx]
        q.check(q.qerl_lora_linear_group(a.x[g], a.z[g], members, a.ws), "qerl_lora_linear_group")

    for i in range(3):
        call(i)
    torch.cuda.synchronize()
    # The launches are captured into one graph (no host gaps between them); the
    # events on the replaying stream bracket all of them.
    g_ = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    with torch.cuda.graph(g_, stream=cs):
        for i in range(reps):
            call(i)
    g_.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g_.replay()
    e1.record()
    torch.cuda.synchronize()
    q.check(q.qerl_read_status(a.ws), "dominant launch status")
    t_ms = e0.elapsed_time(e1) / reps
    alg = group_algorithmic_bytes(lins, m)
    achieved = alg / (t_ms * 1e-3) / 1e9
    names = " + ".join(f"{l.name} {l.n}x{l.k}" for l in lins)
    return {
        "bound": "hbm",
        "kernel": f"qerl_lora_linear_group launch (prep_kernel + mma_kernel), Qwen2.5-7B {names}, "
                  f"M={m}, r={RANK_R}",
        "achieved": round(achieved, 1),
        "peak": hbm_peak,
        "peak_source": "measured hbm_gbs (MEASURED_PEAKS.json)",
        "unit": "GB/s",
        "frac": round(achieved / hbm_peak, 4),
        "traffic": DOMINANT_TRAFFIC_BYTES,
        "algorithmic_bytes_per_call": int(alg),
        "us_per_call": round(t_ms * 1e3, 3),
        "timing": f"CUDA events around one graph replay of {reps} back-to-back launches on the launching "
                  f"stream, weights rotating over {len(layers)} layer copies (> L2)",
    }


# ---------------------------------------------------------------- our arm

def bench_ours(args):
    import nvfp4_weight_quantized_03_gb300 as q

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev_index = torch.cuda.current_device()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    q.lib()
    hbm_peak, bf16_peak, bf16_sust, peak_src = load_peaks()
    shapes = wl.QWEN_7B
    seed = 0

    # ---- setup: quantize N_COPIES layer copies on the device
    layers = [layer_weights(q, shapes, seed, c) for c in range(N_COPIES)]
    acts = [Activations(q, shapes, m, seed) for m in DECODE_MS]
    layer_wbytes = sum(ql.weight_bytes for ql in layers[0])
    step_wbytes = layer_wbytes * len(DECODE_MS)

    def copy_for(step, j):
        return (len(DECODE_MS) * step + j) % N_COPIES

    def sigma_for(step):
        return q.qerl_aqn_sigma(step % NUM_STAGES, NUM_STAGES, SIGMA_START, SIGMA_END)

    # eager warm-up (kernel attributes, driver entry points), then capture graphs
    for j, act in enumerate(acts):
        run_substep(q, layers[copy_for(0, j)], act, sigma_for(0), 0)
    torch.cuda.synchronize()
    for act in acts:
        q.check(q.qerl_read_status(act.ws), "status after warm-up")

    cap_stream = torch.cuda.Stream()
    graphs = {}
    for st in range(NUM_STAGES):
        for j, act in enumerate(acts):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap_stream):
                run_substep(q, layers[copy_for(st, j)], act, sigma_for(st), st)
            graphs[(st, j)] = g
    torch.cuda.synchronize()

    def step(i):
        for j in range(len(DECODE_MS)):
            graphs[(i % NUM_STAGES, j)].replay()

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    # ---- timed region
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(DECODE_MS) + 1)] for _ in range(K)]
    clocks = ClockSampler(dev_index)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(K):
        for j in range(len(DECODE_MS)):
            ev[i][j].record()
            graphs[(i % NUM_STAGES, j)].replay()
        ev[i][-1].record()
    t1.record()
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1), world, "cuda")
    for act in acts:
        q.check(q.qerl_read_status(act.ws), "status after timed region")

    per_m = {}
    sub_bytes_total, sub_time_total = 0.0, 0.0
    for j, m in enumerate(DECODE_MS):
        ts = sorted(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(K))
        t_ms = sum(ts) / K
        alg = sum(linear_algorithmic_bytes(lin, m) for lin in shapes)
        sub_bytes_total += alg
        sub_time_total += t_ms
        flops = sum(linear_flops(lin, m) for lin in shapes)
        t_bw = layer_wbytes / (hbm_peak * 1e9) * 1e3
        t_tc = flops / (bf16_peak * 1e12) * 1e3
        per_m[str(m)] = {
            "ms_per_layer": round(t_ms, 5),
            "weight_GBps": round(layer_wbytes / (t_ms * 1e-3) / 1e9, 1),
            "all_bytes_GBps": round(alg / (t_ms * 1e-3) / 1e9, 1),
            "frac_of_hbm_peak": round(layer_wbytes / (t_ms * 1e-3) / 1e9 / hbm_peak, 4),
            "roofline_frac_max_bw_tc": round(max(t_bw, t_tc) / t_ms, 4),
            "TFLOPs": round(flops / (t_ms * 1e-3) / 1e12, 2),
            "tokens_per_s_per_layer": round(m / (t_ms * 1e-3), 1),
            "us_per_layer_p10_median_p90": [round(_pct(ts, p) * 1e3, 2) for p in (10, 50, 90)],
        }
    value = world * step_wbytes * K / (elapsed_ms * 1e-3) / 1e9

    # ---- prefill (14B-shaped layer, M = 4096) and quantizer throughput
    want = set(EXTRAS) if not args.skip_extra else set(args.extras.split(",")) - {""}
    extra_prefill = bench_prefill(q, args, bf16_peak) if "prefill" in want else None
    extra_quant = bench_quantize(q, hbm_peak) if "quantize" in want else None
    # ---- the other workloads: single 3B q_proj (hot/cold L2), 32B 64-layer stream (+ its
    # quantization), long sustained decode on the 7B stack
    extra_qproj = bench_qproj_3b(q, hbm_peak) if "qproj" in want else None
    extra_sustained = bench_sustained(q, hbm_peak, dev_index) if "sustained" in want else None
    extra_32b = bench_32b_stream(q, hbm_peak) if "32b" in want else None
    extra_mx = bench_mxfp4(q, hbm_peak) if "mxfp4" in want else None
    extra_bwd = bench_backward(q, bf16_peak) if "backward" in want else None
    extra_nf4 = bench_nf4(q, hbm_peak) if "nf4" in want else None

    # ---- the dominant launch, timed per call
    roofline = dominant_call(q, layers, acts, hbm_peak)

    # ---- end to end through the public API with host buffers (no graph)
    e2e = bench_e2e(q, layers, acts, args, copy_for, sigma_for, step_wbytes, world, barrier)

    calls = len(wl.NOISE_GROUPS) if GROUPED else len(shapes)
    launches_per_step = len(DECODE_MS) * (1 + 2 * calls)
    out = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(elapsed_ms / K, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e2m1*e4m3 (exact fp16) x bf16-as-exact-fp16 -> f32 accumulate, bf16 out",
        "data": "synthetic (seeded; random-init weights, no checkpoint)",
        "config": {
            "workload": WORKLOAD,
            "weights": "NVFP4 (E2M1 + E4M3 per 16 along K + FP32 tensor scale) quantized by the library from fp32 "
                       "N(0,0.02^2), 0.5% input channels x10",
            "weight_bytes_per_step": int(step_wbytes),
            "l2": f"weights rotate over {N_COPIES} distinct layer copies "
                  f"({N_COPIES * layer_wbytes / 1e9:.2f} GB) > 129 MB L2; activations stay hot",
            "launch": ("one CUDA graph per (stage, M): 1 AQN sampler launch (4 groups) + "
                       + ("4 grouped linear launches {q,k,v},{o},{gate,up},{down}" if GROUPED
                          else "7 single-linear calls")),
            "parallelism": f"replicas x{world}",
        },
        "per_m": per_m,
        "roofline": roofline,
        "substep_roofline": {
            "what": "whole decode sub-step (AQN sampler + 7 linears) per (M, layer), graph replay",
            "achieved": round(sub_bytes_total / (sub_time_total * 1e-3) / 1e9, 1),
            "unit": "GB/s",
            "frac": round(sub_bytes_total / (sub_time_total * 1e-3) / 1e9 / hbm_peak, 4),
        },
        "gpu_launches": launches_per_step * K,
        "clocks": clk,
        "e2e": e2e,
    }
    if extra_prefill:
        out["prefill"] = extra_prefill
    if extra_quant:
        out["quantize"] = extra_quant
    if extra_qproj:
        out["qproj_3b_m4"] = extra_qproj
    if extra_sustained:
        out["sustained_decode"] = extra_sustained
    if not args.skip_extra:
        out["aqn_schedules"] = aqn_schedule_table(q)
    if extra_32b:
        out["decode_32b_64layers_m16"] = extra_32b["decode"]
        out["quantize_32b_all"] = extra_32b["quantize"]
    if extra_mx:
        out["mxfp4"] = extra_mx
    if extra_bwd:
        out["backward"] = extra_bwd
    if extra_nf4:
        out["nf4"] = extra_nf4
    if rank == 0 and not args.skip_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline_oracle(seconds_budget=args.cpu_budget)
        out["cpu_baseline"]["all_cores"] = cpu_baseline_oracle_all_cores()
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def aqn_schedule_table(q, num_stages=NUM_STAGES, calls=20000):
    """The four sigma decay schedules of the library (host functions) per stage, and their host
    cost per call (the schedule is evaluated once per training step)."""
    names = {q.QERL_SCHEDULE_EXPONENTIAL: "exponential", q.QERL_SCHEDULE_LINEAR: "linear",
             q.QERL_SCHEDULE_COSINE: "cosine", q.QERL_SCHEDULE_LOGARITHMIC: "logarithmic"}
    lib = q.lib()
    out = {"num_stages": num_stages, "sigma_start": SIGMA_START, "sigma_end": SIGMA_END}
    for sch, name in names.items():
        out[name] = [float(f"{q.qerl_aqn_sigma_schedule(sch, st, num_stages, SIGMA_START, SIGMA_END):.6e}")
                     for st in range(num_stages)]
    t = time.perf_counter()
    for i in range(calls):
        lib.qerl_aqn_sigma_schedule(i & 3, i % num_stages, num_stages, SIGMA_START, SIGMA_END)
    out["host_ns_per_call_incl_ctypes"] = round((time.perf_counter() - t) * 1e9 / calls, 1)
    return out


def _pct(sorted_vals, p):
    """p-th percentile (nearest rank) of an ascending list."""
    i = min(len(sorted_vals) - 1, max(0, int(round(p / 100.0 * (len(sorted_vals) - 1)))))
    return sorted_vals[i]


def bench_prefill(q, args, bf16_peak):
    shapes = wl.QWEN_14B
    m = 4096
    sigma = 5e-3
    layer = [QLinear(q, lin, 1, 0, li) for li, lin in enumerate(shapes)]
    act = Activations(q, shapes, m, 1)
    run_substep(q, layer, act, sigma, 0)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=s):
        run_substep(q, layer, act, sigma, 0)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    reps = 50
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    ev[0].record()
    for i in range(reps):
        g.replay()
        ev[i + 1].record()
    torch.cuda.synchronize()
    ts = sorted(ev[i].elapsed_time(ev[i + 1]) for i in range(reps))
    t_ms = sum(ts) / reps
    q.check(q.qerl_read_status(act.ws), "prefill status")
    flops = sum(linear_flops(lin, m) for lin in shapes)
    tf = flops / (t_ms * 1e-3) / 1e12
    # each grouped launch alone (eager, back to back; a launch is ~1 ms, so launch cost is noise)
    per_launch = {}
    for g_name, (x, z, arr) in zip(wl.NOISE_GROUPS, act.group_descs(q, layer)):
        lins = [ql.lin for ql in layer if ql.lin.group == g_name]
        for _ in range(2):
            q.check(q.qerl_lora_linear_group(x, z, arr, act.ws), "qerl_lora_linear_group")
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_rep = 20
        e0.record()
        for _ in range(n_rep):
            q.check(q.qerl_lora_linear_group(x, z, arr, act.ws), "qerl_lora_linear_group")
        e1.record()
        torch.cuda.synchronize()
        lt = e0.elapsed_time(e1) / n_rep
        lf = sum(linear_flops(lin, m) for lin in lins)
        per_launch[g_name] = {"ms": round(lt, 4), "TFLOPs": round(lf / (lt * 1e-3) / 1e12, 1),
                              "frac_of_bf16_peak": round(lf / (lt * 1e-3) / 1e12 / bf16_peak, 4)}
    q.check(q.qerl_read_status(act.ws), "prefill status")
    res = {"workload": "Qwen2.5-14B decoder-layer linears, M=4096 (8 x 512 prompt tokens), r=32 alpha=64, "
                       "AQN sigma=5e-3", "ms_per_layer": round(t_ms, 4), "TFLOPs": round(tf, 1),
           "frac_of_bf16_peak": round(tf / bf16_peak, 4), "peak_TFLOPs": bf16_peak,
           "ms_per_layer_p10_median_p90": [round(_pct(ts, p), 4) for p in (10, 50, 90)],
           "per_launch": per_launch,
           "timing": f"{reps} graph replays of the layer (AQN sampler + 4 grouped launches), one event pair "
                     "each; per_launch: each grouped launch {q,k,v}, {o}, {gate,up}, {down} 20x back to back",
           "note": "fp16 operands run at the bf16 dense rate; peak = measured cuBLAS bf16 burst"}
    del layer, act
    torch.cuda.empty_cache()
    return res


def bench_quantize(q, hbm_peak):
    shapes = wl.QWEN_7B
    Ws = [wl.weight_f32_device(lin.n, lin.k, 2, 0, li).to(torch.bfloat16) for li, lin in enumerate(shapes)]
    outs = [(torch.empty((lin.n, lin.k // 2), dtype=torch.uint8, device="cuda"),
             torch.empty((lin.n, lin.k // 16), dtype=torch.uint8, device="cuda"),
             torch.empty(1, dtype=torch.float32, device="cuda")) for lin in shapes]
    ws = q.workspace(256)

    def run():
        for W, (c, s, S) in zip(Ws, outs):
            q.check(q.qerl_nvfp4_quantize(W, c, s, S, ws), "qerl_nvfp4_quantize")

    run()
    torch.cuda.synchronize()
    reps = 5
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        run()
    e1.record()
    torch.cuda.synchronize()
    t_ms = e0.elapsed_time(e1) / reps
    q.check(q.qerl_read_status(ws), "quantize status")
    nw = sum(lin.n * lin.k for lin in shapes)
    two_pass = nw * (2 + 2 + BYTES_PER_WEIGHT)
    res = {"workload": "NVFP4 quantization of one Qwen2.5-7B layer's 7 matrices from bf16 (233 M weights)",
           "ms": round(t_ms, 4), "GBps_two_pass_bytes": round(two_pass / (t_ms * 1e-3) / 1e9, 1),
           "frac_of_hbm_peak": round(two_pass / (t_ms * 1e-3) / 1e9 / hbm_peak, 4),
           "GBps_single_pass_bytes": round(nw * (2 + BYTES_PER_WEIGHT) / (t_ms * 1e-3) / 1e9, 1),
           "bytes_note": "4.5625 B/weight: bf16 read twice (amax pass + encode pass) + 0.5625 B written; "
                         "single-pass lower bound 2.5625 B/weight"}
    del Ws, outs
    torch.cuda.empty_cache()
    return res


def backward_flops(lin, m, r=RANK_R):
    """dx~ = dy W_hat (2mnk) + s (dy B) A (u: 2mnr, u A: 2mrk); t = x~ A^T (2mkr); dA (2mrk); dB (2mnr)."""
    return 2.0 * m * lin.n * lin.k + 4.0 * m * lin.n * r + 6.0 * m * lin.k * r


def bench_backward(q, bf16_peak, m=4096):
    """The policy-update half: the backward of the 14B-shaped layer's seven linears at M = 4096 (dx~,
    dA, dB per linear; the weights packed transposed once), graph replay."""
    shapes = wl.QWEN_14B
    r = RANK_R
    items = []
    for li, lin in enumerate(shapes):
        W = wl.weight_f32_device(lin.n, lin.k, 6, 0, li)
        codes, scales, S = q.quantize(W)
        del W
        wpt = q.pack_transposed(codes, scales)
        del codes, scales
        A = wl.normal_bf16_device((r, lin.k), 1.0 / math.sqrt(lin.k), 6, li, 2)
        B = wl.normal_bf16_device((lin.n, r), 0.01, 6, li, 3)
        xt = wl.normal_bf16_device((m, lin.k), 1.0, 6, li, 4)
        dy = wl.normal_bf16_device((m, lin.n), 0.01, 6, li, 5)
        dxt = torch.empty((m, lin.k), dtype=torch.bfloat16, device="cuda")
        dA = torch.empty((r, lin.k), dtype=torch.float32, device="cuda")
        dB = torch.empty((lin.n, r), dtype=torch.float32, device="cuda")
        items.append((lin, wpt, S, A, B, xt, dy, dxt, dA, dB))
    ws = q.workspace(max(q.qerl_lora_linear_backward_workspace_size(m, lin.n, lin.k, r) for lin in shapes))

    def layer_bwd():
        for lin, wpt, S, A, B, xt, dy, dxt, dA, dB in items:
            q.check(q.qerl_lora_linear_backward(xt, dy, wpt, S, A, B, ALPHA, dxt, dA, dB, ws),
                    "qerl_lora_linear_backward")

    t_ms, _, pct = _graph_time_ms(layer_bwd, 20)
    q.check(q.qerl_read_status(ws), "backward status")
    flops = sum(backward_flops(lin, m, r) for lin in shapes)
    per = {}
    for lin, wpt, S, A, B, xt, dy, dxt, dA, dB in items:
        def one():
            q.check(q.qerl_lora_linear_backward(xt, dy, wpt, S, A, B, ALPHA, dxt, dA, dB, ws),
                    "qerl_lora_linear_backward")
        lt, _, _ = _graph_time_ms(one, 10)
        lf = backward_flops(lin, m, r)
        per[lin.name] = {"ms": round(lt, 4), "TFLOPs": round(lf / (lt * 1e-3) / 1e12, 1),
                         "frac_of_bf16_peak": round(lf / (lt * 1e-3) / 1e12 / bf16_peak, 4)}
    res = {"workload": "backward of the Qwen2.5-14B-shaped layer's 7 linears, M=4096, r=32 alpha=64: dx~ (bf16), "
                       "dA, dB (fp32)",
           "ms_per_layer": round(t_ms, 4), "TFLOPs": round(flops / (t_ms * 1e-3) / 1e12, 1),
           "frac_of_bf16_peak": round(flops / (t_ms * 1e-3) / 1e12 / bf16_peak, 4),
           "ms_per_layer_p10_median_p90": [round(v, 4) for v in pct], "per_linear": per,
           "flops_note": "2mnk + 4mnr + 6mkr per linear (dx~ base, dy B, (dy B) A, x~ A^T, dA, dB)"}
    del items
    torch.cuda.empty_cache()
    return res


MXFP4_BYTES_PER_WEIGHT = 0.5 + 1.0 / 32  # E2M1 + one E8M0 per 32


def bench_mxfp4(q, hbm_peak, ms=(8, 32)):
    """The format variant: the 7B-shaped layer quantized to MXFP4 by the library (timed), packed,
    then decode through the same grouped launches as the headline (graph replay, weights rotating
    over N_COPIES layer copies).  GB/s on MXFP4's own bytes (0.53125 B/weight) and on the bytes the
    kernels move (the packed layout keeps one scale byte per 16, 0.5625 B/weight)."""
    shapes = wl.QWEN_7B
    Ws = [wl.weight_f32_device(lin.n, lin.k, 5, 0, li).to(torch.bfloat16) for li, lin in enumerate(shapes)]
    outs = [(torch.empty((lin.n, lin.k // 2), dtype=torch.uint8, device="cuda"),
             torch.empty((lin.n, lin.k // 32), dtype=torch.uint8, device="cuda")) for lin in shapes]
    ws = q.workspace(256)

    def quant():
        for W, (c, sc) in zip(Ws, outs):
            q.check(q.qerl_mxfp4_quantize(W, c, sc, ws), "qerl_mxfp4_quantize")

    quant()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(5):
        quant()
    e1.record()
    torch.cuda.synchronize()
    tq = e0.elapsed_time(e1) / 5
    q.check(q.qerl_read_status(ws), "mxfp4 quantize status")
    nw = sum(lin.n * lin.k for lin in shapes)
    res = {"workload": "Qwen2.5-7B-shaped layer in MXFP4 (E2M1 + E8M0 per 32), LoRA r=32, AQN",
           "quantize": {"ms": round(tq, 4), "GBps": round(nw * (2 + MXFP4_BYTES_PER_WEIGHT) / (tq * 1e-3) / 1e9, 1),
                        "bytes_note": "one pass: bf16 read + 0.53125 B/weight written"}}
    del Ws, outs
    layers = [[QLinear(q, lin, 5, c, li, fmt="mxfp4") for li, lin in enumerate(shapes)] for c in range(N_COPIES)]
    mx_bytes = nw * MXFP4_BYTES_PER_WEIGHT
    for m in ms:
        act = Activations(q, shapes, m, 5)
        q.check(q.qerl_aqn_sample(act.z_all, 1e-2, 5), "qerl_aqn_sample")

        def step():
            for c in range(N_COPIES):
                run_substep(q, layers[c], act, 1e-2, c)

        t_ms, _, pct = _graph_time_ms(step, 20)
        q.check(q.qerl_read_status(act.ws), "mxfp4 decode status")
        per_layer_us = t_ms * 1e3 / N_COPIES
        res[f"decode_m{m}"] = {
            "us_per_layer": round(per_layer_us, 2),
            "GBps_mxfp4_bytes": round(mx_bytes / (per_layer_us * 1e-6) / 1e9, 1),
            "GBps_packed_bytes": round(nw * BYTES_PER_WEIGHT / (per_layer_us * 1e-6) / 1e9, 1),
            "frac_of_hbm_peak_packed": round(nw * BYTES_PER_WEIGHT / (per_layer_us * 1e-6) / 1e9 / hbm_peak, 4)}
        del act
    del layers
    torch.cuda.empty_cache()
    return res


def bench_nf4(q, hbm_peak, ms=(8, 32)):
    """The QLoRA format through the same kernels: the 7B-shaped layer NF4-quantized by the library
    (levels recovered by table lookup in the dequantization), decode through the grouped launches,
    weights rotating over N_COPIES layer copies; the same bytes per weight as NVFP4."""
    shapes = wl.QWEN_7B
    layers = [[QLinear(q, lin, 7, c, li, fmt="nf4") for li, lin in enumerate(shapes)] for c in range(N_COPIES)]
    nw = sum(lin.n * lin.k for lin in shapes)
    res = {"workload": "Qwen2.5-7B-shaped layer in NF4 (QLoRA levels, E4M3 per 16 + FP32 tensor scale), LoRA r=32, "
                       "AQN"}
    for m in ms:
        act = Activations(q, shapes, m, 7)

        def step():
            for c in range(N_COPIES):
                run_substep(q, layers[c], act, 1e-2, c)

        t_ms, _, _ = _graph_time_ms(step, 20)
        q.check(q.qerl_read_status(act.ws), "nf4 decode status")
        us = t_ms * 1e3 / N_COPIES
        res[f"decode_m{m}"] = {"us_per_layer": round(us, 2),
                               "weight_GBps": round(nw * BYTES_PER_WEIGHT / (us * 1e-6) / 1e9, 1),
                               "frac_of_hbm_peak": round(nw * BYTES_PER_WEIGHT / (us * 1e-6) / 1e9 / hbm_peak, 4)}
        del act
    del layers
    torch.cuda.empty_cache()
    return res


def _graph_time_ms(fn, reps, warm=2):
    """Capture fn() into one CUDA graph, replay `warm` times, then time `reps` back-to-back replays
    with an event between consecutive ones: (mean ms, graph, [p10, median, p90] ms)."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=s):
        fn()
    for _ in range(warm):
        g.replay()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    ev[0].record()
    for i in range(reps):
        g.replay()
        ev[i + 1].record()
    torch.cuda.synchronize()
    ts = sorted(ev[i].elapsed_time(ev[i + 1]) for i in range(reps))
    return ev[0].elapsed_time(ev[-1]) / reps, g, [_pct(ts, p) for p in (10, 50, 90)]


def bench_qproj_3b(q, hbm_peak):
    """Single Qwen2.5-3B q_proj (2048 x 2048), M = 4, r = 16, alpha = 32, AQN sigma = 1e-2: per-call
    time with the weights hot in L2 (one copy) and cold (64 rotating copies, 151 MB > L2)."""
    lin = wl.QWEN_3B_QPROJ
    m, r, alpha = 4, 16, 32.0
    copies = [QLinear(q, lin, 3, c, r=r) for c in range(64)]
    x = wl.normal_bf16_device((m, lin.k), 1.0, 3, 0, 11)
    z = torch.empty(lin.k, dtype=torch.float32, device="cuda")
    q.check(q.qerl_aqn_sample(z, 1e-2, 3), "qerl_aqn_sample")
    y = torch.empty((m, lin.n), dtype=torch.bfloat16, device="cuda")
    ws = q.workspace(q.qerl_lora_linear_workspace_size(m, lin.n, lin.k, r))
    reps = 64
    res = {"workload": "Qwen2.5-3B q_proj 2048x2048, M=4, LoRA r=16 alpha=32, AQN sigma=1e-2"}
    for name, ncp in (("l2_hot", 1), ("l2_cold", 64)):
        def calls():
            for i in range(reps):
                ql = copies[i % ncp]
                q.check(q.qerl_lora_linear(x, ql.wp, ql.S, z, ql.A, ql.B, alpha, y, ws), "qerl_lora_linear")
        t_ms, _, pct = _graph_time_ms(calls, 50)
        us = t_ms * 1e3 / reps
        alg = linear_algorithmic_bytes(lin, m, r)
        res[name] = {"us_per_call": round(us, 3), "GBps": round(alg / (us * 1e-6) / 1e9, 1),
                     "frac_of_hbm_peak": round(alg / (us * 1e-6) / 1e9 / hbm_peak, 4),
                     "us_per_call_p10_median_p90": [round(v * 1e3 / reps, 3) for v in pct],
                     "timing": f"50 graph replays of {reps} back-to-back calls, one event pair per replay"}
    q.check(q.qerl_read_status(ws), "qproj status")
    del copies
    torch.cuda.empty_cache()
    return res


def bench_32b_stream(q, hbm_peak):
    """Qwen2.5-32B-shaped 64-layer weight stream: every linear quantized by the library from bf16
    ~N(0, 0.02^2) with Student-t(3) outlier channels (each quantize call timed), then one decode
    step at M = 16 through all 448 linears (64 x (AQN sampler + 4 grouped launches)), one graph."""
    shapes = wl.QWEN_32B
    nl = wl.QWEN_32B_LAYERS
    m = 16
    ws_q = q.workspace(256)
    layers = []
    qt_ms, n_weights = 0.0, 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for li in range(nl):
        layer = []
        for j, lin in enumerate(shapes):
            W = wl.weight_heavy_tail_bf16_device(lin.n, lin.k, 32, li, j)
            codes = torch.empty((lin.n, lin.k // 2), dtype=torch.uint8, device="cuda")
            scales = torch.empty((lin.n, lin.k // 16), dtype=torch.uint8, device="cuda")
            S = torch.empty(1, dtype=torch.float32, device="cuda")
            e0.record()
            q.check(q.qerl_nvfp4_quantize(W, codes, scales, S, ws_q), "qerl_nvfp4_quantize")
            e1.record()
            e1.synchronize()
            qt_ms += e0.elapsed_time(e1)
            n_weights += lin.n * lin.k
            ql = QLinear.__new__(QLinear)
            ql.lin, ql.S, ql.wp, ql.w_format = lin, S, q.pack(codes, scales), q.QERL_W_NVFP4
            ql.A = wl.normal_bf16_device((RANK_R, lin.k), 1.0 / math.sqrt(lin.k), 32, li, j, 2)
            ql.B = wl.normal_bf16_device((lin.n, RANK_R), 0.01, 32, li, j, 3)
            layer.append(ql)
            del W, codes, scales
        layers.append(layer)
    q.check(q.qerl_read_status(ws_q), "quantize status")
    act = Activations(q, shapes, m, 32)

    def step():
        for li, layer in enumerate(layers):
            run_substep(q, layer, act, 5e-3, li)

    reps = 50
    t_ms, g, pct = _graph_time_ms(step, reps)
    q.check(q.qerl_read_status(act.ws), "32B step status")
    wbytes = sum(ql.weight_bytes for layer in layers for ql in layer)
    alg = nl * sum(linear_algorithmic_bytes(lin, m) for lin in shapes)
    two_pass = n_weights * (2 + 2 + BYTES_PER_WEIGHT)
    res = {
        "decode": {"workload": "Qwen2.5-32B-shaped 64 decoder layers (448 linears, hidden 5120, intermediate 27648, "
                               "kv 1024), one decode step at M=16, LoRA r=32 alpha=64, per-layer AQN noise",
                   "weight_bytes": int(wbytes), "ms_per_step": round(t_ms, 3),
                   "weight_GBps": round(wbytes / (t_ms * 1e-3) / 1e9, 1),
                   "frac_of_hbm_peak": round(wbytes / (t_ms * 1e-3) / 1e9 / hbm_peak, 4),
                   "all_bytes_GBps": round(alg / (t_ms * 1e-3) / 1e9, 1),
                   "tokens_per_s": round(m / (t_ms * 1e-3), 1),
                   "ms_per_step_p10_median_p90": [round(v, 3) for v in pct],
                   "timing": f"one CUDA graph of the whole step (320 launches), {reps} timed replays"},
        "quantize": {"workload": "nvfp4 quantization of all 448 Qwen2.5-32B-shaped matrices from bf16 "
                                 "N(0,0.02^2) with Student-t(3) outlier channels (0.5%)",
                     "weights": int(n_weights), "ms_total": round(qt_ms, 3),
                     "GBps_two_pass_bytes": round(two_pass / (qt_ms * 1e-3) / 1e9, 1),
                     "frac_of_hbm_peak": round(two_pass / (qt_ms * 1e-3) / 1e9 / hbm_peak, 4),
                     "GBps_single_pass_bytes": round(n_weights * (2 + BYTES_PER_WEIGHT) / (qt_ms * 1e-3) / 1e9, 1),
                     "timing": "CUDA events around each quantize call, summed"},
    }
    del layers, act, g
    torch.cuda.empty_cache()
    return res


def bench_sustained(q, hbm_peak, dev_index, steps=8192):
    """Long-rollout decode on a 28-layer Qwen2.5-7B-shaped stack (3.67 GB NVFP4): `steps`
    back-to-back decode steps per M in {8, 64, 128}, a step being one token pass through all
    28 layers (per layer: one AQN sampler launch for the four noise groups, then the four
    grouped linear launches).  z is resampled every step (sampler counter = step) and sigma
    follows qerl_aqn_stage(step, steps, 10).  Launches are eager (the counter changes every
    step) and go straight to the C entry points with argument lists built once.  Reported:
    GB/s over the run and min / median over consecutive windows of >= 1 s, clocks sampled."""
    shapes = wl.QWEN_7B
    nl = wl.QWEN_7B_LAYERS
    layers = [layer_weights(q, shapes, 47, li) for li in range(nl)]
    lib = q.lib()
    stream = torch.cuda.current_stream().cuda_stream
    step_wbytes = nl * sum(ql.weight_bytes for ql in layers[0])
    sigmas = [q.qerl_aqn_sigma(s, NUM_STAGES, SIGMA_START, SIGMA_END) for s in range(NUM_STAGES)]
    res = {"workload": f"{steps} back-to-back decode steps per M through a {nl}-layer Qwen2.5-7B-shaped stack "
                       f"({step_wbytes / 1e9:.2f} GB NVFP4 + LoRA r=32), AQN z resampled every step, sigma "
                       f"1e-2 -> 5e-4 over 10 stages (qerl_aqn_stage)",
           "launch": "eager: per layer 1 AQN sampler + 4 grouped linear launches"}
    for m in (8, 64, 128):
        act = Activations(q, shapes, m, 7)
        ws_p, ws_n = act.ws.data_ptr(), act.ws.numel() * act.ws.element_size()
        z_p, z_n = act.z_all.data_ptr(), act.z_all.numel()
        calls = []
        for layer in layers:
            per = []
            for g in wl.NOISE_GROUPS:
                members = [(ql.wp, ql.S, ql.A, ql.B, ALPHA, y) for ql, y in zip(layer, act.y) if ql.lin.group == g]
                arr = q.linear_descs(members)
                x = act.x[g]
                per.append((x.data_ptr(), x.shape[0], x.shape[1], x.stride(0), act.z[g].data_ptr(), arr, len(arr)))
            calls.append(per)

        def step(i):
            sg = sigmas[q.qerl_aqn_stage(i, steps, NUM_STAGES)]
            for li, per in enumerate(calls):
                lib.qerl_aqn_sample(z_p, z_n, sg, 7, li, i, stream)
                for xp, mm, kk, ld, zp, arr, cnt in per:
                    lib.qerl_lora_linear_group(xp, mm, kk, ld, zp, arr, cnt, ws_p, ws_n, stream)

        for i in range(2):
            step(i)
        torch.cuda.synchronize()
        q.check(q.qerl_read_status(act.ws), "sustained warm-up status")
        # host cost of enqueuing a step while the launch queue still has room (two steps
        # after a sync); in the long run below the queue is full and the host waits on it
        h0 = time.perf_counter()
        step(0)
        step(1)
        host_free_ms = (time.perf_counter() - h0) * 1e3 / 2
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        clocks = ClockSampler(dev_index)
        clocks.start()
        ev[0].record()
        h0 = time.perf_counter()
        for i in range(steps):
            step(i)
            ev[i + 1].record()
        host_s = time.perf_counter() - h0
        torch.cuda.synchronize()
        clk = clocks.stop()
        q.check(q.qerl_read_status(act.ws), "sustained status")
        dts = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
        total = sum(dts)
        windows, acc_ms, acc_n = [], 0.0, 0
        for d in dts:
            acc_ms += d
            acc_n += 1
            if acc_ms >= 1000.0:
                windows.append(step_wbytes * acc_n / (acc_ms * 1e-3) / 1e9)
                acc_ms, acc_n = 0.0, 0
        gbps = step_wbytes * steps / (total * 1e-3) / 1e9
        res[str(m)] = {"steps": steps, "s_total": round(total / 1e3, 2), "ms_per_step": round(total / steps, 3),
                       "weight_GBps": round(gbps, 1), "frac_of_hbm_peak": round(gbps / hbm_peak, 4),
                       "window_GBps_min": round(min(windows), 1) if windows else None,
                       "window_GBps_median": round(statistics.median(windows), 1) if windows else None,
                       "windows": len(windows), "tokens_per_s": round(m * steps / (total * 1e-3), 1),
                       "host_enqueue_ms_per_step": round(host_s * 1e3 / steps, 3),
                       "host_enqueue_ms_per_step_queue_free": round(host_free_ms, 3),
                       "clocks": clk}
        del calls, act
        torch.cuda.empty_cache()
    del layers
    torch.cuda.empty_cache()
    return res


def bench_e2e(q, layers, acts, args, copy_for, sigma_for, step_wbytes, world, barrier):
    """Same decode step through the public API, eager calls, inputs copied from pinned host
    memory and outputs copied back to pinned host memory inside the timed region.  The
    copies run on a second stream, ordered against the compute by events: each token
    batch's input copy overlaps the previous batches' compute, its output copy the next
    ones' (what a serving loop does with the API's stream argument)."""
    host_x = [torch.empty(a.x_all.shape, dtype=a.x_all.dtype, pin_memory=True).copy_(a.x_all.cpu()) for a in acts]
    host_y = [torch.empty(a.y_all.shape, dtype=a.y_all.dtype, pin_memory=True) for a in acts]
    h2d = sum(a.io_bytes()[0] for a in acts)
    d2h = sum(a.io_bytes()[1] for a in acts)
    # each (layer copy, M) pair's descriptor arrays, built once
    descs = {}
    comp = torch.cuda.current_stream()
    copy_s = torch.cuda.Stream()
    computed = [None] * len(acts)   # compute of batch j done (its x may be overwritten)
    copied_out = [None] * len(acts)  # output copy of batch j done (its y may be overwritten)

    def e2e_step(i):
        loaded = []
        with torch.cuda.stream(copy_s):
            for j, a in enumerate(acts):
                if computed[j] is not None:
                    copy_s.wait_event(computed[j])
                a.x_all.copy_(host_x[j], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(copy_s)
                loaded.append(ev)
        for j, a in enumerate(acts):
            comp.wait_event(loaded[j])
            if copied_out[j] is not None:
                comp.wait_event(copied_out[j])
            c = copy_for(i, j)
            if not GROUPED:
                run_substep(q, layers[c], a, sigma_for(i), i % NUM_STAGES)
            else:
                if (c, j) not in descs:
                    descs[(c, j)] = a.group_descs(q, layers[c])
                q.check(q.qerl_aqn_sample(a.z_all, sigma_for(i), 0, 0, i % NUM_STAGES), "qerl_aqn_sample")
                for x, z, arr in descs[(c, j)]:
                    q.check(q.qerl_lora_linear_group(x, z, arr, a.ws), "qerl_lora_linear_group")
            done = torch.cuda.Event()
            done.record(comp)
            computed[j] = done
            with torch.cuda.stream(copy_s):
                copy_s.wait_event(done)
                host_y[j].copy_(a.y_all, non_blocking=True)
                out = torch.cuda.Event()
                out.record(copy_s)
                copied_out[j] = out

    for i in range(max(2, args.warmup)):
        e2e_step(i)
    torch.cuda.synchronize()
    steps = max(3, min(args.steps, 20))
    barrier()
    t = time.perf_counter()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    for i in range(steps):
        e2e_step(i)
    for ev in copied_out:
        comp.wait_event(ev)  # the last outputs are on the host
    e1.record(comp)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t
    barrier()
    dev_ms = e0.elapsed_time(e1)
    t_s = max_over_ranks(max(wall, dev_ms * 1e-3), world, "cuda")
    return {"value": round(world * step_wbytes * steps / t_s / 1e9, 1), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
            "ms_per_step": round(t_s * 1e3 / steps, 4),
            "wall_ms_per_step": round(wall * 1e3 / steps, 4), "device_ms_per_step": round(dev_ms / steps, 4),
            "path": "python binding -> C ABI, eager calls (no graph); pinned host x/y copies in the timed region on "
                    "a second stream, ordered against the compute by events"}


# ---------------------------------------------------------------- oracle (CPU baseline / reference arm)

def _oracle_layer_sample(cols_per_linear=None, shapes=None, seed=0):
    """Oracle-quantized weights of a 7B-shaped layer (host, from the seeded workload draws)."""
    import oracle
    shapes = shapes or wl.QWEN_7B
    out = []
    for li, lin in enumerate(shapes):
        n = lin.n if cols_per_linear is None else min(lin.n, cols_per_linear)
        W = wl.weight_f32(n, lin.k, seed, 100, li)
        codes, scales, S = oracle.quantize(W)
        A = wl.lora_A_bits(RANK_R, lin.k, seed, 100, li)
        B = wl.lora_B_bits(n, RANK_R, seed, 100, li)
        out.append((lin, n, codes, scales, S, A, B))
    return out


def _oracle_inputs(layer, ms, seed):
    """Seeded activations per (M, input group), drawn before any timing."""
    ks = {lin.group: lin.k for (lin, *_r) in layer}
    return {m: {g: wl.activations_bits(m, k, seed, 200, m, gi) for gi, (g, k) in enumerate(ks.items())} for m in ms}


def _oracle_step(layer, xs, ms, step):
    """One pass of the oracle over the sample: per M, the AQN sigma and noise of
    each group present, then every linear of the sample."""
    import oracle
    wbytes = 0.0
    groups = {lin.group: lin.k for (lin, *_r) in layer}
    for m in ms:
        sig = oracle.aqn_sigma(step % NUM_STAGES, NUM_STAGES, SIGMA_START, SIGMA_END)
        zs = {g: oracle.aqn_sample(k, sig, 0, gi, step % NUM_STAGES) for gi, (g, k) in enumerate(groups.items())}
        for (lin, n, codes, scales, S, A, B) in layer:
            oracle.lora_linear(xs[m][lin.group], codes, scales, S, z=zs[lin.group], A_bits=A, B_bits=B, alpha=ALPHA)
            wbytes += n * lin.k * BYTES_PER_WEIGHT
    return wbytes


def cpu_baseline_oracle(seconds_budget=15.0):
    """The oracle as it stands (single-threaded C, fp64), on a bounded sample of the workload."""
    layer = _oracle_layer_sample()
    xs = _oracle_inputs(layer, DECODE_MS, 0)
    t = time.perf_counter()
    wbytes = 0.0
    ms_done = []
    for m in DECODE_MS:
        if time.perf_counter() - t > seconds_budget and ms_done:
            break
        wbytes += _oracle_step(layer, xs, (m,), 0)
        ms_done.append(m)
    dt = time.perf_counter() - t
    return {"value": round(wbytes / dt / 1e9, 5), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"full 7B-shaped layer (7 linears + 4 AQN samples) at decode M in {ms_done}, one pass each; "
                      f"{dt:.1f} s; plain C fp64, single thread", "host_cpus": os.cpu_count(),
            "host_cpu_model": host_cpu_model()}


def _oracle_slice_worker(idx, nproc, ms, barrier, out_q):
    """All-cores baseline worker: output rows idx::nproc of every linear of the 7B-shaped layer
    (oracle-quantized slices), timed after a common barrier on the system-wide monotonic clock."""
    import oracle
    layer = []
    for li, lin in enumerate(wl.QWEN_7B):
        rows = np.arange(idx, lin.n, nproc)
        W = wl.weight_f32(lin.n, lin.k, 0, 100, li)[rows]
        codes, scales, S = oracle.quantize(W)
        A = wl.lora_A_bits(RANK_R, lin.k, 0, 100, li)
        B = wl.lora_B_bits(lin.n, RANK_R, 0, 100, li)[rows]
        layer.append((lin, len(rows), codes, scales, S, A, B))
    xs = _oracle_inputs(layer, ms, 0)
    barrier.wait()
    t0 = time.monotonic()
    wbytes = _oracle_step(layer, xs, ms, 0)
    out_q.put((t0, time.monotonic(), wbytes))


def cpu_baseline_oracle_all_cores(ms=DECODE_MS):
    """The same oracle on every host core: one spawned process per core, each owning an
    interleaved slice of every linear's output rows; wall time from the common start to the
    last finish."""
    import multiprocessing as mp
    nproc = os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(nproc)
    out_q = ctx.Queue()
    procs = [ctx.Process(target=_oracle_slice_worker, args=(i, nproc, tuple(ms), barrier, out_q))
             for i in range(nproc)]
    for pr in procs:
        pr.start()
    res = [out_q.get() for _ in procs]
    for pr in procs:
        pr.join()
    wall = max(r[1] for r in res) - min(r[0] for r in res)
    wbytes = sum(r[2] for r in res)
    return {"value": round(wbytes / wall / 1e9, 5), "unit": UNIT, "cores": nproc, "kind": "oracle",
            "sample": f"full 7B-shaped layer at decode M in {list(ms)}, output rows split over {nproc} "
                      f"processes; {wall:.2f} s wall", "host_cpu_model": host_cpu_model()}


def bench_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    cols = 256
    layer = [e for e in _oracle_layer_sample(cols_per_linear=cols) if e[0].name in ("q", "down")]
    xs = _oracle_inputs(layer, DECODE_MS, 0)
    for i in range(args.warmup):
        _oracle_step(layer, xs, DECODE_MS, i)
    t = time.perf_counter()
    wbytes = 0.0
    for i in range(args.steps):
        wbytes += _oracle_step(layer, xs, DECODE_MS, i)
    dt = time.perf_counter() - t
    value = wbytes / dt / 1e9
    sample = (f"oracle (plain C fp64, 1 thread) on the q and down linears of the 7B-shaped layer restricted to "
              f"{cols} output columns, M in {list(DECODE_MS)}, 4 AQN samples per M, per step")
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded)", "config": {"workload": WORKLOAD, "sample": sample},
           "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample,
                            "host_cpus": os.cpu_count(), "host_cpu_model": host_cpu_model()},
           "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
           "gpu_launches": 0}
    print(json.dumps(out), flush=True)


def bench_case(args):
    """One linear shape on its own (the command profilers wrap): `--case M,N,K,R` with N a '+'-joined
    list for one grouped launch (e.g. 8,18944+18944,3584,32 for gate + up), `--case-kind backward`
    for the backward of a single linear.  `--case-copies` weight sets (fp32 N(0, 0.02^2) quantized by
    the library) rotate over `--steps` timed calls after `--warmup` untimed ones, CUDA events on the
    current stream (or one graph replay with --case-graph).  Prints one JSON line."""
    m_s, n_s, k_s, r_s = args.case.split(",")
    m, k, r = int(m_s), int(k_s), int(r_s)
    ns = [int(v) for v in n_s.split("+")]
    import nvfp4_weight_quantized_03_gb300 as q
    q.lib()
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    bwd = args.case_kind == "backward"
    if bwd and len(ns) != 1:
        raise SystemExit("--case-kind backward takes one linear")
    sets = []
    for _ in range(args.case_copies):
        members = []
        for n in ns:
            W = torch.randn(n, k, device=dev, generator=gen) * 0.02
            codes, scales, S = q.quantize(W)
            members.append((q.pack_transposed(codes, scales) if bwd else q.pack(codes, scales), S))
            del W, codes, scales
        sets.append(members)
    x = torch.randn(m, k, device=dev, generator=gen).to(torch.bfloat16)
    As = [(torch.randn(r, k, device=dev, generator=gen) / k ** 0.5).to(torch.bfloat16) if r else None for _ in ns]
    Bs = [(torch.randn(n, r, device=dev, generator=gen) * 0.01).to(torch.bfloat16) if r else None for n in ns]
    z = torch.empty(k, dtype=torch.float32, device=dev)
    q.check(q.qerl_aqn_sample(z, 1e-2, 0))
    ys = [torch.empty(m, n, dtype=torch.bfloat16, device=dev) for n in ns]
    if bwd:
        dy = (torch.randn(m, ns[0], device=dev, generator=gen) * 0.01).to(torch.bfloat16)
        dxt = torch.empty(m, k, dtype=torch.bfloat16, device=dev)
        dA = torch.empty(r, k, dtype=torch.float32, device=dev) if r else None
        dB = torch.empty(ns[0], r, dtype=torch.float32, device=dev) if r else None
        ws = q.workspace(q.qerl_lora_linear_backward_workspace_size(m, ns[0], k, r))
    else:
        ws = q.workspace(q.qerl_lora_linear_group_workspace_size(
            m, k, [(wp, S, A_, B_, ALPHA, y) for (wp, S), A_, B_, y in zip(sets[0], As, Bs, ys)]))

    def call(i):
        members = sets[i % args.case_copies]
        if bwd:
            wpt, S = members[0]
            q.check(q.qerl_lora_linear_backward(x, dy, wpt, S, As[0], Bs[0], ALPHA, dxt, dA, dB, ws))
        else:
            q.check(q.qerl_lora_linear_group(
                x, z, [(wp, S, A_, B_, ALPHA, y) for (wp, S), A_, B_, y in zip(members, As, Bs, ys)], ws))

    for i in range(args.warmup):
        call(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if args.case_graph:
        g = torch.cuda.CUDAGraph()
        st = torch.cuda.Stream()
        with torch.cuda.graph(g, stream=st):
            for i in range(args.steps):
                call(i)
        g.replay()
        torch.cuda.synchronize()
        e0.record()
        g.replay()
        e1.record()
    else:
        e0.record()
        for i in range(args.steps):
            call(i)
        e1.record()
    torch.cuda.synchronize()
    q.check(q.qerl_read_status(ws), "case status")
    us = e0.elapsed_time(e1) * 1e3 / args.steps
    wbytes = sum(ns) * k * BYTES_PER_WEIGHT
    flops = sum(2.0 * m * n * k + 2.0 * m * r * (k + n) * (2 if bwd else 1) + (2.0 * m * k * r if bwd else 0.0)
                for n in ns)
    print(json.dumps({"case": args.case, "kind": args.case_kind, "us_per_call": round(us, 3),
                      "weight_GBps": round(wbytes / (us * 1e-6) / 1e9, 1),
                      "TFLOPs": round(flops / (us * 1e-6) / 1e12, 2), "graph": args.case_graph,
                      "calls": args.steps}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--skip-extra", action="store_true",
                    help="skip the prefill, quantizer, 3B q_proj, sustained and 32B-stream measurements")
    ap.add_argument("--extras", default="", help="with --skip-extra: a comma-separated subset of "
                    + ",".join(EXTRAS) + " to run anyway")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--ungrouped", action="store_true", help="seven single-linear calls per layer instead of four "
                    "grouped launches")
    ap.add_argument("--case", default="", help="time one shape instead: M,N,K,R (N '+'-joined for a grouped "
                    "launch), e.g. 8,18944+18944,3584,32")
    ap.add_argument("--case-kind", choices=["forward", "backward"], default="forward")
    ap.add_argument("--case-copies", type=int, default=4, help="weight sets the timed calls rotate over")
    ap.add_argument("--case-graph", action="store_true", help="replay the timed calls as one CUDA graph")
    args = ap.parse_args()
    if args.case:
        bench_case(args)
        return
    global GROUPED
    GROUPED = not args.ungrouped
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        bench_reference(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
