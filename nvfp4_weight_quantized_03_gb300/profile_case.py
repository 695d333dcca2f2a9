"""Time one qerl_lora_linear shape on the current GPU.

A per-shape timing harness (and the command that profilers wrap): builds
`copies` independent NVFP4 weight sets of one N x K linear (random fp32
N(0, 0.02^2) weights quantized by the library), bf16 activations, LoRA
adapters and AQN noise, then times `reps` calls that rotate over the weight
sets, with CUDA events on the current stream.  Prints one JSON line.

    python -m nvfp4_weight_quantized_03_gb300.profile_case --m 8 --n 3584 --k 3584 --r 32 --reps 50

A comma-separated --n (e.g. 18944,18944 for gate + up) times one grouped
launch (qerl_lora_linear_group) of that many linears sharing x, z and K.
"""
import argparse
import json

import torch

import nvfp4_weight_quantized_03_gb300 as q


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--m", type=int, default=8)
    ap.add_argument("--n", type=str, default="3584", help="output features; comma-separated for a group")
    ap.add_argument("--k", type=int, default=3584)
    ap.add_argument("--r", type=int, default=32)
    ap.add_argument("--alpha", type=float, default=64.0)
    ap.add_argument("--sigma", type=float, default=1e-2)
    ap.add_argument("--reps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--copies", type=int, default=4)
    ap.add_argument("--graph", action="store_true", help="replay the timed calls as one CUDA graph")
    a = ap.parse_args()
    ns = [int(v) for v in a.n.split(",")]
    torch.manual_seed(0)
    dev = torch.device("cuda")
    sets = []
    for _ in range(a.copies):
        members = []
        for n in ns:
            W = torch.randn(n, a.k, device=dev) * 0.02
            codes, scales, S = q.quantize(W)
            members.append((q.pack(codes, scales), S))
            del W, codes, scales
        sets.append(members)
    x = torch.randn(a.m, a.k, device=dev).to(torch.bfloat16)
    As = [(torch.randn(a.r, a.k, device=dev) / a.k ** 0.5).to(torch.bfloat16) if a.r else None for _ in ns]
    Bs = [(torch.randn(n, a.r, device=dev) * 0.01).to(torch.bfloat16) if a.r else None for n in ns]
    z = torch.empty(a.k, dtype=torch.float32, device=dev)
    q.check(q.qerl_aqn_sample(z, a.sigma, 0))
    ys = [torch.empty(a.m, n, dtype=torch.bfloat16, device=dev) for n in ns]
    if len(ns) == 1:
        ws = q.workspace(q.qerl_lora_linear_workspace_size(a.m, ns[0], a.k, a.r))
    else:
        ws = q.workspace(q.qerl_lora_linear_group_workspace_size(
            a.m, a.k, [(wp, S, A_, B_, a.alpha, y) for (wp, S), A_, B_, y in zip(sets[0], As, Bs, ys)]))

    def call(i):
        members = sets[i % a.copies]
        if len(ns) == 1:
            wp, S = members[0]
            q.check(q.qerl_lora_linear(x, wp, S, z, As[0], Bs[0], a.alpha, ys[0], ws))
        else:
            q.check(q.qerl_lora_linear_group(
                x, z, [(wp, S, A_, B_, a.alpha, y) for (wp, S), A_, B_, y in zip(members, As, Bs, ys)], ws))

    for i in range(a.warmup):
        call(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if a.graph:
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        with torch.cuda.graph(g, stream=s):
            for i in range(a.reps):
                call(i)
        g.replay()
        torch.cuda.synchronize()
        e0.record()
        g.replay()
        e1.record()
    else:
        e0.record()
        for i in range(a.reps):
            call(i)
        e1.record()
    torch.cuda.synchronize()
    q.check(q.qerl_read_status(ws))
    us = e0.elapsed_time(e1) * 1e3 / a.reps
    n_total = sum(ns)
    wbytes = n_total * a.k * 0.5625
    flops = sum(2.0 * a.m * n * a.k + 2.0 * a.m * a.r * (a.k + n) for n in ns)
    print(json.dumps({"m": a.m, "n": a.n, "k": a.k, "r": a.r, "us_per_call": round(us, 3),
                      "weight_GBps": round(wbytes / (us * 1e-6) / 1e9, 1),
                      "TFLOPs": round(flops / (us * 1e-6) / 1e12, 2), "graph": a.graph}))


if __name__ == "__main__":
    main()
