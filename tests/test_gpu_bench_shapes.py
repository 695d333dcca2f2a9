"""The launches bench.py times, on the bench's own inputs, against the fp64 oracle.

bench.py reports throughput for grouped launches on the Qwen2.5 shapes; this file
checks those very launches (same grouping, same shapes, same seeded device draws
for the weights, x and LoRA adapters, descriptor arrays built once as the bench
does) on sampled outputs:

- 7B decode: {q,k,v}, {o}, {gate,up}, {down} at M in {1, 8, 32, 64, 128} (the
  headline step and the sustained-decode sweep), r = 32, alpha = 64;
- 14B prefill: all seven linears at M = 4096 in the same four groups;
- 32B decode: all seven linears at M = 16 (layer 0 of the 64-layer stream, its
  heavy-tailed bf16 weights).

Weights are quantized by the library and checked bit for bit against the
oracle's quantization of the same fp32 matrix; the noise vector is a host draw
fed to both sides.  Outputs are compared with the oracle on every row (decode)
or 24 sampled rows (prefill) and 40 sampled columns per linear, including the
first and last column (the ragged edges of the tile grid), under the bounds of
the other linear tests (normwise 1e-3, max 2e-3 against bf16(y_hat)).
Source of the operation: QeRL digest, section 3.4, the LoRA forward after
Eq. 2 and "NVFP4 Quantization", Eq. 6.
"""
import math

import numpy as np
import pytest
import torch

import workloads as wl
from helpers import assert_linear_close, dev_bf16

pytestmark = pytest.mark.gpu

RANK, ALPHA = 32, 64.0


@pytest.fixture(scope="module")
def q():
    import nvfp4_weight_quantized_03_gb300 as mod
    mod.lib()
    return mod


class Lin:
    """One linear with the bench's seeded device draws (bench.py QLinear): weights
    wl.weight_f32_device(n, k, seed, copy, index), A / B wl.normal_bf16_device."""

    def __init__(self, q, orc, lin, seed, copy, li, heavy_tail=False):
        if heavy_tail:  # the 32B stream's weights: bf16 with Student-t(3) outlier channels
            W = wl.weight_heavy_tail_bf16_device(lin.n, lin.k, seed, copy, li)
        else:
            W = wl.weight_f32_device(lin.n, lin.k, seed, copy, li)
        self.lin = lin
        codes, scales, self.S = q.quantize(W)
        oc, osc, oS = orc.quantize(W.float().cpu().numpy())
        assert np.array_equal(codes.cpu().numpy(), oc), f"{lin.name}: codes differ from the oracle"
        assert np.array_equal(scales.cpu().numpy(), osc), f"{lin.name}: scales differ from the oracle"
        assert self.S.item() == float(oS)
        self.oc, self.osc, self.oS = oc, osc, oS
        self.wp = q.pack(codes, scales)
        del W, codes, scales
        self.A = wl.normal_bf16_device((RANK, lin.k), 1.0 / math.sqrt(lin.k), seed, copy, li, 2)
        self.B = wl.normal_bf16_device((lin.n, RANK), 0.01, seed, copy, li, 3)
        self.A_bits = self.A.view(torch.int16).cpu().numpy().view(np.uint16)
        self.B_bits = self.B.view(torch.int16).cpu().numpy().view(np.uint16)


_LAYERS = {}


def layer(q, orc, shapes, seed, heavy_tail=False):
    key = (id(shapes), seed)
    if key not in _LAYERS:
        _LAYERS.clear()
        _LAYERS[key] = [Lin(q, orc, lin, seed, 0, li, heavy_tail) for li, lin in enumerate(shapes)]
        torch.cuda.empty_cache()
    return _LAYERS[key]


def sample(n, cnt, seed):
    rs = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, n - 1], rs.choice(n, min(cnt, n), replace=False)]))


def run_groups(q, orc, lins, m, sigma, seed, rows=None, what=""):
    """Every AQN group of the layer as one grouped launch through a descriptor array,
    as bench.py runs them; each member checked on sampled columns."""
    for gi, g in enumerate(wl.NOISE_GROUPS):
        members = [L for L in lins if L.lin.group == g]
        k = members[0].lin.k
        x = wl.normal_bf16_device((m, k), 1.0, seed, m, gi, 11)
        x_bits = x.view(torch.int16).cpu().numpy().view(np.uint16)
        z = wl.noise_vector(k, sigma, seed, m, gi) if sigma else None
        zd = torch.from_numpy(z).cuda() if sigma else None
        ys = [torch.full((m, L.lin.n), float("nan"), dtype=torch.bfloat16, device="cuda") for L in members]
        desc = [(L.wp, L.S, L.A, L.B, ALPHA, y) for L, y in zip(members, ys)]
        ws = q.workspace(q.qerl_lora_linear_group_workspace_size(m, k, desc))
        arr = q.linear_descs(desc)
        q.check(q.qerl_lora_linear_group(x, zd, arr, ws))
        assert q.qerl_read_status(ws) == 0
        xr = x_bits if rows is None else x_bits[rows]
        for j, (L, y) in enumerate(zip(members, ys)):
            cols = sample(L.lin.n, 40, 100 * gi + j)
            ref = orc.lora_linear(xr, L.oc, L.osc, L.oS, z=z, A_bits=L.A_bits, B_bits=L.B_bits, alpha=ALPHA,
                                  cols=cols)
            got = y[:, torch.from_numpy(cols).cuda()]
            if rows is not None:
                got = got[torch.from_numpy(rows).cuda()]
            assert_linear_close(got, ref, orc, what=f"{what} {L.lin.name} m{m}")
        del ys, ws, x


@pytest.mark.parametrize("m", [1, 8, 32, 64, 128])
def test_7b_decode_grouped(q, orc, m):
    """The headline decode step's four grouped launches on the 7B-shaped layer."""
    lins = layer(q, orc, wl.QWEN_7B, 0)
    run_groups(q, orc, lins, m, 1e-2, 0, what="7B")


def test_14b_prefill_grouped(q, orc):
    """The prefill bench: all seven 14B-shaped linears at M = 4096, four grouped launches."""
    lins = layer(q, orc, wl.QWEN_14B, 1)
    m = 4096
    run_groups(q, orc, lins, m, 5e-3, 1, rows=sample(m, 24, 5), what="14B prefill")


def test_32b_decode_grouped(q, orc):
    """One layer of the 32B-shaped stream at M = 16 (K = 27648 for down, N = 27648 for gate/up)."""
    lins = layer(q, orc, wl.QWEN_32B, 32, heavy_tail=True)
    run_groups(q, orc, lins, 16, 5e-3, 32, what="32B")


@pytest.mark.parametrize("m", [8, 64, 128])
def test_7b_decode_graph_replay_is_stable(q, orc, m):
    """The decode step as the bench runs it -- the four grouped launches captured in a CUDA
    graph and replayed back to back, weights rotating over three copies so that they stream
    from HBM -- 100 times: every replay ends with the status word clear, and every output is
    bit-identical to an eager run's (the launches are deterministic, so any barrier or ring
    hand-over that let an MMA read a slot before its data landed would show up here)."""
    lins = layer(q, orc, wl.QWEN_7B, 0)
    copies = [[L.wp] + [L.wp.clone() for _ in range(2)] for L in lins]
    groups = []
    for gi, g in enumerate(wl.NOISE_GROUPS):
        idx = [i for i, L in enumerate(lins) if L.lin.group == g]
        k = lins[idx[0]].lin.k
        x = wl.normal_bf16_device((m, k), 1.0, 0, m, gi, 11)
        zd = torch.from_numpy(wl.noise_vector(k, 1e-2, 0, m, gi)).cuda()
        ys = [torch.empty((m, lins[i].lin.n), dtype=torch.bfloat16, device="cuda") for i in idx]
        arrs = [q.linear_descs([(copies[i][c], lins[i].S, lins[i].A, lins[i].B, ALPHA, y) for i, y in zip(idx, ys)])
                for c in range(3)]
        ws = q.workspace(q.qerl_lora_linear_group_workspace_size(m, k, arrs[0]))
        groups.append((x, zd, arrs, ys, ws))

    def step(c):
        for x, zd, arrs, _, ws in groups:
            q.check(q.qerl_lora_linear_group(x, zd, arrs[c], ws))

    step(0)
    torch.cuda.synchronize()
    ref = [[y.clone() for y in g[3]] for g in groups]
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.graph(graph, stream=s):
        for c in range(3):
            step(c)
    for _ in range(34):
        graph.replay()
    torch.cuda.synchronize()
    for x, zd, arrs, ys, ws in groups:
        assert q.qerl_read_status(ws) == 0
    for g, r in zip(groups, ref):
        for y, y0 in zip(g[3], r):
            assert torch.equal(y.view(torch.int16), y0.view(torch.int16)), f"m{m}: replay differs from eager run"
