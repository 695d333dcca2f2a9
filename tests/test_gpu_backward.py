"""The LoRA linear's backward on the GPU against the fp64 oracle (orc.lora_linear_backward).

QeRL digest, "Low-Rank Adaptation (LoRA) Within Quantized Layers", gradient flow through the
frozen NVFP4 weight: dx~ = dy W_hat + s (dy B) A, dA = s (dy B)^T x~, dB = s dy^T (x~ A^T).
- dx~ (bf16 or fp32) under the linear tests' bounds (it is the forward kernel on the transposed
  problem: the transposed packed layout, dy as the activations, B^T / A^T as the adapters).
- dA and dB (fp32; rank-r sums over the tokens): normwise error <= 1e-5 against the fp64 oracle
  (fp32 accumulation of exact bf16 products: ~sqrt(terms) * 2^-24 relative).
Shapes span several weight tiles and stages with ragged tails, the decode token tiles and the
prefill path (m > 128), r from 8 to 128, and a 14B-shaped linear at m = 4096 (dx~ on sampled
rows, dA and dB in full).
"""
import numpy as np
import pytest
import torch

import workloads as wl
from helpers import assert_linear_close, dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import nvfp4_weight_quantized_03_gb300 as mod
    mod.lib()
    return mod


def _normwise(got, ref):
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def _case(q, orc, m, n, k, r, seed, f32=False, rows=None):
    W = wl.weight_f32(n, k, seed, 0)
    codes, scales, S = q.quantize(torch.from_numpy(W).cuda())
    oc, osc, oS = orc.quantize(W)
    assert np.array_equal(codes.cpu().numpy(), oc)
    wpt = q.pack_transposed(codes, scales)
    xt_bits = wl.activations_bits(m, k, seed + 1, 1)
    dy_bits = wl.activations_bits(m, n, seed + 2, 2, std=0.1)
    A_bits = wl.lora_A_bits(r, k, seed + 3, 2) if r else None
    B_bits = wl.lora_B_bits(n, r, seed + 4, 3, std=0.05) if r else None
    alpha = 2.0 * r if r else 0.0
    dxt = torch.full((m, k), float("nan"), dtype=torch.float32 if f32 else torch.bfloat16, device="cuda")
    dA = torch.full((r, k), float("nan"), dtype=torch.float32, device="cuda") if r else None
    dB = torch.full((n, r), float("nan"), dtype=torch.float32, device="cuda") if r else None
    ws = q.workspace(q.qerl_lora_linear_backward_workspace_size(m, n, k, r))
    q.check(q.qerl_lora_linear_backward(dev_bf16(xt_bits), dev_bf16(dy_bits), wpt, S,
                                        dev_bf16(A_bits) if r else None, dev_bf16(B_bits) if r else None, alpha,
                                        dxt, dA, dB, ws))
    assert q.qerl_read_status(ws) == 0
    dy = wl.bf16_bits_to_f32(dy_bits).astype(np.float64)
    if rows is None:
        ref_dxt, ref_dA, ref_dB = orc.lora_linear_backward(xt_bits, oc, osc, oS, A_bits, B_bits, alpha, dy)
        got_dxt = dxt
    else:
        ref_dxt = orc.lora_linear_backward(xt_bits[rows], oc, osc, oS, A_bits, B_bits, alpha, dy[rows])[0]
        got_dxt = dxt[torch.from_numpy(rows).cuda()]
        _, ref_dA, ref_dB = orc.lora_linear_backward(xt_bits, oc, osc, oS, A_bits, B_bits, alpha, dy,
                                                     want_dxt=False)
    assert_linear_close(got_dxt, ref_dxt, orc, bf16_out=not f32, what=f"dx~ m{m} n{n} k{k} r{r}")
    if r:
        for name, got, ref in (("dA", dA, ref_dA), ("dB", dB, ref_dB)):
            g = got.cpu().numpy().astype(np.float64)
            assert np.all(np.isfinite(g)), name
            assert _normwise(g, ref) <= 1e-5, (name, _normwise(g, ref))


@pytest.mark.parametrize("m,n,k,r", [(1, 256, 512, 16), (8, 512, 3584, 32), (17, 3584, 512, 32),
                                     (33, 384, 2048, 8), (64, 1024, 960, 64), (100, 384, 2048, 32),
                                     (128, 1024, 1024, 128), (300, 512, 576, 16), (260, 1536, 1024, 32)])
def test_backward_matches_oracle(q, orc, m, n, k, r):
    _case(q, orc, m, n, k, r, seed=400 + m)


def test_backward_fp32_input_gradient_and_no_lora(q, orc):
    _case(q, orc, 12, 768, 1024, 32, seed=420, f32=True)
    _case(q, orc, 40, 512, 1024, 0, seed=421)


def test_backward_14b_shape_m4096(q, orc):
    """A 14B-shaped linear (k/v: n = 1024, k = 5120) at the prefill batch: dx~ on sampled rows,
    dA and dB in full."""
    m = 4096
    rows = np.unique(np.concatenate([[0, m - 1], wl.rng(430, 1).choice(m, 22, replace=False)]))
    _case(q, orc, m, 1024, 5120, 32, seed=431, rows=rows)


def test_backward_empty_batch_zero_fills(q):
    n, k, r = 256, 512, 16
    codes = torch.zeros((n, k // 2), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((n, k // 16), dtype=torch.uint8, device="cuda")
    wpt = q.pack_transposed(codes, scales)
    S = torch.ones(1, device="cuda")
    A = torch.zeros((r, k), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((n, r), dtype=torch.bfloat16, device="cuda")
    dA = torch.full((r, k), 7.0, device="cuda")
    dB = torch.full((n, r), 7.0, device="cuda")
    x = torch.empty((0, k), dtype=torch.bfloat16, device="cuda")
    dy = torch.empty((0, n), dtype=torch.bfloat16, device="cuda")
    dxt = torch.empty((0, k), dtype=torch.bfloat16, device="cuda")
    ws = q.workspace(q.qerl_lora_linear_backward_workspace_size(0, n, k, r))
    q.check(q.qerl_lora_linear_backward(x, dy, wpt, S, A, B, 32.0, dxt, dA, dB, ws))
    torch.cuda.synchronize()
    assert torch.all(dA == 0) and torch.all(dB == 0)
