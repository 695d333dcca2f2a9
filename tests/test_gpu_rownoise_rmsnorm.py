"""Per-rollout noise and the noise-merged RMSNorm, on the GPU, against the fp64 oracle.

- Per-row noise (QeRL digest, "Adaptive Quantization Noise": each rollout sees its
  own noise sample): qerl_lora_linear_group_rowz with z [m][k] against
  orc.lora_linear with the same per-row z, over the decode (shared-slab, pair)
  and prefill kernel paths; identical rows reproduce the broadcast call bit for bit.
- RMSNorm with the noise merged into its weight ("Noise Merging", Eq. 10-11):
  qerl_rmsnorm_noise against orc.rmsnorm_noise bit for bit (both compute in fp64
  and round once to bf16; the only difference is the order of the squares' sum,
  ~1e-16 relative, so a value may round the other way only when the oracle's
  fp64 value lies within 2^-40 of a bf16 rounding midpoint), and the fused
  qerl_rmsnorm_lora_linear_group against the oracle linear of the oracle's x~
  under the linear tests' bounds.
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


def _weights(q, orc, n, k, seed):
    W = wl.weight_f32(n, k, seed, 0)
    codes, scales, S = q.quantize(torch.from_numpy(W).cuda())
    oc, osc, oS = orc.quantize(W)
    assert np.array_equal(codes.cpu().numpy(), oc) and np.array_equal(scales.cpu().numpy(), osc)
    return q.pack(codes, scales), S, oc, osc, oS


def _row_noise(m, k, sigma, seed):
    return (wl.rng(seed, 9).standard_normal((m, k)) * sigma).astype(np.float32)


@pytest.mark.parametrize("m,n,k,r", [(1, 256, 512, 16), (8, 512, 3584, 32), (17, 384, 1024, 32),
                                     (100, 384, 2048, 32), (128, 512, 18944, 32), (300, 256, 576, 16)])
def test_per_row_noise_matches_oracle(q, orc, m, n, k, r):
    wp, S, oc, osc, oS = _weights(q, orc, n, k, seed=71)
    x_bits = wl.activations_bits(m, k, 72, 1)
    A_bits, B_bits = wl.lora_A_bits(r, k, 73, 2), wl.lora_B_bits(n, r, 74, 3)
    z = _row_noise(m, k, 1e-2, 75)
    # a padded row stride, to check that ldz is honoured
    zbuf = torch.zeros((m, k + 16), dtype=torch.float32, device="cuda")
    zbuf[:, :k] = torch.from_numpy(z).cuda()
    y = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    desc = [(wp, S, dev_bf16(A_bits), dev_bf16(B_bits), 2.0 * r, y)]
    ws = q.workspace(q.qerl_lora_linear_group_workspace_size(m, k, desc))
    q.check(q.qerl_lora_linear_group_rowz(dev_bf16(x_bits), zbuf[:, :k], desc, ws))
    assert q.qerl_read_status(ws) == 0
    rows = None if m <= 128 else np.unique(np.concatenate([[0, m - 1], np.arange(0, m, 7)]))
    ref = orc.lora_linear(x_bits if rows is None else x_bits[rows], oc, osc, oS,
                          z=z if rows is None else z[rows], A_bits=A_bits, B_bits=B_bits, alpha=2.0 * r)
    got = y if rows is None else y[torch.from_numpy(rows).cuda()]
    assert_linear_close(got, ref, orc, what=f"per-row noise m{m} n{n} k{k}")


def test_identical_noise_rows_equal_the_broadcast(q, orc):
    m, n, k, r = 8, 384, 1024, 16
    wp, S, *_ = _weights(q, orc, n, k, seed=81)
    x = dev_bf16(wl.activations_bits(m, k, 82, 1))
    A, B = dev_bf16(wl.lora_A_bits(r, k, 83, 2)), dev_bf16(wl.lora_B_bits(n, r, 84, 3))
    zv = torch.from_numpy(wl.noise_vector(k, 1e-2, 85)).cuda()
    y1 = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    y2 = torch.empty_like(y1)
    ws = q.workspace(q.qerl_lora_linear_group_workspace_size(m, k, [(wp, S, A, B, 32.0, y1)]))
    q.check(q.qerl_lora_linear_group(x, zv, [(wp, S, A, B, 32.0, y1)], ws))
    q.check(q.qerl_lora_linear_group_rowz(x, zv.expand(m, k).contiguous(), [(wp, S, A, B, 32.0, y2)], ws))
    assert q.qerl_read_status(ws) == 0
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def _hidden_bits(m, k, seed, scale=1.0):
    """A pre-norm hidden state: N(0, scale^2) with a few large channels (as residual streams have)."""
    h = wl.rng(seed, 10).standard_normal((m, k)).astype(np.float32) * np.float32(scale)
    h[:, wl.outlier_channels(k, seed, 11)] *= 20.0
    return wl.to_bf16_bits(h)


def _midpoint_flip_ok(got_bits, ref64, ref_bits):
    """Positions where got differs from ref: allowed only as a 1-ulp flip with the oracle's
    fp64 value within 2^-40 (relative) of the bf16 rounding midpoint."""
    diff = got_bits != ref_bits
    if not diff.any():
        return True
    g = got_bits[diff].astype(np.int64)
    rb = ref_bits[diff].astype(np.int64)
    adjacent = (((g ^ rb) & 0x8000) == 0) & (np.abs((g & 0x7FFF) - (rb & 0x7FFF)) == 1)
    gv = (got_bits[diff].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    rv = (ref_bits[diff].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    mid = (gv + rv) / 2.0
    v = ref64[diff]
    return bool(np.all(adjacent & (np.abs(v - mid) <= 2.0 ** -40 * np.abs(v))))


@pytest.mark.parametrize("m,k,with_noise", [(1, 512, True), (8, 3584, True), (33, 5120, False), (300, 2048, True)])
def test_rmsnorm_noise_bits(q, orc, m, k, with_noise):
    h_bits = _hidden_bits(m, k, 90 + m)
    w_bits = wl.rmsnorm_weight_bits(k, 91)
    Z = wl.noise_vector(k, 1e-2, 92) if with_noise else None
    out = torch.full((m, k), float("nan"), dtype=torch.bfloat16, device="cuda")
    q.check(q.qerl_rmsnorm_noise(dev_bf16(h_bits), dev_bf16(w_bits), None if Z is None else torch.from_numpy(Z).cuda(),
                                 1e-6, out))
    torch.cuda.synchronize()
    ref64, ref_bits = orc.rmsnorm_noise(h_bits, w_bits, Z, 1e-6)
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert _midpoint_flip_ok(got, ref64, ref_bits), f"m{m} k{k}: {(got != ref_bits).sum()} values differ"


def test_rmsnorm_zero_row(q, orc):
    m, k = 3, 256
    h_bits = _hidden_bits(m, k, 95)
    h_bits[1] = 0
    w_bits = wl.rmsnorm_weight_bits(k, 96)
    out = torch.full((m, k), float("nan"), dtype=torch.bfloat16, device="cuda")
    q.check(q.qerl_rmsnorm_noise(dev_bf16(h_bits), dev_bf16(w_bits), None, 1e-6, out))
    torch.cuda.synchronize()
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.all(got[1] == 0)
    assert np.array_equal(got, orc.rmsnorm_noise(h_bits, w_bits, None, 1e-6)[1])


@pytest.mark.parametrize("m", [4, 64, 100, 260])
def test_rmsnorm_fused_linear(q, orc, m):
    """RMSNorm_noise -> the grouped linear (two linears of the normalised input, LoRA on one)."""
    k = 1024
    h_bits = _hidden_bits(m, k, 97)
    w_bits = wl.rmsnorm_weight_bits(k, 98)
    Z = wl.noise_vector(k, 5e-3, 99)
    shapes = [(512, 16), (256, 0)]
    lins, ys = [], []
    for i, (n, r) in enumerate(shapes):
        wp, S, oc, osc, oS = _weights(q, orc, n, k, seed=100 + i)
        A_bits = wl.lora_A_bits(r, k, 102 + i, 2) if r else None
        B_bits = wl.lora_B_bits(n, r, 104 + i, 3) if r else None
        y = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
        lins.append((wp, S, dev_bf16(A_bits) if r else None, dev_bf16(B_bits) if r else None, 2.0 * r, y))
        ys.append((y, oc, osc, oS, A_bits, B_bits, 2.0 * r))
    ws = q.workspace(q.qerl_rmsnorm_lora_linear_group_workspace_size(m, k, lins))
    q.check(q.qerl_rmsnorm_lora_linear_group(dev_bf16(h_bits), dev_bf16(w_bits), torch.from_numpy(Z).cuda(), 1e-6,
                                             lins, ws))
    assert q.qerl_read_status(ws) == 0
    xt_bits = orc.rmsnorm_noise(h_bits, w_bits, Z, 1e-6)[1]
    for y, oc, osc, oS, A_bits, B_bits, alpha in ys:
        ref = orc.lora_linear(xt_bits, oc, osc, oS, z=None, A_bits=A_bits, B_bits=B_bits, alpha=alpha)
        assert_linear_close(y, ref, orc, what=f"rmsnorm fused m{m} n{oc.shape[0]}")


@pytest.mark.parametrize("m", [1, 13, 16])
def test_grouped_lora_ranks_per_row_noise(q, orc, m):
    """Four linears of one input with ranks 32, 8, 24 and 16 at up to 16 tokens (four LoRA tiles of
    the prep kernel per K slice, one per linear, each with its own rank padding), with per-row
    noise and a ragged row count: every output against the oracle."""
    k = 1536
    shapes = [(384, 32), (256, 8), (128, 24), (512, 16)]
    x_bits = wl.activations_bits(m, k, 92, 1)
    z = _row_noise(m, k, 1e-2, 93)
    x, zd = dev_bf16(x_bits), torch.from_numpy(z).cuda()
    descs, refs = [], []
    for i, (n, r) in enumerate(shapes):
        wp, S, oc, osc, oS = _weights(q, orc, n, k, seed=94 + i)
        A_bits, B_bits = wl.lora_A_bits(r, k, 100 + i, 2), wl.lora_B_bits(n, r, 110 + i, 3)
        y = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
        descs.append((wp, S, dev_bf16(A_bits), dev_bf16(B_bits), 2.0 * r, y))
        refs.append(orc.lora_linear(x_bits, oc, osc, oS, z=z, A_bits=A_bits, B_bits=B_bits, alpha=2.0 * r))
    ws = q.workspace(q.qerl_lora_linear_group_workspace_size(m, k, descs))
    q.check(q.qerl_lora_linear_group_rowz(x, zd, descs, ws))
    assert q.qerl_read_status(ws) == 0
    for (n, r), d, ref in zip(shapes, descs, refs):
        assert_linear_close(d[5], ref, orc, what=f"grouped ranks m{m} n{n} r{r}")
