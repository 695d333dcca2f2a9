"""The sharding contract on one GPU (the partitions a multi-GPU deployment would use,
each shard run by the library as its own call):

- N-split (column parallel: q/k/v/gate/up): each shard's amax -> max -> qerl_nvfp4_tensor_scale
  -> qerl_nvfp4_quantize_with_scale gives the whole tensor's codes and scales bit for bit; the
  shards' linears (their rows of B, the same A, x and z) concatenate to the whole linear.
- K-split (row parallel: o/down): shards along K on 16-block boundaries (codes, scales, A, x,
  z sliced; the whole B); the linear is linear in x~ along K, LoRA term included
  ((x~_1 A_1^T + x~_2 A_2^T) B^T), so the shards' fp32 outputs sum to the whole output.

Compared in fp32 output mode against the unsharded call (only the summation order differs)
and in bf16 against the fp64 oracle.  Source: QeRL digest, "NVFP4 Quantization" Eq. 6 and
the LoRA forward after Eq. 2.
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


def _quantize_sharded(q, shards):
    """Quantize shards (device fp32) with the scale of their union."""
    ws = q.workspace(q.qerl_nvfp4_quantize_workspace_size())
    amaxes = []
    for W in shards:
        a = torch.empty(1, dtype=torch.float32, device="cuda")
        q.check(q.qerl_nvfp4_amax(W, a, ws))
        amaxes.append(a)
    amax = torch.stack(amaxes).max().reshape(1).contiguous()  # one process: the all-reduce(max)
    S = torch.empty(1, dtype=torch.float32, device="cuda")
    q.check(q.qerl_nvfp4_tensor_scale(amax, S))
    out = []
    for W in shards:
        n, k = W.shape
        codes = torch.empty((n, k // 2), dtype=torch.uint8, device="cuda")
        scales = torch.empty((n, k // 16), dtype=torch.uint8, device="cuda")
        q.check(q.qerl_nvfp4_quantize_with_scale(W, S, codes, scales, ws))
        out.append((codes, scales))
    assert q.qerl_read_status(ws) == 0
    return out, S


def test_n_and_k_sharded_quantization_bit_identical(q, orc):
    n, k = 18944, 3584  # the 7B gate projection
    W = wl.weight_f32_device(n, k, 3, 1)
    codes, scales, S = q.quantize(W)
    (c0, s0), (c1, s1) = _quantize_sharded(q, [W[: n // 2].contiguous(), W[n // 2:].contiguous()])[0]
    assert torch.equal(torch.cat([c0, c1]), codes) and torch.equal(torch.cat([s0, s1]), scales)
    kk = 1792  # K split on a 16-block boundary
    shards, S2 = _quantize_sharded(q, [W[:, :kk].contiguous(), W[:, kk:].contiguous()])
    assert S2.item() == S.item()
    assert torch.equal(torch.cat([shards[0][0], shards[1][0]], dim=1), codes)
    assert torch.equal(torch.cat([shards[0][1], shards[1][1]], dim=1), scales)
    oc, osc, oS = orc.quantize(W.cpu().numpy())
    assert np.array_equal(codes.cpu().numpy(), oc) and float(oS) == S.item()


def _linear(q, x, wp, S, z, A, B, alpha, n, ydt=torch.float32):
    m, k = x.shape
    y = torch.full((m, n), float("nan"), dtype=ydt, device="cuda")
    ws = q.workspace(q.qerl_lora_linear_workspace_size(m, n, k, 0 if A is None else A.shape[0]))
    q.check(q.qerl_lora_linear(x, wp, S, z, A, B, alpha, y, ws))
    assert q.qerl_read_status(ws) == 0
    return y


@pytest.mark.parametrize("m", [8, 128])
def test_column_and_row_parallel_linear(q, orc, m):
    n, k, r = 1024, 3584, 32
    Wf = wl.weight_f32(n, k, 4, 1)
    W = torch.from_numpy(Wf).cuda()
    x_bits = wl.activations_bits(m, k, 4, 2)
    A_bits, B_bits = wl.lora_A_bits(r, k, 4, 3), wl.lora_B_bits(n, r, 4, 4)
    z = wl.noise_vector(k, 1e-2, 4, 5)
    x, A, B, zd = dev_bf16(x_bits), dev_bf16(A_bits), dev_bf16(B_bits), torch.from_numpy(z).cuda()
    codes, scales, S = q.quantize(W)
    y_full = _linear(q, x, q.pack(codes, scales), S, zd, A, B, 64.0, n)
    ref = orc.lora_linear(x_bits, *orc.quantize(Wf), z=z, A_bits=A_bits, B_bits=B_bits, alpha=64.0)
    assert_linear_close(y_full, ref, orc, bf16_out=False, what="unsharded")
    # column parallel: rows of W and B split, x, z and A replicated
    shards, Ss = _quantize_sharded(q, [W[: n // 2].contiguous(), W[n // 2:].contiguous()])
    ys = [_linear(q, x, q.pack(c, s), Ss, zd, A, B[h * n // 2:(h + 1) * n // 2].contiguous(), 64.0, n // 2)
          for h, (c, s) in enumerate(shards)]
    y_col = torch.cat(ys, dim=1)
    assert torch.allclose(y_col, y_full, rtol=1e-5, atol=1e-6 * y_full.abs().max().item())
    # row parallel: K split, partial outputs summed (the all-reduce of y)
    kk = k // 2
    shards, Ss = _quantize_sharded(q, [W[:, :kk].contiguous(), W[:, kk:].contiguous()])
    parts = []
    for h, (c, s) in enumerate(shards):
        sl = slice(h * kk, (h + 1) * kk)
        parts.append(_linear(q, x[:, sl].contiguous(), q.pack(c, s), Ss, zd[sl].contiguous(),
                             A[:, sl].contiguous(), B, 64.0, n))
    y_row = parts[0] + parts[1]
    assert torch.allclose(y_row, y_full, rtol=1e-4, atol=1e-5 * y_full.abs().max().item())
    assert_linear_close(y_row, ref, orc, bf16_out=False, what="row parallel")
