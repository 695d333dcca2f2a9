"""NF4 through the kernels, against the fp64 oracle.

QeRL digest, "NVFP4 Quantization" (comparison to other 4-bit formats) and "QLoRA's 4-bit
Quantization Addresses Memory but Degrades Speed": NF4's levels sit
at Gaussian quantiles and are recovered through a lookup table.
- qerl_nf4_quantize: codes, E4M3 scales and tensor scale bit-exact against orc.nf4_quantize (both
  decide each code in fp32 against fp32 level midpoints; each side computes its levels itself).
- The linear with w_format = QERL_W_NF4 against orc.nf4_lora_linear on the decode, pair and
  prefill paths, and a group mixing NF4 and NVFP4.  Unlike E2M1 x E4M3 (exact in fp16), an NF4
  level is irrational: the kernel holds it in fp16 and rounds level x block scale to fp16, a
  relative error of at most 2^-11 + 2^-11 (+ their product) per weight.  So the bound is derived
  from that arithmetic, element by element:
      |y - bf16(y_hat)| <= 2^-10 * (1 + 2^-10) * sum_k |x~_k w_hat_k| + 2^-7 |y_hat| + tiny,
  the last term covering one bf16 output flip; plus the normwise bound 2e-3 (twice the E2M1
  linears': the per-weight rounding is systematic per level, so it does not average out).
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


def _to_dev(W_np, bf16):
    if bf16:
        return torch.from_numpy(wl.to_bf16_bits(W_np).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(W_np, dtype=np.float32)).cuda()


def _quant_same(q, orc, W_np, bf16=False):
    codes, scales, S = q.nf4_quantize(_to_dev(W_np, bf16))
    Wo = wl.bf16_bits_to_f32(wl.to_bf16_bits(W_np)) if bf16 else np.ascontiguousarray(W_np, dtype=np.float32)
    oc, osc, oS = orc.nf4_quantize(Wo)
    assert float(S.cpu()[0]) == oS
    assert np.array_equal(scales.cpu().numpy(), osc)
    assert np.array_equal(codes.cpu().numpy(), oc)
    return codes, scales, S, oc, osc, oS


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("n,k", [(1, 32), (37, 96), (256, 3584), (130, 5120)])
def test_quantize_bit_exact(q, orc, n, k, bf16):
    _quant_same(q, orc, wl.weight_f32(n, k, 600 + n, 1), bf16=bf16)


def test_quantize_ranges(q, orc):
    rng = wl.rng(610, 1)
    W = rng.standard_normal((32, 512)).astype(np.float32)
    W = (W.reshape(-1, 16) * np.logspace(-30, 30, W.size // 16)[:, None]).astype(np.float32).reshape(32, 512)
    W[4] = 0.0
    _quant_same(q, orc, W)


def _assert_nf4_close(orc, y_gpu, ref, x_bits, z, codes, scales, S, what):
    got = y_gpu.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got)), what
    xt = wl.bf16_bits_to_f32(orc.noise_apply(x_bits, z)).astype(np.float64)
    mag = np.abs(xt) @ np.abs(orc.nf4_dequant(codes, scales, S)).T  # sum_k |x~_k w_hat_k|
    ref_b = (orc.f64_to_bf16(ref).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    bound = 2.0 ** -10 * (1 + 2.0 ** -10) * mag + 2.0 ** -7 * np.abs(ref) + 1e-30
    err = np.abs(got - ref_b)
    assert np.all(err <= bound), f"{what}: worst err/bound {np.max(err / bound):.3f}"
    norm = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert norm <= 2e-3, f"{what}: normwise {norm:.3e}"


def _case(q, orc, m, n, k, r, seed, mixed=False):
    codes, scales, S, oc, osc, oS = _quant_same(q, orc, wl.weight_f32(n, k, seed, 0))
    wp = q.pack(codes, scales)
    x_bits = wl.activations_bits(m, k, seed + 1, 1)
    A_bits = wl.lora_A_bits(r, k, seed + 2, 2) if r else None
    B_bits = wl.lora_B_bits(n, r, seed + 3, 3) if r else None
    z = wl.noise_vector(k, 1e-2, seed + 4)
    y = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    descs = [(wp, S, dev_bf16(A_bits) if r else None, dev_bf16(B_bits) if r else None, 2.0 * r, y, q.QERL_W_NF4)]
    if mixed:  # a second, NVFP4 linear in the same launch
        W2 = wl.weight_f32(n, k, seed + 5, 0)
        c2, s2, S2 = q.quantize(torch.from_numpy(W2).cuda())
        oc2, osc2, oS2 = orc.quantize(W2)
        y2 = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
        descs.append((q.pack(c2, s2), S2, None, None, 0.0, y2))
    ws = q.workspace(q.qerl_lora_linear_group_workspace_size(m, k, descs))
    q.check(q.qerl_lora_linear_group(dev_bf16(x_bits), torch.from_numpy(z).cuda(), descs, ws))
    assert q.qerl_read_status(ws) == 0
    rows = None if m <= 128 else np.unique(np.concatenate([[0, m - 1], np.arange(0, m, 13)]))
    xs = x_bits if rows is None else x_bits[rows]
    ref = orc.nf4_lora_linear(xs, oc, osc, oS, z=z, A_bits=A_bits, B_bits=B_bits, alpha=2.0 * r)
    got = y if rows is None else y[torch.from_numpy(rows).cuda()]
    _assert_nf4_close(orc, got, ref, xs, z, oc, osc, oS, what=f"nf4 m{m} n{n} k{k} r{r}")
    if mixed:
        ref2 = orc.lora_linear(xs, oc2, osc2, oS2, z=z)
        got2 = y2 if rows is None else y2[torch.from_numpy(rows).cuda()]
        assert_linear_close(got2, ref2, orc, what=f"nvfp4 beside nf4 m{m}")


@pytest.mark.parametrize("m,n,k,r", [(1, 256, 512, 16), (8, 512, 3584, 32), (33, 384, 1024, 32),
                                     (100, 384, 2048, 32), (128, 512, 18944, 32), (300, 256, 576, 16)])
def test_linear_matches_oracle(q, orc, m, n, k, r):
    _case(q, orc, m, n, k, r, seed=620 + m)


@pytest.mark.parametrize("m", [8, 128, 260])
def test_group_mixing_nf4_and_nvfp4(q, orc, m):
    _case(q, orc, m, 384, 1024, 16, seed=640 + m, mixed=True)
