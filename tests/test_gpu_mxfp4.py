"""MXFP4 through the kernels, against the fp64 oracle.

QeRL digest, "NVFP4 Quantization", the comparison with MXFP4 (E2M1 elements, one E8M0
power-of-two scale per 32 elements, no tensor scale).
- qerl_mxfp4_quantize: codes and E8M0 scales bit-exact against orc.mxfp4_quantize (fp32 and
  bf16 inputs, strided rows, zero blocks, subnormal and huge magnitudes, heavy tails).
- qerl_mxfp4_pack + the linear: y against orc.mxfp4_lora_linear under the linear tests' bounds,
  on the decode (shared-slab, pair) and prefill kernel paths, with noise and LoRA.
- The packed layout's range: a block scale exactly 2^-17 of the largest is exact; one further
  below records QERL_ERR_RANGE.
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


def _to_dev(W_np, bf16, ld=None):
    if bf16:
        Wt = torch.from_numpy(wl.to_bf16_bits(W_np).view(np.int16)).view(torch.bfloat16)
    else:
        Wt = torch.from_numpy(np.ascontiguousarray(W_np, dtype=np.float32))
    n, k = Wt.shape
    if ld is not None and ld > k:
        big = torch.zeros((n, ld), dtype=Wt.dtype)
        big[:, :k] = Wt
        return big.cuda()[:, :k]
    return Wt.cuda()


def _oracle_input(W_np, bf16):
    return wl.bf16_bits_to_f32(wl.to_bf16_bits(W_np)) if bf16 else np.ascontiguousarray(W_np, dtype=np.float32)


def _assert_quant_same(q, orc, W_np, bf16=False, ld=None):
    ws = q.workspace(q.qerl_nvfp4_quantize_workspace_size())
    codes, scales = q.mxfp4_quantize(_to_dev(W_np, bf16, ld), ws)
    assert q.qerl_read_status(ws) == 0
    oc, osc = orc.mxfp4_quantize(_oracle_input(W_np, bf16))
    assert np.array_equal(scales.cpu().numpy(), osc)
    assert np.array_equal(codes.cpu().numpy(), oc)
    return codes, scales


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("n,k,ld", [(1, 32, None), (37, 96, 128), (256, 3584, None), (130, 18944, None)])
def test_quantize_bit_exact(q, orc, n, k, ld, bf16):
    _assert_quant_same(q, orc, wl.weight_f32(n, k, 300 + n, 1), bf16=bf16, ld=ld)


def test_quantize_heavy_tail_bf16(q, orc):
    bits = wl.weight_heavy_tail_bf16(512, 5120, 310, 1)
    _assert_quant_same(q, orc, wl.bf16_bits_to_f32(bits), bf16=True)


def test_quantize_ranges_and_zero_blocks(q, orc):
    """Block magnitudes from fp32 subnormals to 1e36 (E8M0 clamps at both ends), all-zero blocks,
    and every E2M1 midpoint of a block whose max is 4 (so 2^e = 1)."""
    rng = wl.rng(311, 1)
    n, k = 64, 1024
    W = rng.standard_normal((n, k)).astype(np.float32)
    mags = np.logspace(-44, 36, n * (k // 32)).astype(np.float64)
    W = (W.reshape(-1, 32) * mags[:, None]).astype(np.float32).reshape(n, k)
    W[3, 64:96] = 0.0
    W[5] = 0.0
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 4.0], np.float32)
    W[7, :32] = np.concatenate([mids, -mids, mids * 0.999, mids * 1.001])
    assert np.all(np.isfinite(W))
    _assert_quant_same(q, orc, W)


def test_quantize_nonfinite_is_reported(q):
    W = torch.ones((4, 64), dtype=torch.float32, device="cuda")
    W[2, 17] = float("inf")
    ws = q.workspace(q.qerl_nvfp4_quantize_workspace_size())
    codes = torch.empty((4, 32), dtype=torch.uint8, device="cuda")
    scales = torch.empty((4, 2), dtype=torch.uint8, device="cuda")
    q.check(q.qerl_mxfp4_quantize(W, codes, scales, ws))
    assert q.STATUS_NAMES[q.qerl_read_status(ws)] == "QERL_ERR_NONFINITE"


def _mx_linear_case(q, orc, m, n, k, r, seed, z_kind="vec", group=False):
    W = wl.weight_f32(n, k, seed, 0)
    codes, scales = _assert_quant_same(q, orc, W)
    ws_p = q.workspace(q.qerl_nvfp4_quantize_workspace_size())
    wp, S = q.mxfp4_pack(codes, scales, ws_p)
    assert q.qerl_read_status(ws_p) == 0
    oc, osc = codes.cpu().numpy(), scales.cpu().numpy()
    x_bits = wl.activations_bits(m, k, seed + 1, 1)
    A_bits = wl.lora_A_bits(r, k, seed + 2, 2) if r else None
    B_bits = wl.lora_B_bits(n, r, seed + 3, 3) if r else None
    if z_kind == "vec":
        z = wl.noise_vector(k, 1e-2, seed + 4)
        zd = torch.from_numpy(z).cuda()
    elif z_kind == "rows":
        z = (wl.rng(seed + 4, 9).standard_normal((m, k)) * 1e-2).astype(np.float32)
        zd = torch.from_numpy(z).cuda()
    else:
        z, zd = None, None
    y = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    desc = [(wp, S, dev_bf16(A_bits) if r else None, dev_bf16(B_bits) if r else None, 2.0 * r, y)]
    if group or z_kind == "rows":
        ws = q.workspace(q.qerl_lora_linear_group_workspace_size(m, k, desc))
        fn = q.qerl_lora_linear_group_rowz if z_kind == "rows" else q.qerl_lora_linear_group
        q.check(fn(dev_bf16(x_bits), zd, desc, ws))
        assert q.qerl_read_status(ws) == 0
    else:
        ws = q.workspace(q.qerl_lora_linear_workspace_size(m, n, k, r))
        q.check(q.qerl_lora_linear(dev_bf16(x_bits), wp, S, zd, desc[0][2], desc[0][3], 2.0 * r, y, ws))
        assert q.qerl_read_status(ws) == 0
    rows = None if m <= 128 else np.unique(np.concatenate([[0, m - 1], np.arange(0, m, 11)]))
    zr = z if (z is None or z.ndim == 1 or rows is None) else z[rows]
    ref = orc.mxfp4_lora_linear(x_bits if rows is None else x_bits[rows], oc, osc, z=zr, A_bits=A_bits,
                                B_bits=B_bits, alpha=2.0 * r)
    got = y if rows is None else y[torch.from_numpy(rows).cuda()]
    assert_linear_close(got, ref, orc, what=f"mxfp4 m{m} n{n} k{k} r{r}")


@pytest.mark.parametrize("m,n,k,r", [(1, 256, 512, 16), (4, 2048, 2048, 16), (8, 512, 3584, 32),
                                     (33, 384, 1024, 32), (100, 384, 2048, 32), (128, 512, 18944, 32),
                                     (300, 256, 576, 0)])
def test_linear_matches_oracle(q, orc, m, n, k, r):
    _mx_linear_case(q, orc, m, n, k, r, seed=320 + m)


def test_linear_group_and_row_noise(q, orc):
    _mx_linear_case(q, orc, 8, 768, 1024, 32, seed=340, group=True)
    _mx_linear_case(q, orc, 64, 384, 1024, 16, seed=341, z_kind="rows")
    _mx_linear_case(q, orc, 16, 256, 512, 8, seed=342, z_kind=None)


def _pack_status(q, codes_np, scales_np):
    codes = torch.from_numpy(codes_np).cuda()
    scales = torch.from_numpy(scales_np).cuda()
    ws = q.workspace(q.qerl_nvfp4_quantize_workspace_size())
    wp, S = q.mxfp4_pack(codes, scales, ws)
    return q.qerl_read_status(ws), wp, float(S.cpu()[0])


def test_pack_range(q, orc):
    """Block scales spanning exactly 2^17 pack exactly (the linear matches the oracle); a span of
    2^18 records QERL_ERR_RANGE; an all-zero weight gives S = 1."""
    n, k, m = 128, 512, 4
    rng = wl.rng(350, 1)
    codes = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    scales = rng.integers(120, 138, size=(n, k // 32)).astype(np.uint8)   # span 17: 120 .. 137
    scales[0, 0], scales[1, 1] = 120, 137
    st, wp, S = _pack_status(q, codes, scales)
    assert st == 0 and S == 2.0 ** (137 - 135)
    x_bits = wl.activations_bits(m, k, 351, 1)
    y = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = q.workspace(q.qerl_lora_linear_workspace_size(m, n, k, 0))
    q.check(q.qerl_lora_linear(dev_bf16(x_bits), wp, torch.tensor([S], device="cuda"), None, None, None, 0.0, y, ws))
    assert q.qerl_read_status(ws) == 0
    assert_linear_close(y, orc.mxfp4_lora_linear(x_bits, codes, scales), orc, what="span 2^17")
    scales[2, 3] = 119
    codes[2, 48:64] = 0x11                                                  # block 3 of row 2 non-zero
    st, _, _ = _pack_status(q, codes, scales)
    assert q.STATUS_NAMES[st] == "QERL_ERR_RANGE"
    codes[2, 48:64] = 0x88                                                  # -0 codes only: holds nothing
    st, _, _ = _pack_status(q, codes, scales)
    assert st == 0
    st, _, S0 = _pack_status(q, np.zeros_like(codes), scales)
    assert st == 0 and S0 == 1.0
