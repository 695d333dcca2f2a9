"""GPU NVFP4 quantizer vs the oracle: codes, scales and tensor scale bit-exact."""
import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import nvfp4_weight_quantized_03_gb300 as mod
    mod.lib()
    return mod


def _gpu_quant(q, W_np, bf16=False, ld=None):
    if bf16:
        Wt = torch.from_numpy(wl.to_bf16_bits(W_np).view(np.int16)).view(torch.bfloat16)
    else:
        Wt = torch.from_numpy(np.ascontiguousarray(W_np, dtype=np.float32))
    n, k = Wt.shape
    if ld is not None and ld > k:
        big = torch.zeros((n, ld), dtype=Wt.dtype)
        big[:, :k] = Wt
        Wd = big.cuda()[:, :k]
    else:
        Wd = Wt.cuda()
    codes, scales, S = q.quantize(Wd)
    return codes.cpu().numpy(), scales.cpu().numpy(), S.cpu().numpy()[0]


def _oracle_input(W_np, bf16):
    return wl.bf16_bits_to_f32(wl.to_bf16_bits(W_np)) if bf16 else np.ascontiguousarray(W_np, dtype=np.float32)


def _assert_same(q, orc, W_np, bf16=False, ld=None):
    c, s, S = _gpu_quant(q, W_np, bf16, ld)
    oc, osc, oS = orc.quantize(_oracle_input(W_np, bf16))
    assert S == oS
    assert np.array_equal(s, osc), np.argwhere(s != osc)[:5]
    assert np.array_equal(c, oc), np.argwhere(c != oc)[:5]


@pytest.mark.parametrize("n,k", [(1, 32), (3, 64), (17, 96), (200, 2048), (129, 3584)])
@pytest.mark.parametrize("bf16", [False, True])
def test_quantize_bit_exact_small(q, orc, n, k, bf16):
    _assert_same(q, orc, wl.weight_f32(n, k, 100 + n, k), bf16)


def test_quantize_strided_rows(q, orc):
    _assert_same(q, orc, wl.weight_f32(40, 256, 3, 0), False, ld=320)
    _assert_same(q, orc, wl.weight_f32(40, 256, 3, 0), True, ld=264)


def test_quantize_heavy_tail_bf16(q, orc):
    bits = wl.weight_heavy_tail_bf16(256, 5120, 0, 1)
    W = wl.bf16_bits_to_f32(bits)
    _assert_same(q, orc, W, True)


@pytest.mark.parametrize("std", [1e-30, 1e-6, 1.0, 1e6, 1e30])
def test_quantize_ranges(q, orc, std):
    _assert_same(q, orc, wl.weight_f32(64, 512, 7, 1, std=std))


def test_quantize_zero_and_tiny(q, orc):
    _assert_same(q, orc, np.zeros((8, 64), np.float32))
    W = np.zeros((8, 64), np.float32)
    W[3, 5] = np.float32(1e-44)  # subnormal: S underflows to 0 -> 1
    _assert_same(q, orc, W)


def test_quantize_all_rounding_ties(q, orc):
    """Blocks whose elements sit exactly on every E2M1 midpoint (ties) and whose
    block maxima put r exactly on E4M3 midpoints."""
    levels = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)
    mids = (levels[:-1] + levels[1:]) / 2
    rs = np.random.default_rng(0)
    n, k = 64, 256
    S0 = 2.0 ** -8
    W = np.zeros((n, k), np.float64)
    W[0, 0] = 2688 * S0  # fixes S = S0
    for i in range(n):
        for b in range(k // 16):
            if i == 0 and b == 0:
                continue
            sc = float(orc.e4m3_decode(int(rs.integers(8, 0x7E))))
            blk = rs.choice(np.concatenate([mids, levels, -mids]), 16) * sc
            blk[0] = 6 * sc  # makes r = sc exactly
            W[i, b * 16:(b + 1) * 16] = blk * S0
    # a few blocks whose r falls on an E4M3 midpoint
    e4 = np.array([orc.e4m3_decode(c) for c in range(0x7F)])
    for j, b in enumerate(range(1, 9)):
        midr = (e4[20 + 7 * j] + e4[21 + 7 * j]) / 2
        W[1, b * 16:(b + 1) * 16] = 0
        W[1, b * 16] = 6 * midr * S0
    W32 = W.astype(np.float32)
    assert np.array_equal(W32.astype(np.float64), W)  # construction is exact
    _assert_same(q, orc, W32)


def test_quantize_nonfinite_sets_status(q):
    W = torch.ones((4, 64), dtype=torch.float32, device="cuda")
    W[2, 7] = float("nan")
    codes = torch.empty((4, 32), dtype=torch.uint8, device="cuda")
    scales = torch.empty((4, 4), dtype=torch.uint8, device="cuda")
    S = torch.empty(1, dtype=torch.float32, device="cuda")
    ws = q.workspace(q.qerl_nvfp4_quantize_workspace_size())
    assert q.qerl_nvfp4_quantize(W, codes, scales, S, ws) == 0
    assert q.qerl_read_status(ws) == 6
    assert torch.isnan(S).item()
    assert q.qerl_read_status(ws) == 0  # reading clears the word
    W[2, 7] = float("inf")
    assert q.qerl_nvfp4_quantize(W, codes, scales, S, ws) == 0
    assert q.qerl_read_status(ws) == 6


def test_quantize_with_given_scale_and_amax(q, orc):
    W = wl.weight_f32(48, 512, 9, 0)
    Wd = torch.from_numpy(W).cuda()
    ws = q.workspace(256)
    amax = torch.empty(1, dtype=torch.float32, device="cuda")
    q.check(q.qerl_nvfp4_amax(Wd, amax, ws))
    assert amax.item() == float(np.abs(W).max())
    S_given = np.float32(3.0) * np.float32(np.abs(W).max() / 2688.0)
    Sd = torch.tensor([S_given], dtype=torch.float32, device="cuda")
    codes = torch.empty((48, 256), dtype=torch.uint8, device="cuda")
    scales = torch.empty((48, 32), dtype=torch.uint8, device="cuda")
    q.check(q.qerl_nvfp4_quantize_with_scale(Wd, Sd, codes, scales, ws))
    assert q.qerl_read_status(ws) == 0
    oc, osc, _ = orc.quantize(W, S=S_given)
    assert np.array_equal(scales.cpu().numpy(), osc)
    assert np.array_equal(codes.cpu().numpy(), oc)


@pytest.mark.parametrize("name,n,k,bf16", [("7B gate, fp32", 18944, 3584, False),
                                           ("32B down, bf16 heavy tail", 5120, 27648, True)])
def test_quantize_full_size(q, orc, name, n, k, bf16):
    if bf16:
        W = wl.bf16_bits_to_f32(wl.weight_heavy_tail_bf16(n, k, 0, 2))
    else:
        W = wl.weight_f32(n, k, 0, 3)
    _assert_same(q, orc, W, bf16)
