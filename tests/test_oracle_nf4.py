"""Pins for the oracle's NF4 format (the QLoRA 4-bit format the digest contrasts with NVFP4).

QeRL digest, "NVFP4 Quantization" (comparison to other 4-bit formats) and "QLoRA's 4-bit
Quantization Addresses Memory but Degrades Speed": NF4 places its
levels at quantiles of the Gaussian and recovers them through a lookup table.  The construction
(evenly spaced probabilities, 8 positive / 7 negative quantiles and an exact zero, normalised to
[-1, 1]) is a reading; it is pinned to scipy's normal quantile function, which the oracle does not
use (it bisects erfc).  The encoder is pinned by brute-force nearest levels, the quantizer by
recomputing each block's scale and each element's level in numpy, and the linear by the plain
matmul and by bit-equality with the NVFP4 linear on a weight both formats hold.
"""
import numpy as np
import pytest

import workloads as wl

scipy_stats = pytest.importorskip("scipy.stats")


def _construction():
    p = ((1 - 1 / 32) + (1 - 1 / 30)) / 2
    pos = scipy_stats.norm.ppf(0.5 + np.arange(1, 9) / 8 * (p - 0.5))
    neg = -scipy_stats.norm.ppf(0.5 + np.arange(1, 8) / 7 * (p - 0.5))
    top = scipy_stats.norm.ppf(p)
    return np.sort(np.concatenate([neg, [0.0], pos]) / top)


def test_levels_are_normalised_gaussian_quantiles(orc):
    lv = orc.nf4_levels()
    assert np.max(np.abs(lv - _construction())) < 1e-13
    assert lv[0] == -1.0 and lv[15] == 1.0 and lv[7] == 0.0
    assert np.all(np.diff(lv) > 0) and (lv < 0).sum() == 7 and (lv > 0).sum() == 8


def test_encoder_is_the_nearest_level(orc):
    lv = orc.nf4_levels()
    mids64 = (lv[:-1] + lv[1:]) / 2
    mids = mids64.astype(np.float32)
    qs = np.linspace(-1.2, 1.2, 4801).astype(np.float32)
    for q in qs:
        if np.min(np.abs(float(q) - mids64)) < 1e-6:
            continue
        assert orc.nf4_encode(q) == int(np.argmin(np.abs(lv - float(q))))
    for i, m in enumerate(mids):  # on a midpoint: up; one ulp below: down
        assert orc.nf4_encode(m) == i + 1
        assert orc.nf4_encode(np.nextafter(m, np.float32(-2))) == i
    assert orc.nf4_encode(np.float32(-0.0)) == 7 and orc.nf4_encode(np.float32(5.0)) == 15


def test_quantizer_scales_and_codes(orc):
    W = wl.weight_f32(24, 256, 500, 1)
    codes, scales, S = orc.nf4_quantize(W)
    assert S == np.float32(np.max(np.abs(W))) / np.float32(448.0)
    lv = orc.nf4_levels()
    mids = ((lv[:-1] + lv[1:]) / 2).astype(np.float32)
    for i in range(W.shape[0]):
        for b in range(W.shape[1] // 16):
            blk = W[i, 16 * b:16 * b + 16]
            amax_b = np.float32(np.max(np.abs(blk)))
            assert scales[i, b] == orc.e4m3_encode(float(amax_b / np.float32(S)))
            sc = np.float32(S) * np.float32(orc.e4m3_decode(int(scales[i, b])))
            q = (blk / sc).astype(np.float32)
            want = np.searchsorted(mids, q, side="right")
            got = [(codes[i, 8 * b + t // 2] >> (4 * (t % 2))) & 0xF for t in range(16)]
            assert list(want) == got


def test_linear_is_the_plain_matmul_of_the_dequantized_weight(orc):
    m, n, k = 4, 80, 256
    codes, scales, S = orc.nf4_quantize(wl.weight_f32(n, k, 501, 1))
    x_bits = wl.activations_bits(m, k, 502, 1)
    x = wl.bf16_bits_to_f32(x_bits).astype(np.float64)
    ref = x @ orc.nf4_dequant(codes, scales, S).T
    got = orc.nf4_lora_linear(x_bits, codes, scales, S)
    assert np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_linear_equals_the_nvfp4_linear_on_a_shared_weight(orc):
    """Codes for -1, 0, +1 only: NF4 codes 0 / 7 / 15 and E2M1 codes 0xA / 0 / 0x2 decode to the
    same values under the same scales, so both oracle linears agree bit for bit."""
    rng = wl.rng(503, 1)
    m, n, k, r = 5, 24, 128, 8
    sym = rng.integers(0, 3, size=(n, k))
    nf4 = np.array([0, 7, 15], np.uint8)[sym]
    e2m1 = np.array([0xA, 0x0, 0x2], np.uint8)[sym]
    pack = lambda c: (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
    scales = rng.integers(0x20, 0x60, size=(n, k // 16)).astype(np.uint8)
    x_bits = wl.activations_bits(m, k, 504, 1)
    z = (rng.standard_normal(k) * 1e-2).astype(np.float32)
    A_bits, B_bits = wl.lora_A_bits(r, k, 505, 2), wl.lora_B_bits(n, r, 506, 3)
    a = orc.nf4_lora_linear(x_bits, pack(nf4), scales, 0.25, z=z, A_bits=A_bits, B_bits=B_bits, alpha=16.0)
    b = orc.lora_linear(x_bits, pack(e2m1), scales, 0.25, z=z, A_bits=A_bits, B_bits=B_bits, alpha=16.0)
    assert np.array_equal(a, b)
