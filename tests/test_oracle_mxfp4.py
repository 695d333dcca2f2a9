"""Pins for the oracle's MXFP4 format (the 4-bit format the digest compares with NVFP4).

QeRL digest, "NVFP4 Quantization", comparison to other 4-bit formats: E2M1 elements with one
shared E8M0 scale per block of 32 elements.  The scale rule is the OCP MX reading
X = 2^(floor(log2(amax)) - 2).  Pinned by properties of that rule (the block max lands in
[4, 8) X), brute-force nearest levels, exact round trips, idempotence, the error bound, and the
digest's own comparison (coarser blocks, larger error than NVFP4).
"""
import math

import numpy as np
import pytest

import workloads as wl
from conftest import read_golden

LEVELS = sorted({abs(float(v)) for _, v in read_golden("e2m1_levels.txt")})  # 0, .5, 1, 1.5, 2, 3, 4, 6


def _nearest_level(q):
    """Brute force: the E2M1 magnitude nearest to q >= 0, ties to the even code, saturating at 6."""
    best = min(range(len(LEVELS)), key=lambda i: (abs(LEVELS[i] - q), i % 2))
    return LEVELS[best]


def test_e8m0_decodes_to_doubling_powers_of_two(orc):
    assert orc.e8m0_decode(127) == 1.0
    for c in range(254):
        assert orc.e8m0_decode(c + 1) == 2.0 * orc.e8m0_decode(c)
    assert math.isnan(orc.e8m0_decode(255))


def _blocks(W, scales, orc):
    n, k = W.shape
    for i in range(n):
        for b in range(k // 32):
            yield W[i, 32 * b:32 * b + 32], orc.e8m0_decode(int(scales[i, b])), (i, b)


def test_block_max_lands_in_four_to_eight_scales(orc):
    W = wl.weight_f32(16, 256, 0, 11)
    codes, scales = orc.mxfp4_quantize(W)
    for blk, X, _ in _blocks(W, scales, orc):
        assert 4.0 <= np.abs(blk).max() / X < 8.0


def test_every_element_is_its_nearest_level(orc):
    W = wl.weight_f32(8, 128, 1, 12)
    codes, scales = orc.mxfp4_quantize(W)
    Wh = orc.mxfp4_dequant(codes, scales)
    for blk, X, (i, b) in _blocks(W, scales, orc):
        for j, w in enumerate(blk):
            got = Wh[i, 32 * b + j]
            assert abs(got) / X == _nearest_level(abs(float(w)) / X)
            assert got == 0.0 or np.sign(got) == np.sign(w)


def test_representable_tensor_round_trips(orc):
    g = wl.rng(0, 13)
    n, k = 4, 128
    W = np.empty((n, k), np.float32)
    for i in range(n):
        for b in range(k // 32):
            X = 2.0 ** int(g.integers(-20, 10))
            lv = np.array(LEVELS, np.float64)[g.integers(0, len(LEVELS), 32)] * g.choice([-1.0, 1.0], 32)
            lv[int(g.integers(0, 32))] = 6.0  # the block max sets the scale to X
            W[i, 32 * b:32 * b + 32] = (lv * X).astype(np.float32)
    codes, scales = orc.mxfp4_quantize(W)
    assert np.array_equal(orc.mxfp4_dequant(codes, scales), W.astype(np.float64))


def test_idempotent_and_error_bound(orc):
    W = wl.weight_f32(16, 256, 2, 14)
    codes, scales = orc.mxfp4_quantize(W)
    Wh = orc.mxfp4_dequant(codes, scales)
    c2, s2 = orc.mxfp4_quantize(Wh.astype(np.float32))
    assert np.array_equal(c2, codes) and np.array_equal(s2, scales)
    for blk, X, (i, b) in _blocks(W, scales, orc):
        assert np.abs(blk - Wh[i, 32 * b:32 * b + 32]).max() <= 2.0 * X  # 2X: the saturated tail


def test_coarser_than_nvfp4(orc):
    """The digest's comparison: 32-element power-of-two scales lose more than NVFP4's 16-element
    E4M3 scales on the same weights."""
    W = wl.weight_f32(64, 1024, 3, 15)
    codes, scales = orc.mxfp4_quantize(W)
    e_mx = np.sqrt(np.mean((orc.mxfp4_dequant(codes, scales) - W) ** 2))
    nc, ns, S = orc.quantize(W)
    e_nv = np.sqrt(np.mean((orc.dequant(nc, ns, S) - W) ** 2))
    assert e_nv < e_mx


def test_zero_block_and_bad_input(orc):
    W = np.zeros((2, 64), np.float32)
    codes, scales = orc.mxfp4_quantize(W)
    assert np.all(codes == 0) and np.all(scales == 0)
    W[1, 5] = np.inf
    with pytest.raises(Exception):
        orc.mxfp4_quantize(W)
    with pytest.raises(Exception):
        orc.mxfp4_quantize(np.ones((1, 48), np.float32))


# ---- the MXFP4 linear (orc_mxfp4_lora_linear) --------------------------------------------

def _mx_weights(orc, n, k, seed):
    W = wl.weight_f32(n, k, seed, 0)
    return orc.mxfp4_quantize(W)


def test_mx_linear_is_the_plain_matmul_of_the_dequantized_weight(orc):
    """No noise, no LoRA: y = x . W_hat^T with W_hat from the MXFP4 decoder, checked against a
    numpy fp64 matmul (only the summation order differs)."""
    m, n, k = 5, 96, 256
    codes, scales = _mx_weights(orc, n, k, 201)
    x_bits = wl.activations_bits(m, k, 202, 1)
    x = (x_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = x @ orc.mxfp4_dequant(codes, scales).T
    got = orc.mxfp4_lora_linear(x_bits, codes, scales)
    assert np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_mx_linear_equals_the_nvfp4_linear_on_a_shared_weight(orc):
    """An NVFP4 weight whose tensor scale and block scales are powers of two, equal over each pair of
    16-blocks, is also an MXFP4 weight (E8M0 code = log2(S * dec(s)) + 127).  Both oracle linears
    must then agree bit for bit, noise, per-row noise, LoRA and column subsets included (this pins
    the 32-block scale index and the absence of a tensor scale in the MXFP4 row decoder)."""
    rng = np.random.default_rng(203)
    m, n, k, r = 6, 40, 192, 8
    codes = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    exps = rng.integers(-9, 9, size=(n, k // 32))                      # E4M3 holds 2^-9 .. 2^8 exactly
    e4m3 = np.where(exps >= -6, (exps + 7) << 3, 1 << (exps + 9)).astype(np.uint8)
    nv_scales = np.repeat(e4m3, 2, axis=1)
    assert all(orc.e4m3_decode(int(e4m3[i, j])) == 2.0 ** int(exps[i, j]) for i in range(n) for j in range(k // 32))
    S_exp = -3
    mx_scales = (exps + S_exp + 127).astype(np.uint8)
    x_bits = wl.activations_bits(m, k, 204, 1)
    z = (rng.standard_normal((m, k)) * 1e-2).astype(np.float32)
    A_bits, B_bits = wl.lora_A_bits(r, k, 205, 2), wl.lora_B_bits(n, r, 206, 3)
    cols = np.array([0, 3, 17, 39, 5])
    for zz in (None, z[0], z):
        nv = orc.lora_linear(x_bits, codes, nv_scales, 2.0 ** S_exp, z=zz, A_bits=A_bits, B_bits=B_bits,
                             alpha=16.0, cols=cols)
        mx = orc.mxfp4_lora_linear(x_bits, codes, mx_scales, z=zz, A_bits=A_bits, B_bits=B_bits, alpha=16.0,
                                   cols=cols)
        assert np.array_equal(nv, mx)
