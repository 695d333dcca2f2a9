"""Pins for the oracle's NVFP4 quantizer and dequantizer.

QeRL digest, section 3.4 "NVFP4 Quantization": Eq. 6 dequant
W_hat = S_FP32 * (S_E4M3 (.) W_tilde), one E4M3 scale per 16 contiguous
elements, one FP32 tensor scale.  The encoder is a reading (nearest level,
scales from block amax with the tensor scale amax/(6*448)); these tests pin it
by brute force, by exact reconstruction and by invariants.
"""
import numpy as np
import pytest

import workloads as wl
from conftest import read_golden

LEVELS = [float(v) for _, v in read_golden("e2m1_levels.txt")]


def _unpack(codes):
    lo = codes & 0xF
    hi = codes >> 4
    out = np.empty((codes.shape[0], codes.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    return out


def _level_value(c):
    v = np.array(LEVELS)[c & 7]
    return np.where(c & 8, -v, v)


@pytest.fixture(scope="module")
def wmat():
    return wl.weight_f32(24, 256, 11, 0)


def test_shapes_and_zero_tensor(orc):
    W = np.zeros((3, 64), np.float32)
    codes, scales, S = orc.quantize(W)
    assert codes.shape == (3, 32) and scales.shape == (3, 4)
    assert S == 1.0 and not codes.any() and not scales.any()


def test_nonfinite_rejected(orc):
    for bad in (np.nan, np.inf, -np.inf):
        W = np.ones((2, 32), np.float32)
        W[1, 5] = bad
        with pytest.raises(orc.OracleError):
            orc.quantize(W)


def test_k_must_be_multiple_of_32(orc):
    with pytest.raises(orc.OracleError):
        orc.quantize(np.ones((2, 48), np.float32))


def test_block_scale_is_nearest_e4m3_of_block_ratio(orc, wmat):
    """Brute force over all 127 non-negative finite E4M3 codes for every block."""
    codes, scales, S = orc.quantize(wmat)
    e4 = np.array([orc.e4m3_decode(c) for c in range(0x7F)])
    blocks = np.abs(wmat).reshape(wmat.shape[0], -1, 16).max(axis=2).astype(np.float32)
    r = (blocks / np.float32(6.0)) / np.float32(S)  # fp32 ops, the reading's order
    for (i, b), rv in np.ndenumerate(r):
        d = np.abs(e4 - float(rv))
        cand = np.nonzero(d == d.min())[0]
        want = cand[0] if cand.size == 1 else [c for c in cand if c % 2 == 0][0]
        if rv > 448.0:
            want = 0x7E
        assert scales[i, b] == want, (i, b, rv)


def test_every_element_is_nearest_level(orc, wmat):
    """Each code is the nearest E2M1 level to w / (S * dec(scale)) (fp32 quotient),
    ties to the even code; this pins the element encode, the nibble order and the
    use of the decoded (not the raw) scale."""
    codes, scales, S = orc.quantize(wmat)
    c = _unpack(codes)
    sc = (np.float32(S) * np.array([orc.e4m3_decode(s) for s in scales.ravel()], dtype=np.float32)
          .reshape(scales.shape)).astype(np.float32)
    sc_full = np.repeat(sc, 16, axis=1)
    q = (wmat / sc_full).astype(np.float32)
    lv = np.array(LEVELS)
    for idx in zip(*np.nonzero(np.ones_like(c, bool))):
        qa = abs(float(q[idx]))
        d = np.abs(lv - qa)
        cand = np.nonzero(d == d.min())[0]
        want = cand[0] if cand.size == 1 else [x for x in cand if x % 2 == 0][0]
        if qa > 6.0:
            want = 7
        if want != 0 and q[idx] < 0:
            want |= 8
        assert c[idx] == want, (idx, q[idx])


def test_tensor_scale_uses_full_ranges(orc, wmat):
    """The block holding amax(|W|) gets the largest E4M3 scale (448) and its
    largest element the largest E2M1 level (6): S = amax / (6 * 448)."""
    codes, scales, S = orc.quantize(wmat)
    i, j = np.unravel_index(np.argmax(np.abs(wmat)), wmat.shape)
    assert scales[i, j // 16] == 0x7E
    assert _unpack(codes)[i, j] & 7 == 7
    amax = float(np.abs(wmat).max())
    assert abs(float(S) * 6 * 448 - amax) <= 2e-7 * amax


def test_exactly_representable_weights_roundtrip(orc):
    """Build W = S0 * dec(s_b) * level with S0 a power of two and a +-6 in every
    block: quantization must return exactly those codes, scales and S0."""
    rs = np.random.default_rng(12)
    n, k = 6, 128
    S0 = np.float32(2.0 ** -9)
    sc_codes = rs.integers(1, 0x7F, size=(n, k // 16)).astype(np.uint8)
    sc_codes[0, 0] = 0x7E  # one block at the top scale so amax = S0 * 2688
    lvl = rs.integers(0, 16, size=(n, k)).astype(np.uint8)
    lvl[lvl == 8] = 0
    lvl[:, ::16] = 7  # a 6 in every block
    dec = np.vectorize(orc.e4m3_decode)(sc_codes)
    W = (S0 * np.repeat(dec, 16, axis=1) * _level_value(lvl)).astype(np.float32)
    # exactness of the construction itself
    assert np.array_equal(W.astype(np.float64), float(S0) * np.repeat(dec, 16, axis=1) * _level_value(lvl))
    codes, scales, S = orc.quantize(W)
    assert S == S0
    assert np.array_equal(scales, sc_codes)
    assert np.array_equal(_unpack(codes), lvl)
    assert np.array_equal(orc.dequant(codes, scales, S), W.astype(np.float64))


def test_dequant_is_eq6(orc, wmat):
    """Eq. 6 element by element from the printed levels and torch's E4M3 decode."""
    import torch
    codes, scales, S = orc.quantize(wmat)
    dq = orc.dequant(codes, scales, S)
    e4 = torch.from_numpy(scales.copy()).view(torch.float8_e4m3fn).double().numpy()
    want = float(S) * (np.repeat(e4, 16, axis=1) * _level_value(_unpack(codes)))
    assert np.array_equal(dq, want)


def test_idempotent(orc):
    """Q(D(Q(W))) == Q(W): codes, scales and the tensor scale S."""
    for seed in range(6):
        W = wl.weight_f32(16, 512, 20 + seed, 0, std=10.0 ** (seed - 3))
        codes, scales, S = orc.quantize(W)
        W2 = orc.dequant(codes, scales, S).astype(np.float32)
        c2, s2, S2 = orc.quantize(W2)
        assert S2 == S
        assert np.array_equal(s2, scales)
        assert np.array_equal(c2, codes)


def test_tensor_scale_fixed_point_many(orc):
    """For S = fl(a / 2688): fl(fl(S * 2688) / 2688) == S on 4M random a.  This is
    what idempotence needs (the dequantized maximum is fl(S * 2688)).  It does
    NOT hold for arbitrary fp32 S (about 16% fail), only for quotients by 2688."""
    rs = np.random.default_rng(13)
    a = (rs.uniform(1, 2, 4000000) * 2.0 ** rs.integers(-60, 60, 4000000)).astype(np.float32)
    S = (a / np.float32(2688.0)).astype(np.float32)
    back = ((S * np.float32(2688.0)).astype(np.float32) / np.float32(2688.0)).astype(np.float32)
    assert np.array_equal(back, S)


def test_quantization_error_bound_eq5(orc, wmat):
    """Eq. 5 error Q(w) - w per element is at most half the gap between the two
    levels around w / sc (times sc) for unclipped elements, and the clip error
    for |w / sc| > 6."""
    codes, scales, S = orc.quantize(wmat)
    dq = orc.dequant(codes, scales, S)
    sc = float(S) * np.repeat(np.vectorize(orc.e4m3_decode)(scales), 16, axis=1)
    err = np.abs(dq - wmat.astype(np.float64))
    q = np.abs(wmat / sc)
    gaps = np.where(q < 2, 0.25, np.where(q < 4, 0.5, 1.0))
    bound = np.where(q <= 6, gaps * sc, (q - 6) * sc) * (1 + 1e-6)
    assert np.all(err <= bound + 1e-30)


def test_storage_matches_4p5_bits(orc):
    """Packed storage is 4.5 bits per weight (0.5 B code + 1/16 B scale)."""
    W = wl.weight_f32(32, 2048, 1, 0)
    codes, scales, S = orc.quantize(W)
    assert (codes.nbytes + scales.nbytes) * 8 / W.size == 4.5
