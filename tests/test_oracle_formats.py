"""Pins for the oracle's element formats (E2M1, E4M3, bf16 rounding).

Each check compares the oracle with something other than itself: the level
set printed in the QeRL digest (section 3.4 "NVFP4 Quantization"), brute-force
nearest search, or torch's own float8_e4m3fn / bfloat16 conversions.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import read_golden

LEVELS = [float(v) for _, v in read_golden("e2m1_levels.txt")]


def brute_e2m1(v: float) -> int:
    """Nearest of the printed levels; on an exact tie the even code wins; |v| > 6 -> 6."""
    a = abs(v)
    best, bestd = None, None
    for code, lv in enumerate(LEVELS):
        d = abs(Fraction(a) - Fraction(lv))
        if bestd is None or d < bestd or (d == bestd and code % 2 == 0):
            best, bestd = code, d
    if best != 0 and np.signbit(v):
        best |= 8
    return best


def test_e2m1_decode_matches_printed_levels(orc):
    for code, lv in enumerate(LEVELS):
        assert orc.e2m1_decode(code) == lv
        assert orc.e2m1_decode(code | 8) == -lv
    assert max(LEVELS) == 6.0  # q_max


def test_e2m1_encode_bruteforce_dense_sweep(orc):
    pts = set()
    for lv in LEVELS:
        pts.add(lv)
    mids = [(LEVELS[i] + LEVELS[i + 1]) / 2 for i in range(len(LEVELS) - 1)]
    for p in mids + LEVELS + [6.5, 7.0, 12.0, 1e30]:
        f = np.float32(p)
        pts.update([float(f), float(np.nextafter(f, np.float32(0))), float(np.nextafter(f, np.float32(np.inf)))])
    rs = np.random.default_rng(1)
    pts.update(rs.uniform(0, 8, 4000).astype(np.float32).tolist())
    pts.update((np.arange(0, 8 * 64 + 1) / 64.0).tolist())  # every 1/64 incl. all midpoints
    for p in sorted(pts):
        for v in (p, -p):
            v32 = float(np.float32(v))
            assert orc.e2m1_encode(v32) == brute_e2m1(v32), v32


def test_e2m1_roundtrip_every_level_at_scales(orc):
    for scale in (1.0, 2.0 ** -3, 2.0 ** 5):
        for code in range(16):
            if code == 8:
                continue
            v = orc.e2m1_decode(code) * scale
            c = orc.e2m1_encode(np.float32(v / scale))
            assert c == code
    # -0 and tiny negatives encode as +0 (reading)
    assert orc.e2m1_encode(-0.0) == 0
    assert orc.e2m1_encode(-0.1) == 0


def test_e4m3_decode_all_codes_vs_torch(orc):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        v = orc.e4m3_decode(c)
        if np.isnan(ref[c]):
            assert np.isnan(v), c
        else:
            assert v == ref[c], c


def test_e4m3_golden_points(orc):
    for h, v in read_golden("e4m3_points.txt"):
        c = int(h, 16)
        assert orc.e4m3_decode(c) == float(v)
        assert orc.e4m3_encode(float(v)) == c


def test_e4m3_encode_vs_torch_cast(orc):
    # every positive finite code value, the midpoints between neighbours, +-1 ulp
    vals = sorted({orc.e4m3_decode(c) for c in range(0x7F)})
    pts = set(vals)
    for a, b in zip(vals[:-1], vals[1:]):
        mid = np.float32((a + b) / 2)
        pts.update([float(mid), float(np.nextafter(mid, np.float32(0))), float(np.nextafter(mid, np.float32(1e9)))])
    pts.update(np.random.default_rng(2).uniform(0, 464, 20000).astype(np.float32).tolist())
    pts.update((np.random.default_rng(3).uniform(0, 1, 5000) * 2.0 ** -6).astype(np.float32).tolist())
    arr = np.array(sorted(p for p in pts if p <= 464.0), dtype=np.float32)
    ref = torch.from_numpy(arr).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(float(v)) for v in arr], dtype=np.uint8)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(arr[i], got[i], ref[i]) for i in bad[:10]]


def test_e4m3_saturates(orc):
    for v in (448.0, 463.9, 464.0, 465.0, 1000.0, 3e38):
        assert orc.e4m3_encode(v) == 0x7E


def test_noise_apply_matches_torch_fp32_then_bf16(orc):
    import workloads as wl
    rs = np.random.default_rng(4)
    x = wl.to_bf16_bits(rs.standard_normal((5, 96)).astype(np.float32) * 3)
    z = (rs.standard_normal(96) * 0.05).astype(np.float32)
    got = orc.noise_apply(x, z)
    xf = torch.from_numpy(wl.bf16_bits_to_f32(x))
    ref = (xf * (1.0 + torch.from_numpy(z))).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)
    assert np.array_equal(orc.noise_apply(x, None), x)


def exact_bf16_round(d: float) -> float:
    """Nearest bf16 to d by exact rational comparison of the two bracketing bf16 values."""
    if d == 0:
        return 0.0
    f = np.float32(d)  # a nearby float; bracket around it in bf16 steps
    bits = int(np.array([f], dtype=np.float32).view(np.uint32)[0]) & 0xFFFF0000
    cands = []
    for delta in (-2, -1, 0, 1, 2):
        b = (bits + (delta << 16)) & 0xFFFFFFFF
        c = float(np.array([b], dtype=np.uint32).view(np.float32)[0])
        if np.isfinite(c):
            cands.append(c)
    D = Fraction(d)
    best = min(cands, key=lambda c: (abs(Fraction(c) - D),
                                     int(np.array([c], dtype=np.float32).view(np.uint32)[0] >> 16) & 1))
    return best


def test_f64_to_bf16_single_rounding(orc):
    rs = np.random.default_rng(5)
    d = np.concatenate([rs.standard_normal(3000) * 10.0 ** rs.integers(-30, 30, 3000),
                        [1.0 + 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -40, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8)]])
    got = orc.f64_to_bf16(d)
    gotf = (got.astype(np.uint32) << 16).view(np.float32)
    for i in range(d.size):
        assert gotf[i] == exact_bf16_round(float(d[i])), d[i]


@pytest.mark.parametrize("lv", [0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
def test_e2m1_times_e4m3_exact_in_fp16_and_bf16(orc, lv):
    """Every level x every finite E4M3 scale is exactly representable in fp16 and
    bf16 (<= 6 significant bits, magnitude in [2^-10, 2688]): dequantizing a
    weight to 16 bits before the contraction loses nothing."""
    for c in range(0x7F):
        p = lv * orc.e4m3_decode(c)
        assert float(np.float16(p)) == p
        assert float(torch.tensor(p, dtype=torch.float64).to(torch.bfloat16).to(torch.float64)) == p
