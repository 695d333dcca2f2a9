"""Pins for the oracle's RMSNorm with the noise merged into its scale.

QeRL digest, "Noise Merging": Eq. 10 (RMSNorm_noise(x) = (w + Z) * x / sqrt(mean(x^2) + delta))
and Eq. 11 (the merged noise is the per-channel factor (1 + Z / w) on the plain RMSNorm output).
Pinned by a library routine (torch's rms_norm) for Z = 0, by Eq. 11, and by properties of the
normalisation itself.
"""
import numpy as np
import torch

import workloads as wl


def _inputs(m=6, k=256, seed=0, sigma=1e-2):
    h = wl.activations_bits(m, k, seed, 500)
    w = wl.rmsnorm_weight_bits(k, seed, 501)
    Z = wl.noise_vector(k, sigma, seed, 502)
    return h, w, Z


def test_without_noise_is_torch_rms_norm(orc):
    h, w, _ = _inputs()
    out64, bits = orc.rmsnorm_noise(h, w, None, 1e-6)
    ht = torch.from_numpy(wl.bf16_bits_to_f32(h).astype(np.float64))
    wt = torch.from_numpy(wl.bf16_bits_to_f32(w).astype(np.float64))
    ref = torch.nn.functional.rms_norm(ht, (ht.shape[1],), weight=wt, eps=1e-6).numpy()
    np.testing.assert_allclose(out64, ref, rtol=1e-13, atol=0)
    assert np.array_equal(bits, orc.f64_to_bf16(out64))


def test_eq11_merged_noise_is_a_channel_factor(orc):
    for seed in range(3):
        h, w, Z = _inputs(seed=seed, sigma=1e-2 * (seed + 1))
        noisy, _ = orc.rmsnorm_noise(h, w, Z)
        plain, _ = orc.rmsnorm_noise(h, w, None)
        factor = 1.0 + Z.astype(np.float64) / wl.bf16_bits_to_f32(w).astype(np.float64)
        np.testing.assert_allclose(noisy, plain * factor, rtol=1e-13, atol=0)


def test_power_of_two_scaling_of_the_input_is_invisible(orc):
    h, w, Z = _inputs()
    a, _ = orc.rmsnorm_noise(h, w, Z, 0.0)
    for scale in (8.0, 0.25):
        hs = wl.to_bf16_bits(wl.bf16_bits_to_f32(h) * np.float32(scale))  # exact in bf16
        b, _ = orc.rmsnorm_noise(hs, w, Z, 0.0)
        assert np.array_equal(a, b)


def test_unit_scale_gives_unit_rms(orc):
    h, _, _ = _inputs(m=5, k=384)
    ones = wl.to_bf16_bits(np.ones(384, np.float32))
    out, _ = orc.rmsnorm_noise(h, ones, None, 0.0)
    np.testing.assert_allclose((out ** 2).mean(axis=1), 1.0, rtol=1e-14)


def test_zero_row(orc):
    h = np.zeros((2, 64), np.uint16)
    w = wl.rmsnorm_weight_bits(64, 0, 503)
    out, bits = orc.rmsnorm_noise(h, w, None, 1e-6)
    assert np.all(out == 0.0) and np.all(bits == 0)
    out0, _ = orc.rmsnorm_noise(h, w, None, 0.0)
    assert np.all(np.isnan(out0))  # 0 / 0, as the definition gives with delta = 0
