"""Pins for the oracle's linear layer y = x_tilde W_hat^T + (alpha/r) (x_tilde A^T) B^T.

QeRL digest, section 3.4: "Low-Rank Adaptation" (Eq. 2, W + BA
with A in R^{r x k}, B in R^{d x r}: forward x W^T + x A^T B^T, both branches on
the same noisy activations), "Noise
Merging" (Eq. 9-12: the merged noise is a per-input-channel factor (1 + z)),
"NVFP4 Quantization" (Eq. 6).  Special cases reduce to a plain matmul, the
LoRA term is checked through linearity in B, Eq. 12's weight-side form is
checked against the activation-side form, and a tiny case is recomputed with
exact rational arithmetic.
"""
from fractions import Fraction

import numpy as np
import torch

import workloads as wl
from conftest import read_golden

LEVELS = [float(v) for _, v in read_golden("e2m1_levels.txt")]


def _case(m=3, n=40, k=96, r=4, seed=0, sigma=0.05):
    W = wl.weight_f32(n, k, seed, 0)
    x = wl.activations_bits(m, k, seed, 1)
    A = wl.lora_A_bits(r, k, seed, 2)
    B = wl.lora_B_bits(n, r, seed, 3, std=0.3)
    z = wl.noise_vector(k, sigma, seed, 4)
    return W, x, A, B, z


def test_no_noise_no_lora_is_plain_dequant_gemm(orc):
    W, x, A, B, z = _case()
    codes, scales, S = orc.quantize(W)
    Wh = orc.dequant(codes, scales, S)
    y = orc.lora_linear(x, codes, scales, S)
    ref = wl.bf16_bits_to_f32(x).astype(np.float64) @ Wh.T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    yB0 = orc.lora_linear(x, codes, scales, S, A_bits=A, B_bits=np.zeros_like(B), alpha=8.0)
    assert np.allclose(yB0, ref, rtol=1e-12, atol=1e-12)


def test_lora_term_is_linear_in_B(orc):
    W, x, A, B, z = _case()
    codes, scales, S = orc.quantize(W)
    alpha, r = 8.0, A.shape[0]
    y1 = orc.lora_linear(x, codes, scales, S, z=z, A_bits=A, B_bits=B, alpha=alpha)
    y0 = orc.lora_linear(x, codes, scales, S, z=z, A_bits=A, B_bits=np.zeros_like(B), alpha=alpha)
    xt = wl.bf16_bits_to_f32(orc.noise_apply(x, z)).astype(np.float64)
    lora = (alpha / r) * ((xt @ wl.bf16_bits_to_f32(A).astype(np.float64).T) @ wl.bf16_bits_to_f32(B).astype(np.float64).T)
    assert np.allclose(y1 - y0, lora, rtol=1e-10, atol=1e-12)
    assert np.abs(lora).max() > 1e-3  # the term is not trivially zero


def test_eq12_weight_side_noise_equals_activation_side(orc):
    """Without the bf16 rounding of x_tilde, x (1+z) W_hat^T == x (W_hat (.) (1+z))^T
    with (1+z) scaling the INPUT channels (columns of W_hat, N x K)."""
    W, x, A, B, z = _case(n=24, k=64)
    codes, scales, S = orc.quantize(W)
    Wh = orc.dequant(codes, scales, S)
    y = orc.lora_linear(x, codes, scales, S, z=z, round_xt=False)
    xf = wl.bf16_bits_to_f32(x).astype(np.float64)
    ref = xf @ (Wh * (1.0 + z.astype(np.float64))[None, :]).T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-13)
    # applying the noise on the output channels instead would not match
    k, n = W.shape[1], W.shape[0]
    assert n != k


def test_zero_noise_identical_to_none(orc):
    W, x, A, B, z = _case()
    codes, scales, S = orc.quantize(W)
    a = orc.lora_linear(x, codes, scales, S, z=None, A_bits=A, B_bits=B, alpha=4.0)
    b = orc.lora_linear(x, codes, scales, S, z=np.zeros_like(z), A_bits=A, B_bits=B, alpha=4.0)
    assert np.array_equal(a, b)


def test_column_subset_matches_full(orc):
    W, x, A, B, z = _case()
    codes, scales, S = orc.quantize(W)
    full = orc.lora_linear(x, codes, scales, S, z=z, A_bits=A, B_bits=B, alpha=4.0)
    cols = np.array([39, 0, 17, 17, 5])
    sub = orc.lora_linear(x, codes, scales, S, z=z, A_bits=A, B_bits=B, alpha=4.0, cols=cols)
    assert np.array_equal(sub, full[:, cols])


def test_tiny_case_exact_rationals(orc):
    """m=2, k=32, n=3, r=2 recomputed with Fractions from the printed E2M1 levels,
    torch's E4M3 decode and torch's fp32-multiply-then-bf16 noise rounding."""
    m, n, k, r = 2, 3, 32, 2
    W, x, A, B, z = _case(m=m, n=n, k=k, r=r, seed=5, sigma=0.2)
    codes, scales, S = orc.quantize(W)
    alpha = 6.0
    y = orc.lora_linear(x, codes, scales, S, z=z, A_bits=A, B_bits=B, alpha=alpha)

    e4 = torch.from_numpy(scales.copy()).view(torch.float8_e4m3fn).double().numpy()
    xf = torch.from_numpy(wl.bf16_bits_to_f32(x))
    xt = (xf * (1.0 + torch.from_numpy(z))).to(torch.bfloat16).double().numpy()
    Af = wl.bf16_bits_to_f32(A).astype(np.float64)
    Bf = wl.bf16_bits_to_f32(B).astype(np.float64)

    def wv(i, j):
        byte = int(codes[i, j // 2])
        c = (byte >> 4) if j % 2 else (byte & 0xF)
        v = Fraction(LEVELS[c & 7]) * (-1 if c & 8 else 1)
        return Fraction(float(S)) * Fraction(float(e4[i, j // 16])) * v

    for mi in range(m):
        t = [sum(Fraction(float(xt[mi, kk])) * Fraction(float(Af[j, kk])) for kk in range(k)) for j in range(r)]
        for c in range(n):
            base = sum(Fraction(float(xt[mi, kk])) * wv(c, kk) for kk in range(k))
            lora = Fraction(alpha) / r * sum(t[j] * Fraction(float(Bf[c, j])) for j in range(r))
            exact = float(base + lora)
            assert abs(y[mi, c] - exact) <= 1e-13 * max(1.0, abs(exact))


def test_output_rounding_to_bf16(orc):
    y = np.array([1.0, 1.0 + 2 ** -8, -3.3, 1e-40, 7e38])
    b = orc.f64_to_bf16(y)
    back = (b.astype(np.uint32) << 16).view(np.float32)
    assert back[0] == 1.0 and back[1] == 1.0  # tie to even
    assert np.isinf(back[4])


# Per-row (per-rollout) noise: the digest's AQN section says each rollout may see a different
# epsilon; the broadcast of Eq. 9 is the case where every row gets the same vector.


def test_per_row_noise_with_identical_rows_is_the_broadcast(orc):
    W, x, A, B, z = _case()
    codes, scales, S = orc.quantize(W)
    zz = np.tile(z, (x.shape[0], 1))
    a = orc.lora_linear(x, codes, scales, S, z=z, A_bits=A, B_bits=B, alpha=4.0)
    b = orc.lora_linear(x, codes, scales, S, z=zz, A_bits=A, B_bits=B, alpha=4.0)
    assert np.array_equal(a, b)
    assert np.array_equal(orc.noise_apply(x, z), orc.noise_apply(x, zz))


def test_per_row_noise_reaches_only_its_row(orc):
    W, x, A, B, z = _case(m=4)
    codes, scales, S = orc.quantize(W)
    zz = np.tile(z, (4, 1))
    zz[2] = wl.noise_vector(z.size, 0.05, 0, 9)
    base = orc.lora_linear(x, codes, scales, S, z=z, A_bits=A, B_bits=B, alpha=4.0)
    y = orc.lora_linear(x, codes, scales, S, z=zz, A_bits=A, B_bits=B, alpha=4.0)
    for i in (0, 1, 3):
        assert np.array_equal(y[i], base[i])
    assert not np.array_equal(y[2], base[2])
    # and row 2 is the broadcast linear of its own noise vector
    alone = orc.lora_linear(x[2:3], codes, scales, S, z=zz[2], A_bits=A, B_bits=B, alpha=4.0)
    assert np.array_equal(y[2:3], alone)


def test_per_row_noise_eq12_each_row(orc):
    """Eq. 12 per row: row i of x (1 + z_i) W_hat^T equals x_i (W_hat (.) (1 + z_i))^T."""
    W, x, A, B, z = _case(n=24, k=64, m=3)
    codes, scales, S = orc.quantize(W)
    Wh = orc.dequant(codes, scales, S)
    zz = np.stack([wl.noise_vector(64, 0.05, 0, 20 + i) for i in range(3)])
    y = orc.lora_linear(x, codes, scales, S, z=zz, round_xt=False)
    xf = wl.bf16_bits_to_f32(x).astype(np.float64)
    for i in range(3):
        ref = xf[i] @ (Wh * (1.0 + zz[i].astype(np.float64))[None, :]).T
        assert np.allclose(y[i], ref, rtol=1e-12, atol=1e-13)
