"""Pins for the oracle's LoRA backward through the frozen NVFP4 weight.

QeRL digest, "Low-Rank Adaptation (LoRA) Within Quantized Layers" (Eq. 2 and its gradient flow:
only A and B train; the quantized base weight stays frozen and passes the input gradient).
The forward oracle is linear in x~, in A and in B, so a central difference of
f = <dy, y> under a bf16-exact perturbation of one entry equals that entry's gradient up to fp64
rounding: the backward is pinned to the independently written forward, entry by entry.
"""
import numpy as np

import workloads as wl

M, N, K, R, ALPHA = 3, 32, 64, 8, 16.0


def _grid_bits(shape, seed, step, span):
    """bf16 bits of values on a grid of `step` within +-span (exact in bf16, and so is +-step)."""
    g = wl.rng(seed, 600)
    v = g.integers(-int(span / step), int(span / step) + 1, size=shape).astype(np.float32) * np.float32(step)
    return wl.to_bf16_bits(v)


def _setup(orc, seed=0):
    W = wl.weight_f32(N, K, seed, 601)
    codes, scales, S = orc.quantize(W)
    xt = _grid_bits((M, K), seed * 10 + 1, 2.0 ** -4, 4.0)
    A = _grid_bits((R, K), seed * 10 + 2, 2.0 ** -8, 0.25)
    B = _grid_bits((N, R), seed * 10 + 3, 2.0 ** -10, 0.0625)
    dy = wl.rng(seed, 602).standard_normal((M, N))
    return codes, scales, S, xt, A, B, dy


def _f(orc, codes, scales, S, xt, A, B, dy):
    y = orc.lora_linear(xt, codes, scales, S, z=None, A_bits=A, B_bits=B, alpha=ALPHA)
    return float(np.sum(dy * y))


def _bump(bits, idx, delta):
    v = wl.bf16_bits_to_f32(bits).copy()
    v[idx] += np.float32(delta)
    out = wl.to_bf16_bits(v)
    assert wl.bf16_bits_to_f32(out)[idx] == v[idx]  # the perturbed value is exact
    return out


def _check_entries(orc, which, grad, delta, args, n_entries=24, seed=0):
    codes, scales, S, xt, A, B, dy = args
    arrays = {"xt": xt, "A": A, "B": B}
    g = wl.rng(seed, 603, len(which))
    shape = arrays[which].shape
    scale = np.abs(grad).max()
    for _ in range(n_entries):
        idx = tuple(int(g.integers(0, s)) for s in shape)
        plus, minus = dict(arrays), dict(arrays)
        plus[which] = _bump(arrays[which], idx, delta)
        minus[which] = _bump(arrays[which], idx, -delta)
        fd = (_f(orc, codes, scales, S, plus["xt"], plus["A"], plus["B"], dy)
              - _f(orc, codes, scales, S, minus["xt"], minus["A"], minus["B"], dy)) / (2 * delta)
        assert abs(fd - grad[idx]) <= 1e-9 * scale, (which, idx, fd, grad[idx])


def test_input_gradient_is_the_central_difference(orc):
    args = _setup(orc)
    codes, scales, S, xt, A, B, dy = args
    dxt, _, _ = orc.lora_linear_backward(xt, codes, scales, S, A, B, ALPHA, dy)
    _check_entries(orc, "xt", dxt, 2.0 ** -4, args)


def test_adapter_gradients_are_the_central_difference(orc):
    args = _setup(orc, seed=1)
    codes, scales, S, xt, A, B, dy = args
    _, dA, dB = orc.lora_linear_backward(xt, codes, scales, S, A, B, ALPHA, dy)
    _check_entries(orc, "A", dA, 2.0 ** -8, args, seed=1)
    _check_entries(orc, "B", dB, 2.0 ** -10, args, seed=1)


def test_base_part_is_the_adjoint_of_the_forward(orc):
    """Without LoRA: <dy, xt W^T> = <dy W, xt> (the frozen weight passes the gradient back)."""
    codes, scales, S, xt, _, _, dy = _setup(orc, seed=2)
    y = orc.lora_linear(xt, codes, scales, S, z=None)
    dxt, dA, dB = orc.lora_linear_backward(xt, codes, scales, S, None, None, ALPHA, dy)
    assert dA is None and dB is None
    lhs = float(np.sum(dy * y))
    rhs = float(np.sum(dxt * wl.bf16_bits_to_f32(xt).astype(np.float64)))
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs))


def test_adapter_gradients_alone_match_the_full_call(orc):
    """want_dxt=False skips only the input gradient: dA and dB are bit-identical to the full call."""
    codes, scales, S, xt, A, B, dy = _setup(orc, seed=5)
    _, dA, dB = orc.lora_linear_backward(xt, codes, scales, S, A, B, ALPHA, dy)
    dxt2, dA2, dB2 = orc.lora_linear_backward(xt, codes, scales, S, A, B, ALPHA, dy, want_dxt=False)
    assert dxt2 is None
    assert np.array_equal(dA, dA2) and np.array_equal(dB, dB2)
