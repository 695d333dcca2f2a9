"""The GPU parity comparison itself: exact bf16 rounding passes, a one-ulp
flip is excused only when the exact value sits at the rounding midpoint, and
any other deviation counts toward the max bound."""
import numpy as np
import torch

from helpers import MAX_TOL, linear_errors


def _bf16_tensor(orc, vals):
    b = orc.f64_to_bf16(np.asarray(vals, dtype=np.float64))
    return torch.from_numpy((b.astype(np.uint32) << 16).view(np.float32).copy())


def test_exact_rounding_is_zero_error(orc):
    ref = np.random.default_rng(0).standard_normal(1000)
    norm, mx, flips = linear_errors(_bf16_tensor(orc, ref), ref, orc)
    assert norm == 0.0 and mx == 0.0 and flips == 0


def test_midpoint_flip_is_excused_but_counted_in_normwise(orc):
    ref = np.random.default_rng(1).standard_normal(1000)
    ref[0] = 1.0 + 2.0 ** -8 + 1e-12  # just above the midpoint between 1 and 1 + 2^-7
    y = _bf16_tensor(orc, ref)
    y[0] = 1.0  # the other rounding candidate
    norm, mx, flips = linear_errors(y, ref, orc)
    assert flips == 1 and mx == 0.0 and norm > 0.0


def test_off_midpoint_error_fails(orc):
    ref = np.random.default_rng(2).standard_normal(1000)
    ref[3] = 3.0 * np.abs(ref).max()
    y = _bf16_tensor(orc, ref)
    y[3] = float(y[3]) * (1 + 2.0 ** -6)
    norm, mx, flips = linear_errors(y, ref, orc)
    assert flips == 0 and mx > MAX_TOL
