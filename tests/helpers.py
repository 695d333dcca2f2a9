"""Shared helpers for the GPU parity tests (comparison bounds, tensor moves)."""
import numpy as np

# Output tolerance for the linear (fp32 accumulation, bf16 output), measured
# against bf16_RN(y_hat), the bf16 rounding of the oracle's exact fp64 result:
#   normwise  ||y - bf16(y_hat)|| / ||y_hat||          <= 1e-3
#   max       max|y - bf16(y_hat)| / max|y_hat|         <= 2e-3
# An element may instead sit one bf16 ulp away, but only when y_hat lies within
# 2^-16 (relative) of the midpoint between the two bf16 values: fp32
# accumulation legitimately rounds such values either way.  Any other
# deviation counts toward the max bound.  fp32 outputs are compared with y_hat.
NORM_TOL = 1e-3
MAX_TOL = 2e-3
FLIP_MIDPOINT_REL = 2.0 ** -16


def dev_bf16(bits: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def linear_errors(y_gpu, ref_f64: np.ndarray, oracle_mod, bf16_out: bool = True):
    """(normwise, max, excused_flips) errors of a GPU output against the fp64 oracle result."""
    got = y_gpu.float().cpu().numpy().astype(np.float64)
    ref_f64 = np.asarray(ref_f64, dtype=np.float64)
    if bf16_out:
        ref_cmp = (oracle_mod.f64_to_bf16(ref_f64).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    else:
        ref_cmp = ref_f64
    den_n = np.linalg.norm(ref_f64)
    den_m = np.abs(ref_f64).max()
    d = got - ref_cmp
    norm = np.linalg.norm(d) / den_n if den_n > 0 else np.linalg.norm(d)
    ad = np.abs(d)
    flips = np.zeros(d.shape, dtype=bool)
    if bf16_out:
        mid = (got + ref_cmp) / 2.0
        # y and bf16(y_hat) adjacent bf16 values and y_hat at their midpoint
        gb = oracle_mod.f64_to_bf16(got).astype(np.int64)
        rb = oracle_mod.f64_to_bf16(ref_cmp).astype(np.int64)
        same_sign = ((gb ^ rb) & 0x8000) == 0
        adjacent = same_sign & (np.abs((gb & 0x7FFF) - (rb & 0x7FFF)) == 1)
        flips = adjacent & (np.abs(ref_f64 - mid) <= FLIP_MIDPOINT_REL * np.abs(ref_f64))
        del mid
    counted = np.where(flips, 0.0, ad)
    mx = counted.max() / den_m if den_m > 0 else counted.max()
    return float(norm), float(mx), int(flips.sum())


def assert_linear_close(y_gpu, ref_f64, oracle_mod, bf16_out=True, what=""):
    norm, mx, flips = linear_errors(y_gpu, ref_f64, oracle_mod, bf16_out)
    assert np.all(np.isfinite(y_gpu.float().cpu().numpy())), f"{what}: non-finite output"
    assert norm <= NORM_TOL and mx <= MAX_TOL, f"{what}: normwise {norm:.3e} max {mx:.3e} (midpoint flips {flips})"
    return norm, mx
