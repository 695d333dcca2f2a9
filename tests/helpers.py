"""Shared helpers for the GPU parity tests (comparison bounds, tensor moves)."""
import numpy as np

# Output tolerance for the linear (fp32 accumulation, bf16 output), measured
# against the oracle's fp64 result y_hat:
#   normwise  ||y - bf16(y_hat)|| / ||y_hat||          <= 1e-3
#   max       max|y - bf16(y_hat)| / max|y_hat|         <= 2e-3
NORM_TOL = 1e-3
MAX_TOL = 2e-3


def dev_bf16(bits: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def linear_errors(y_gpu, ref_f64: np.ndarray, oracle_mod, bf16_out: bool = True):
    """(normwise, max) errors of a GPU output against the fp64 oracle result."""
    got = y_gpu.float().cpu().numpy().astype(np.float64)
    if bf16_out:
        ref_cmp = (oracle_mod.f64_to_bf16(ref_f64).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    else:
        ref_cmp = ref_f64
    den_n = np.linalg.norm(ref_f64)
    den_m = np.abs(ref_f64).max()
    d = got - ref_cmp
    norm = np.linalg.norm(d) / den_n if den_n > 0 else np.linalg.norm(d)
    mx = np.abs(d).max() / den_m if den_m > 0 else np.abs(d).max()
    return float(norm), float(mx)


def assert_linear_close(y_gpu, ref_f64, oracle_mod, bf16_out=True, what=""):
    norm, mx = linear_errors(y_gpu, ref_f64, oracle_mod, bf16_out)
    assert np.all(np.isfinite(y_gpu.float().cpu().numpy())), f"{what}: non-finite output"
    assert norm <= NORM_TOL and mx <= MAX_TOL, f"{what}: normwise {norm:.3e} max {mx:.3e}"
    return norm, mx
