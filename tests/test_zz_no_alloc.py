"""qerl_lora_linear_noalloc (the linear on the library's own fixed scratch
array) against qerl_lora_linear with a caller workspace.

Named to be collected last: it must pass both alone in a fresh process (its
first call then does the per-device set-up) and after every other test.
Two calls in a row, on different problems, are each compared with the
workspace entry point on the same inputs, within the linear's parity bounds
(normwise 1e-3, max 2e-3); the first is also checked against the oracle.
A problem whose scratch exceeds the array must be rejected untouched.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from helpers import MAX_TOL, NORM_TOL, assert_linear_close, dev_bf16, linear_errors

pytestmark = pytest.mark.gpu

QERL_ERR_WORKSPACE = 7


@pytest.fixture(scope="module")
def q():
    import nvfp4_weight_quantized_03_gb300 as mod
    mod.lib()
    return mod


class Problem:
    def __init__(self, q, m, n, k, r, sigma, seed):
        self.m, self.n, self.k, self.r = m, n, k, r
        self.W = wl.weight_f32(n, k, seed, 0)
        codes, scales, self.S = q.quantize(torch.from_numpy(self.W).cuda())
        self.wp = q.pack(codes, scales)
        self.x_bits = wl.activations_bits(m, k, seed, 1)
        self.A_bits = wl.lora_A_bits(r, k, seed, 2) if r else None
        self.B_bits = wl.lora_B_bits(n, r, seed, 3) if r else None
        self.z = wl.noise_vector(k, sigma, seed, 4) if sigma else None
        self.alpha = 2.0 * r
        self.x = dev_bf16(self.x_bits)
        self.A = dev_bf16(self.A_bits) if r else None
        self.B = dev_bf16(self.B_bits) if r else None
        self.zd = torch.from_numpy(self.z).cuda() if sigma else None

    def out(self, dtype):
        return torch.full((self.m, self.n), float("nan"), dtype=dtype, device="cuda")

    def with_workspace(self, q, dtype):
        y = self.out(dtype)
        ws = q.workspace(q.qerl_lora_linear_workspace_size(self.m, self.n, self.k, self.r))
        q.check(q.qerl_lora_linear(self.x, self.wp, self.S, self.zd, self.A, self.B, self.alpha, y, ws))
        assert q.qerl_read_status(ws) == 0
        return y

    def noalloc(self, q, dtype):
        y = self.out(dtype)
        q.check(q.qerl_lora_linear_noalloc(self.x, self.wp, self.S, self.zd, self.A, self.B, self.alpha, y))
        torch.cuda.synchronize()
        return y


def _close_to_workspace_result(y, y_ref, orc, what):
    bf16 = y.dtype == torch.bfloat16
    norm, mx, _ = linear_errors(y, y_ref.double().cpu().numpy(), orc, bf16_out=bf16)
    assert np.all(np.isfinite(y.float().cpu().numpy())), f"{what}: non-finite output"
    assert norm <= NORM_TOL and mx <= MAX_TOL, f"{what}: normwise {norm:.3e} max {mx:.3e}"


def test_noalloc_two_calls_match_workspace_entry_point(q, orc):
    p1 = Problem(q, 8, 512, 1024, 16, 1e-2, seed=21)
    p2 = Problem(q, 3, 384, 576, 8, 0.0, seed=22)
    ref1 = p1.with_workspace(q, torch.bfloat16)
    ref2 = p2.with_workspace(q, torch.float32)

    y1 = p1.noalloc(q, torch.bfloat16)
    y2 = p2.noalloc(q, torch.float32)
    _close_to_workspace_result(y1, ref1, orc, "first noalloc call")
    _close_to_workspace_result(y2, ref2, orc, "second noalloc call")

    o1 = orc.lora_linear(p1.x_bits, *orc.quantize(p1.W), z=p1.z, A_bits=p1.A_bits, B_bits=p1.B_bits,
                         alpha=p1.alpha)
    assert_linear_close(y1, o1, orc, what="first noalloc call vs oracle")


def test_noalloc_rejects_oversize_problem(q):
    m, n, k = 1024, 128, 8192  # staged activations alone need 16 MiB
    x = torch.zeros((m, k), dtype=torch.bfloat16, device="cuda")
    wp = torch.zeros(q.qerl_nvfp4_packed_size(n, k), dtype=torch.uint8, device="cuda")
    S = torch.ones(1, device="cuda")
    y = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert q.qerl_lora_linear_noalloc(x, wp, S, None, None, None, 0.0, y) == QERL_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.isnan(y.float()).all()


def test_noalloc_rejects_like_workspace_entry_point(q):
    """Calls the workspace entry point rejects are rejected here with the same code,
    before anything is enqueued (the output stays untouched): a rank that is not a
    multiple of 8, a rank above 128, and a misaligned x."""
    m, n, k = 4, 128, 256
    x_full = torch.zeros((m, k + 8), dtype=torch.bfloat16, device="cuda")
    x = x_full[:, :k]
    wp = torch.zeros(q.qerl_nvfp4_packed_size(n, k), dtype=torch.uint8, device="cuda")
    S = torch.ones(1, device="cuda")
    ws = q.workspace(q.qerl_lora_linear_workspace_size(m, n, k, 136))
    cases = [
        ("rank 12", x, torch.zeros((12, k), dtype=torch.bfloat16, device="cuda"),
         torch.zeros((n, 12), dtype=torch.bfloat16, device="cuda")),
        ("rank 136", x, torch.zeros((136, k), dtype=torch.bfloat16, device="cuda"),
         torch.zeros((n, 136), dtype=torch.bfloat16, device="cuda")),
        ("misaligned x", x_full.view(-1)[1:1 + m * k].view(m, k), None, None),
    ]
    for what, xx, A, B in cases:
        y = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
        want = q.qerl_lora_linear(xx, wp, S, None, A, B, 1.0, y, ws)
        got = q.qerl_lora_linear_noalloc(xx, wp, S, None, A, B, 1.0, y)
        torch.cuda.synchronize()
        assert want != 0, what
        assert got == want, f"{what}: noalloc {got}, workspace entry point {want}"
        assert torch.isnan(y.float()).all(), f"{what}: output written by a rejected call"
