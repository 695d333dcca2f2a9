"""Failure detection without a GPU fault: a bounded wait that runs out.

Every mbarrier wait in the kernels is bounded (clock64); when the bound passes,
the waiting role records QERL_ERR_TIMEOUT in the workspace status word, raises
the CTA's abort flag so the other roles stop waiting, and the kernel returns
normally.  A test-only build of the library (QERL_TEST_HOOKS; the shipped
library has no such switch) lets this test shorten the bound to ~1 ms and give
the accumulator barrier one arrival that never comes: the epilogue's wait then
runs out after every MMA and every copy of the CTA has completed, so nothing is
left in flight when it gives up.  The call must come back with the status set,
quickly, and the next call on the same workspace, with the hooks off, must be
correct -- the context stays usable.  Run in a subprocess (its own CUDA context
and its own copy of the library).
"""
import json
import os
import subprocess
import sys

import pytest

from conftest import ROOT

pytestmark = pytest.mark.gpu

_SCRIPT = r"""
import ctypes, json, os, sys, time
import numpy as np
import torch
sys.path.insert(0, os.environ["QERL_ROOT"])
sys.path.insert(0, os.path.join(os.environ["QERL_ROOT"], "tests"))
import nvfp4_weight_quantized_03_gb300 as q
from nvfp4_weight_quantized_03_gb300 import build
import oracle
import workloads as wl
from helpers import linear_errors
q._build.LIB = build.build(test_hooks=True)
L = q.lib()
L.qerl_test_set_hooks.restype = ctypes.c_int
L.qerl_test_set_hooks.argtypes = [ctypes.c_longlong, ctypes.c_int]
out = {}
for name, (m, n, k, r) in {"no_cluster": (4, 256, 256, 16), "k_split_cluster": (8, 512, 3584, 32)}.items():
    W = wl.weight_f32(n, k, 61, 0)
    codes, scales, S = q.quantize(torch.from_numpy(W).cuda())
    wp = q.pack(codes, scales)
    x_bits = wl.activations_bits(m, k, 62, 1)
    A_bits, B_bits = wl.lora_A_bits(r, k, 63, 2), wl.lora_B_bits(n, r, 64, 3)
    dev = lambda b: torch.from_numpy(b.view(np.int16)).cuda().view(torch.bfloat16)
    x, A, B = dev(x_bits), dev(A_bits), dev(B_bits)
    ws = q.workspace(q.qerl_lora_linear_workspace_size(m, n, k, r))
    y = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert L.qerl_test_set_hooks(2_000_000, 1) == 0   # ~1 ms at GB300 clocks; one arrival never comes
    torch.cuda.synchronize()
    t0 = time.time()
    st_call = q.qerl_lora_linear(x, wp, S, None, A, B, 2.0 * r, y, ws)
    st_dev = q.qerl_read_status(ws)                    # synchronizes
    dt = time.time() - t0
    assert L.qerl_test_set_hooks(4_000_000_000, 0) == 0
    y2 = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    st_call2 = q.qerl_lora_linear(x, wp, S, None, A, B, 2.0 * r, y2, ws)
    st_dev2 = q.qerl_read_status(ws)
    ref = oracle.lora_linear(x_bits, *oracle.quantize(W), A_bits=A_bits, B_bits=B_bits, alpha=2.0 * r)
    norm, mx, _ = linear_errors(y2, ref, oracle)
    out[name] = {"call": st_call, "status": st_dev, "seconds": dt, "call2": st_call2, "status2": st_dev2,
                 "norm2": norm, "max2": mx, "finite2": bool(torch.isfinite(y2.float()).all().item())}
print(json.dumps(out))
"""


def test_bounded_wait_runs_out_and_context_survives(tmp_path):
    script = tmp_path / "timeout_case.py"
    script.write_text(_SCRIPT)
    env = dict(os.environ, QERL_ROOT=str(ROOT))
    r = subprocess.run([sys.executable, str(script)], capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-3000:]
    res = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])
    for name, c in res.items():
        assert c["call"] == 0, name                     # argument checks passed; the launch went out
        assert c["status"] == 5, (name, c)              # QERL_ERR_TIMEOUT recorded by the kernel
        assert c["seconds"] < 5.0, (name, c)            # the kernel returned (no hang)
        assert c["call2"] == 0 and c["status2"] == 0, (name, c)
        assert c["finite2"] and c["norm2"] <= 1e-3 and c["max2"] <= 2e-3, (name, c)
