"""The sharding contract of the quantizer, on two gloo ranks (CPU, no GPU).

A weight split across devices (column- or row-parallel) must quantize to the
codes and scales of the whole tensor: every shard uses the whole tensor's S,
which needs the global amax.  Each rank holds one shard (rows 0..n/2 or n/2..n
of a seeded W), takes its local amax, all-reduces it with the library's
global_amax helper (torch.distributed, max), derives S by the quantizer's rule
(S = amax / 2688 in fp32, QeRL digest "NVFP4 Quantization", Eq. 6 with the
tensor scale read of the design notes) and quantizes its shard with the oracle.
The ranks' S must equal the oracle's S of the whole tensor, and their codes and
scales the whole tensor's rows, bit for bit."""
import os
import subprocess
import sys

import numpy as np

from conftest import ROOT

_SCRIPT = r"""
import os, sys
import numpy as np
import torch
import torch.distributed as dist
sys.path.insert(0, os.environ["QERL_ROOT"])
import oracle
import workloads as wl
import nvfp4_weight_quantized_03_gb300 as q
dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
n, k = 96, 256
W = wl.weight_f32(n, k, 5, 1)
shard = W[rank * n // world:(rank + 1) * n // world]
amax = torch.tensor([float(np.abs(shard).max())], dtype=torch.float32)
q.global_amax(amax)
S = np.float32(amax.item()) / np.float32(2688.0)
if S == 0:
    S = np.float32(1.0)
codes, scales, S_out = oracle.quantize(shard, S=float(S))
np.savez(os.path.join(os.environ["QERL_OUT"], f"rank{rank}.npz"), codes=codes, scales=scales, S=np.float32(S_out),
         amax=np.float32(amax.item()))
dist.destroy_process_group()
"""


def test_sharded_quantization_matches_whole_tensor(tmp_path, orc):
    import workloads as wl
    script = tmp_path / "shard.py"
    script.write_text(_SCRIPT)
    env = dict(os.environ, QERL_ROOT=str(ROOT), QERL_OUT=str(tmp_path))
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", "29547", str(script)],
                       capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    parts = [np.load(tmp_path / f"rank{i}.npz") for i in range(2)]
    W = wl.weight_f32(96, 256, 5, 1)
    codes, scales, S = orc.quantize(W)
    assert all(float(p["amax"]) == float(np.abs(W).max()) for p in parts)  # every rank sees the global amax
    assert all(float(p["S"]) == float(S) for p in parts)
    assert np.array_equal(np.concatenate([p["codes"] for p in parts]), codes)
    assert np.array_equal(np.concatenate([p["scales"] for p in parts]), scales)
