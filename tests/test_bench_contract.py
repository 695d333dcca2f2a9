"""bench.py's reference arm (the oracle on host cores) against the output contract, on CPU:
one JSON line with the metric, unit, direction, a cpu_baseline object, an e2e object with no
host-device bytes and no GPU launches; under torch.distributed.run with two ranks only rank 0
prints (the other exits 0 without work)."""
import json
import os
import subprocess
import sys

import pytest

from conftest import ROOT

BENCH = os.path.join(ROOT, "bench.py")


def _json_lines(out):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def _check(line):
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "dtype", "data", "config", "cpu_baseline", "e2e", "gpu_launches"):
        assert key in line, key
    assert line["value"] > 0 and line["unit"] == "GB/s" and line["higher_is_better"] is True
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    e2e = line["e2e"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0 and e2e["value"] == line["value"]
    assert line["gpu_launches"] == 0 and line["dtype"] == "f64"


def test_reference_arm_single_process():
    env = dict(os.environ)
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        env.pop(k, None)
    r = subprocess.run([sys.executable, BENCH, "--impl", "reference", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check(lines[0])
    assert lines[0]["n_gpus"] == 1 and lines[0]["steps"] == 1 and lines[0]["warmup"] == 3


def test_reference_arm_two_ranks_rank0_reports():
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", "29533", BENCH, "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1, r.stdout[-2000:]
    _check(lines[0])
    assert lines[0]["n_gpus"] == 2


_RANKS_SCRIPT = r"""
import os, sys
import torch.distributed as dist
sys.path.insert(0, os.environ["QERL_ROOT"])
import bench
world, rank, _ = bench.dist_env()
dist.init_process_group("gloo")
got = bench.max_over_ranks(1.5 + rank, world, "cpu")
with open(os.path.join(os.environ["QERL_OUT"], f"rank{rank}.txt"), "w") as f:
    f.write(f"{rank} {world} {got}")
dist.destroy_process_group()
"""


def test_timing_is_max_over_two_gloo_ranks(tmp_path):
    """The replica path's job time is the slowest rank's, and every rank sees it (two gloo ranks)."""
    script = tmp_path / "ranks.py"
    script.write_text(_RANKS_SCRIPT)
    env = dict(os.environ, QERL_ROOT=str(ROOT), QERL_OUT=str(tmp_path))
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", "29541", str(script)],
                       capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    got = [(tmp_path / f"rank{i}.txt").read_text().split() for i in range(2)]
    assert got == [["0", "2", "2.5"], ["1", "2", "2.5"]]


def test_aqn_schedule_table():
    """The bench's schedule table: every schedule starts at sigma_start, ends at sigma_end and
    decreases; the host cost is reported."""
    import importlib
    sys.path.insert(0, str(ROOT))
    bench = importlib.import_module("bench")
    import nvfp4_weight_quantized_03_gb300 as q
    t = bench.aqn_schedule_table(q, calls=100)
    for name in ("exponential", "linear", "cosine", "logarithmic"):
        sig = t[name]
        assert len(sig) == t["num_stages"] and sig[0] == t["sigma_start"]
        assert abs(sig[-1] - t["sigma_end"]) <= 1e-9 and all(b < a for a, b in zip(sig, sig[1:]))
    assert t["host_ns_per_call_incl_ctypes"] > 0
