"""C-ABI checks that need no GPU: the library builds and loads, exports every
entry point declared in include/qerl.h, its host-only functions agree with the
oracle, and argument validation rejects bad calls before touching the device.
Also checks that the product package and the oracle never import each other."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

from conftest import ROOT

import nvfp4_weight_quantized_03_gb300 as q


@pytest.fixture(scope="module")
def L():
    from nvfp4_weight_quantized_03_gb300 import build
    build.build()
    return q.lib()


def declared_symbols():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"QERL_API\s+[\w\s\*]+?\b(qerl_\w+)\s*\(", text)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(L):
    names = declared_symbols()
    assert len(names) >= 12
    out = subprocess.run(["nm", "-D", "--defined-only", q.lib_path()], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r" T (\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        getattr(L, n)  # resolvable through ctypes too


def test_status_strings(L):
    for code, name in q.STATUS_NAMES.items():
        assert q.status_string(code) == name
    assert q.status_string(99) == "QERL_ERR_UNKNOWN"


def test_host_schedule_matches_oracle(L, orc):
    for K in (1, 2, 5, 10):
        for stage in range(-2, K + 3):
            for s0, s1 in ((1e-2, 5e-4), (0.1, 1e-3)):
                assert q.qerl_aqn_sigma(stage, K, s0, s1) == orc.aqn_sigma(stage, K, s0, s1)
    for sch in range(4):
        for K in (1, 2, 5, 10):
            for stage in range(-2, K + 3):
                lib_v = q.qerl_aqn_sigma_schedule(sch, stage, K, 1e-2, 5e-4)
                orc_v = orc.aqn_sigma_schedule(sch, stage, K, 1e-2, 5e-4)
                assert abs(lib_v - orc_v) <= 4e-16 * abs(orc_v), (sch, K, stage)
    import math
    assert math.isnan(q.qerl_aqn_sigma_schedule(4, 1, 10, 1e-2, 5e-4))
    header = open(os.path.join(ROOT, "include", "qerl.h")).read()
    enum = dict(re.findall(r"QERL_SCHEDULE_(\w+) = (\d+)", header))
    assert len(enum) == 4
    for name, val in enum.items():
        assert getattr(q, "QERL_SCHEDULE_" + name) == int(val)
    for total in (1, 7, 600, 8192):
        for K in (1, 3, 10):
            for step in list(range(-2, 30)) + [total - 1, total, 5 * total]:
                assert q.qerl_aqn_stage(step, total, K) == orc.aqn_stage(step, total, K)


# The validation tests pass fake (non-dereferenceable) pointers; a call that
# unexpectedly passed validation would launch on them.  They only run where no
# GPU is visible, so such a mistake cannot reach a device.
no_gpu_only = pytest.mark.skipif(__import__("torch").cuda.is_available(),
                                 reason="fake-pointer validation tests run only without a GPU")


def _lin(L, **kw):
    a = dict(x=0x1000, m=4, k=128, ldx=128, w=0x2000, ts=0x4000, n=256, z=None, A=None,
             B=None, r=0, alpha=0.0, y=0x5000, ydt=q.QERL_BF16, ws=0x10000, wsb=1 << 30, stream=None)
    a.update(kw)
    return L.qerl_lora_linear(a["x"], a["m"], a["k"], a["ldx"], a["w"], a["ts"], a["n"], a["z"], a["A"], a["B"],
                              a["r"], a["alpha"], a["y"], a["ydt"], a["ws"], a["wsb"], a["stream"])


@no_gpu_only
def test_linear_validation(L):
    E = q.STATUS_NAMES
    name = lambda st: E[st]
    assert name(_lin(L, k=96, ldx=96)) == "QERL_ERR_UNSUPPORTED_SHAPE"
    assert name(_lin(L, k=0)) == "QERL_ERR_INVALID_ARGUMENT"
    assert name(_lin(L, m=-1)) == "QERL_ERR_INVALID_ARGUMENT"
    assert name(_lin(L, ldx=64)) == "QERL_ERR_INVALID_ARGUMENT"
    assert name(_lin(L, A=0x6000)) == "QERL_ERR_INVALID_ARGUMENT"  # A without B
    assert name(_lin(L, A=0x6000, B=0x7000, r=0)) == "QERL_ERR_INVALID_ARGUMENT"
    assert name(_lin(L, A=0x6000, B=0x7000, r=129)) == "QERL_ERR_UNSUPPORTED_SHAPE"
    assert name(_lin(L, ydt=7)) == "QERL_ERR_INVALID_ARGUMENT"
    assert name(_lin(L, x=None)) == "QERL_ERR_INVALID_ARGUMENT"
    assert name(_lin(L, x=0x1008)) == "QERL_ERR_MISALIGNED"
    assert name(_lin(L, ldx=132)) == "QERL_ERR_MISALIGNED"
    assert name(_lin(L, w=0x2004)) == "QERL_ERR_MISALIGNED"
    assert name(_lin(L, w=None)) == "QERL_ERR_INVALID_ARGUMENT"
    assert name(_lin(L, z=0x8004)) == "QERL_ERR_MISALIGNED"
    assert name(_lin(L, ws=None)) == "QERL_ERR_WORKSPACE"
    need = L.qerl_lora_linear_workspace_size(4, 256, 128, 0)
    assert name(_lin(L, wsb=need - 1)) == "QERL_ERR_WORKSPACE"
    assert name(_lin(L, ws=0x10080)) == "QERL_ERR_MISALIGNED"
    assert _lin(L, m=0) == 0 and _lin(L, n=0) == 0  # empty problems are no-ops


def _desc(**kw):
    a = dict(wpacked=0x2000, tensor_scale=0x4000, n=256, A=None, B=None, r=0, alpha=0.0, y=0x5000,
             y_dtype=q.QERL_BF16)
    a.update(kw)
    d = q.LinearDesc()
    for f, v in a.items():
        setattr(d, f, v)
    return d


def _group(L, descs, **kw):
    a = dict(x=0x1000, m=4, k=128, ldx=128, z=None, ws=0x10000, wsb=1 << 30)
    a.update(kw)
    arr = (q.LinearDesc * max(len(descs), 1))(*descs)
    return L.qerl_lora_linear_group(a["x"], a["m"], a["k"], a["ldx"], a["z"], arr if descs else None,
                                    len(descs), a["ws"], a["wsb"], None)


@no_gpu_only
def test_group_validation(L):
    E = q.STATUS_NAMES
    ok = _desc()
    assert E[_group(L, [])] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[_group(L, [ok] * 5)] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[_group(L, [ok, _desc(y_dtype=5)])] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[_group(L, [ok, _desc(w_format=2)])] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[_group(L, [ok, _desc(A=0x6000)])] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[_group(L, [ok, _desc(A=0x6000, B=0x7000, r=12)])] == "QERL_ERR_UNSUPPORTED_SHAPE"
    assert E[_group(L, [ok, _desc(wpacked=0x2008)])] == "QERL_ERR_MISALIGNED"
    assert E[_group(L, [ok, _desc(wpacked=None)])] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[_group(L, [ok, _desc(y=0x5001)])] == "QERL_ERR_MISALIGNED"
    assert E[_group(L, [ok, _desc(y=0x5002, y_dtype=q.QERL_F32)])] == "QERL_ERR_MISALIGNED"
    assert E[_group(L, [ok], k=96, ldx=96)] == "QERL_ERR_UNSUPPORTED_SHAPE"
    # a member with n == 0 is dropped before its pointers are checked; all empty: no-op
    assert _group(L, [_desc(n=0, wpacked=None, y=None)], m=4) == 0
    assert _group(L, [ok, ok], m=0) == 0
    # the group workspace covers every member's LoRA partials
    lo = L.qerl_lora_linear_group_workspace_size(4, 128, (q.LinearDesc * 1)(ok), 1)
    hi = L.qerl_lora_linear_group_workspace_size(
        4, 128, (q.LinearDesc * 2)(ok, _desc(A=0x6000, B=0x7000, r=64)), 2)
    assert 0 < lo < hi
    assert E[_group(L, [ok, _desc(A=0x6000, B=0x7000, r=64)], wsb=hi - 1)] == "QERL_ERR_WORKSPACE"
    assert L.qerl_lora_linear_group_workspace_size(4, 128, (q.LinearDesc * 1)(ok), 5) == 0


def test_linear_descs_built_once():
    """A group's descriptor array, built once, carries each member's fields and is passed
    through unchanged by the group call's marshalling."""
    y = torch.empty((4, 256), dtype=torch.bfloat16)
    y32 = torch.empty((4, 128), dtype=torch.float32)
    A = torch.empty((16, 128), dtype=torch.bfloat16)
    B = torch.empty((256, 16), dtype=torch.bfloat16)
    arr = q.linear_descs([(0x2000, 0x3000, A, B, 32.0, y), (0x4000, 0x3010, None, None, 0.0, y32)])
    assert q._descs(arr) is arr
    d0, d1 = arr[0], arr[1]
    assert (d0.wpacked, d0.tensor_scale, d0.n, d0.r, d0.alpha) == (0x2000, 0x3000, 256, 16, 32.0)
    assert (d0.A, d0.B, d0.y, d0.y_dtype) == (A.data_ptr(), B.data_ptr(), y.data_ptr(), q.QERL_BF16)
    assert (d1.wpacked, d1.n, d1.r, d1.A, d1.B, d1.y_dtype) == (0x4000, 128, 0, None, None, q.QERL_F32)


@no_gpu_only
def test_pack_validation(L):
    E = q.STATUS_NAMES
    pk = lambda **kw: L.qerl_nvfp4_pack(kw.get("codes", 0x2000), kw.get("scales", 0x3000), kw.get("n", 4),
                                        kw.get("k", 128), kw.get("packed", 0x8000), None)
    assert E[pk(k=96)] == "QERL_ERR_UNSUPPORTED_SHAPE"
    assert E[pk(n=-1)] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[pk(packed=None)] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[pk(codes=0x2008)] == "QERL_ERR_MISALIGNED"
    assert E[pk(scales=0x3002)] == "QERL_ERR_MISALIGNED"
    assert pk(n=0) == 0


def test_packed_size(L):
    # one 18432-byte block per 128 rows x 256 K, partial tiles rounded up
    assert L.qerl_nvfp4_packed_size(128, 256) == 18432
    assert L.qerl_nvfp4_packed_size(129, 256) == 2 * 18432
    assert L.qerl_nvfp4_packed_size(3584, 3584) == 28 * 14 * 18432
    assert L.qerl_nvfp4_packed_size(512, 320) == 4 * 2 * 18432
    assert L.qerl_nvfp4_packed_size(0, 256) == 0


def test_workspace_size_grows(L):
    a = L.qerl_lora_linear_workspace_size(1, 128, 64, 0)
    b = L.qerl_lora_linear_workspace_size(128, 128, 3584, 32)
    assert a >= 256 and a % 256 == 0 and b > a
    assert b >= 128 * 3584 * 2 + 128 * 32 * 4
    assert L.qerl_nvfp4_quantize_workspace_size() == 256


@no_gpu_only
def test_quantize_validation(L):
    E = q.STATUS_NAMES
    qz = lambda **kw: L.qerl_nvfp4_quantize(
        kw.get("W", 0x1000), kw.get("dt", q.QERL_F32), kw.get("n", 4), kw.get("k", 64), kw.get("ld", 64),
        kw.get("codes", 0x2000), kw.get("scales", 0x3000), kw.get("ts", 0x4000), kw.get("ws", 0x10000),
        kw.get("wsb", 256), None)
    assert E[qz(k=48, ld=48)] == "QERL_ERR_UNSUPPORTED_SHAPE"
    assert E[qz(dt=5)] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[qz(ld=32)] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[qz(W=0x1004)] == "QERL_ERR_MISALIGNED"
    assert E[qz(ld=66)] == "QERL_ERR_MISALIGNED"
    assert E[qz(codes=0x2008)] == "QERL_ERR_MISALIGNED"
    assert E[qz(ts=None)] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[qz(wsb=255)] == "QERL_ERR_WORKSPACE"
    assert E[L.qerl_aqn_sample(None, -1, 1.0, 0, 0, 0, None)] == "QERL_ERR_INVALID_ARGUMENT"
    assert L.qerl_aqn_sample(None, 0, 1.0, 0, 0, 0, None) == 0


def test_mxfp4_validation(L):
    """The MXFP4 entry points reject bad arguments on the host, before any device work."""
    E = q.STATUS_NAMES
    qz = lambda **kw: L.qerl_mxfp4_quantize(
        kw.get("W", 0x1000), kw.get("dt", q.QERL_BF16), kw.get("n", 4), kw.get("k", 64), kw.get("ld", 64),
        kw.get("codes", 0x2000), kw.get("scales", 0x3000), kw.get("ws", 0x10000), kw.get("wsb", 256), None)
    assert E[qz(k=48, ld=48)] == "QERL_ERR_UNSUPPORTED_SHAPE"
    assert E[qz(dt=7)] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[qz(ld=32)] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[qz(W=0x1002)] == "QERL_ERR_MISALIGNED"
    assert E[qz(codes=0x2004)] == "QERL_ERR_MISALIGNED"
    assert E[qz(scales=None)] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[qz(wsb=128)] == "QERL_ERR_WORKSPACE"
    assert E[qz(ws=0x10080)] == "QERL_ERR_MISALIGNED"
    pk = lambda **kw: L.qerl_mxfp4_pack(
        kw.get("codes", 0x2000), kw.get("scales", 0x3001), kw.get("n", 4), kw.get("k", kw.get("k", 128)),
        kw.get("packed", 0x4000), kw.get("ts", 0x5000), kw.get("ws", 0x10000), kw.get("wsb", 256), None)
    assert E[pk(k=96)] == "QERL_ERR_UNSUPPORTED_SHAPE"
    assert E[pk(k=65536 + 64)] == "QERL_ERR_UNSUPPORTED_SHAPE"
    assert E[pk(n=-1)] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[pk(ts=None)] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[pk(packed=None)] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[pk(packed=0x4008)] == "QERL_ERR_MISALIGNED"
    assert E[pk(codes=0x2001)] == "QERL_ERR_MISALIGNED"
    assert E[pk(wsb=0)] == "QERL_ERR_WORKSPACE"
    assert L.qerl_status_string(8) == b"QERL_ERR_RANGE"


def test_backward_validation(L):
    """The backward and the transposed pack reject bad arguments on the host."""
    E = q.STATUS_NAMES
    bw = lambda **kw: L.qerl_lora_linear_backward(
        kw.get("xt", 0x1000), kw.get("m", 4), kw.get("k", 512), kw.get("ldxt", 512), kw.get("dy", 0x2000),
        kw.get("n", 256), kw.get("lddy", 256), kw.get("wp", 0x3000), kw.get("ts", 0x4000), kw.get("A", 0x5000),
        kw.get("B", 0x6000), kw.get("r", 16), 32.0, kw.get("dxt", 0x7000), kw.get("dt", q.QERL_BF16),
        kw.get("dA", 0x8000), kw.get("dB", 0x9000), kw.get("ws", 0x10000), kw.get("wsb", 0), None)
    assert E[bw(n=96, lddy=96)] == "QERL_ERR_UNSUPPORTED_SHAPE"
    assert E[bw(k=48, ldxt=48)] == "QERL_ERR_UNSUPPORTED_SHAPE"
    assert E[bw(k=96, ldxt=96)] == "QERL_ERR_UNSUPPORTED_SHAPE"
    assert E[bw(r=12)] == "QERL_ERR_UNSUPPORTED_SHAPE"
    assert E[bw(r=136)] == "QERL_ERR_UNSUPPORTED_SHAPE"
    assert E[bw(B=None)] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[bw(dt=9)] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[bw(lddy=128)] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[bw(dy=None)] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[bw(xt=None)] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[bw(dy=0x2008)] == "QERL_ERR_MISALIGNED"
    assert E[bw(ldxt=516)] == "QERL_ERR_MISALIGNED"
    assert E[bw(wp=0x3004)] == "QERL_ERR_MISALIGNED"
    assert E[bw()] == "QERL_ERR_WORKSPACE"
    assert L.qerl_lora_linear_backward_workspace_size(4, 256, 512, 16) > 0
    pt = lambda **kw: L.qerl_nvfp4_pack_transposed(kw.get("codes", 0x1000), kw.get("scales", 0x2000),
                                                   kw.get("n", 256), kw.get("k", 512), kw.get("out", 0x3000), None)
    assert E[pt(n=96)] == "QERL_ERR_UNSUPPORTED_SHAPE"
    assert E[pt(k=48)] == "QERL_ERR_UNSUPPORTED_SHAPE"
    assert E[pt(n=65536 + 64)] == "QERL_ERR_UNSUPPORTED_SHAPE"
    assert E[pt(out=None)] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[pt(codes=0x1008)] == "QERL_ERR_MISALIGNED"


def test_nf4_quantize_validation(L):
    E = q.STATUS_NAMES
    qz = lambda **kw: L.qerl_nf4_quantize(
        kw.get("W", 0x1000), kw.get("dt", q.QERL_F32), kw.get("n", 4), kw.get("k", 64), kw.get("ld", 64),
        kw.get("codes", 0x2000), kw.get("scales", 0x3000), kw.get("ts", 0x4000), kw.get("ws", 0x10000),
        kw.get("wsb", 256), None)
    assert E[qz(k=48, ld=48)] == "QERL_ERR_UNSUPPORTED_SHAPE"
    assert E[qz(dt=5)] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[qz(ts=None)] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[qz(codes=0x2008)] == "QERL_ERR_MISALIGNED"
    assert E[qz(wsb=255)] == "QERL_ERR_WORKSPACE"


def test_product_and_oracle_are_independent():
    pkg = os.path.join(ROOT, "nvfp4_weight_quantized_03_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "oracle" not in re.findall(r"(?:import|from)\s+(\w+)", text), fn
                assert "qerl_oracle" not in text, fn
    for fn in os.listdir(os.path.join(ROOT, "oracle")):
        if fn.endswith((".py", ".c", ".h")):
            text = open(os.path.join(ROOT, "oracle", fn)).read()
            assert "nvfp4_weight_quantized_03_gb300" not in re.findall(r"(?:import|from)\s+([\w.]+)", text), fn
            assert "#include" not in text or ("qerl_ptx" not in text and "qerl.h" not in text), fn


@pytest.mark.parametrize("lang,std", [("c", "-std=c99"), ("c++", "-std=c++11")])
def test_header_is_plain_c_and_cpp(lang, std):
    """include/qerl.h is a C ABI: it compiles as pedantic C99 and as C++11 on its own."""
    import shutil
    cc = shutil.which("gcc")
    if cc is None:
        pytest.skip("no gcc")
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            r = subprocess.run([cc, "-fsyntax-only", "-x", lang, std, "-Wall", "-Wextra", "-pedantic", "-Werror",
                                os.path.join(ROOT, "include", fn)], capture_output=True, text=True)
            assert r.returncode == 0, r.stderr


@no_gpu_only
def test_rowz_and_rmsnorm_validation(L):
    """Argument checks of the per-row-noise and RMSNorm entry points (no device work)."""
    E = q.STATUS_NAMES
    arr = (q.LinearDesc * 1)(_desc())
    rowz = lambda z, ldz: L.qerl_lora_linear_group_rowz(0x1000, 4, 128, 128, z, ldz, arr, 1, 0x10000, 1 << 30, None)
    assert E[rowz(0x8000, 64)] == "QERL_ERR_INVALID_ARGUMENT"      # a row stride shorter than a row
    assert E[rowz(0x8000, 130)] == "QERL_ERR_MISALIGNED"           # rows not 16-byte aligned
    assert E[rowz(0x8004, 0)] == "QERL_ERR_MISALIGNED"
    rms = lambda **kw: L.qerl_rmsnorm_lora_linear_group(
        kw.get("h", 0x1000), kw.get("m", 4), 128, 128, kw.get("w", 0x3000), kw.get("Z", None),
        kw.get("delta", 1e-6), arr, 1, 0x10000, kw.get("wsb", 1 << 30), None)
    assert E[rms(delta=-1.0)] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[rms(delta=float("nan"))] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[rms(w=None)] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[rms(w=0x3008)] == "QERL_ERR_MISALIGNED"
    assert E[rms(Z=0x3004)] == "QERL_ERR_MISALIGNED"
    assert E[rms(m=70000)] == "QERL_ERR_UNSUPPORTED_SHAPE"
    need = L.qerl_rmsnorm_lora_linear_group_workspace_size(4, 128, arr, 1)
    assert E[rms(wsb=need - 1)] == "QERL_ERR_WORKSPACE"
    # with a LoRA branch the workspace also holds the normalised activations
    arr2 = (q.LinearDesc * 1)(_desc(A=0x6000, B=0x7000, r=16))
    assert (L.qerl_rmsnorm_lora_linear_group_workspace_size(4, 128, arr2, 1)
            >= L.qerl_lora_linear_group_workspace_size(4, 128, arr2, 1) + 4 * 128 * 2)
    norm = lambda **kw: L.qerl_rmsnorm_noise(kw.get("h", 0x1000), 4, kw.get("k", 128), kw.get("ldh", 128), 0x3000,
                                             None, 1e-6, kw.get("out", 0x5000), kw.get("ldo", 128), None)
    assert E[norm(k=124)] == "QERL_ERR_UNSUPPORTED_SHAPE"
    assert E[norm(ldh=100)] == "QERL_ERR_INVALID_ARGUMENT"
    assert E[norm(out=0x5008)] == "QERL_ERR_MISALIGNED"
    assert E[norm(ldo=132)] == "QERL_ERR_MISALIGNED"
    assert E[norm(out=None)] == "QERL_ERR_INVALID_ARGUMENT"
