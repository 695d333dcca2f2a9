"""Build libqerl.so in-tree with nvcc for sm_103a (GB300).

Each .cu file compiles in its own nvcc process (in parallel), then one link
step produces nvfp4_weight_quantized_03_gb300/libqerl.so.  No cmake, no torch
extension machinery: the library is plain C ABI + CUDA runtime.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libqerl.so")
SOURCES = ["api.cu", "quantize.cu", "aqn.cu", "linear.cu", "backward.cu", "noalloc.cu"]
HEADERS = ["qerl_ptx.cuh", "qerl_internal.h", os.path.join("..", "..", "include", "qerl.h")]

GENCODE = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "-Xcudafe", "--diag_suppress=177"]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


# A test-only variant (QERL_TEST_HOOKS: settable wait limit and a barrier
# arrival that never comes), loaded only by the failure-detection test.
LIB_TEST_HOOKS = os.path.join(HERE, "libqerl_testhooks.so")


def build(force: bool = False, verbose: bool = False, test_hooks: bool = False) -> str:
    nvcc = nvcc_path()
    build_dir = BUILD + ("_hooks" if test_hooks else "")
    lib_out = LIB_TEST_HOOKS if test_hooks else LIB
    extra = ["-DQERL_TEST_HOOKS"] if test_hooks else []
    os.makedirs(build_dir, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS]
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s, *hdrs]):
            jobs.append([nvcc, *GENCODE, *NVCC_FLAGS, *extra, "-c", s, "-o", o])
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            results = list(ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs))
        for cmd, res in zip(jobs, results):
            if verbose or res.returncode != 0:
                sys.stderr.write(res.stdout + res.stderr)
            if res.returncode != 0:
                raise RuntimeError(f"nvcc failed: {' '.join(cmd)}")
    if force or jobs or _stale(lib_out, objs):
        tmp = lib_out + f".tmp{os.getpid()}"
        cmd = [nvcc, *GENCODE, "-shared", "-o", tmp, *objs, "-lcudart_static", "-ldl", "-lpthread", "-lrt"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            sys.stderr.write(res.stdout + res.stderr)
            raise RuntimeError("link failed")
        os.replace(tmp, lib_out)
    return lib_out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
