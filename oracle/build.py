"""Compile the plain-C oracle into oracle/_build/libqerl_oracle.so.

Test infrastructure only: the CUDA library never links or loads it.
Flags keep every float operation a single IEEE operation (no contraction
into FMA, no fast-math), so fp32 decisions match the stated op order.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "qerl_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
OUT = os.path.join(OUT_DIR, "libqerl_oracle.so")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off",
          "-fno-strict-aliasing", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Build the oracle library if missing or older than its source; return its path."""
    if (not force and os.path.exists(OUT)
            and os.path.getmtime(OUT) >= os.path.getmtime(SRC)):
        return OUT
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = OUT + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
