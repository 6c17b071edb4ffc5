"""Build the CPU oracle (plain C, gcc).  Building the checker is not using it:
only the tests, the smoke check and the benchmark's CPU-baseline leg load it."""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
LIBDIR = os.path.join(HERE, "_lib")


def command(src=None, out=None):
    """The gcc command for the oracle library (src, out: another source and
    library path, for the planted-mistake tests)."""
    os.makedirs(LIBDIR, exist_ok=True)
    return ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread",
            src or os.path.join(HERE, "moe_oracle.c"), "-I", HERE, "-o", out or os.path.join(LIBDIR, "liboracle.so"),
            "-lm"]


def build() -> None:
    p = subprocess.run(command(), stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if p.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + p.stdout.decode(errors="replace"))


if __name__ == "__main__":
    build()
