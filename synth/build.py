"""Build the synthetic-input generator: a host library (gcc) and its GPU twin (nvcc, sm_103a)."""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
LIBDIR = os.path.join(HERE, "_lib")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


def commands():
    os.makedirs(LIBDIR, exist_ok=True)
    host = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
            os.path.join(HERE, "synth.c"), "-o", os.path.join(LIBDIR, "libsynth_host.so"), "-lm"]
    gpu = [NVCC, "-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
           "-fmad=false", "-Xcompiler", "-fPIC", "-shared", os.path.join(HERE, "synth_gpu.cu"),
           "-o", os.path.join(LIBDIR, "libsynth_gpu.so")]
    return [host, gpu]


def build() -> None:
    procs = [subprocess.Popen(c, stdout=subprocess.PIPE, stderr=subprocess.STDOUT) for c in commands()]
    errs = []
    for c, p in zip(commands(), procs):
        out, _ = p.communicate()
        if p.returncode != 0:
            errs.append(" ".join(c) + "\n" + out.decode(errors="replace"))
    if errs:
        raise RuntimeError("synth build failed:\n" + "\n".join(errs))


if __name__ == "__main__":
    build()
