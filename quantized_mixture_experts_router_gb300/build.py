"""Build libmoe_v41.so in-tree: every .cu under csrc/ compiled for sm_103a in
parallel, then linked into one shared library exporting the C-ABI of
include/moe_v41.h."""
from __future__ import annotations

import glob
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
SO = os.path.join(OUT_DIR, "libmoe_v41.so")
# measurement support, not part of the library: the tensor-core rate microbenchmark bench.py --mma-rates runs
PEAKS_SRC = os.path.join(HERE, "peaks", "mma_rate.cu")
PEAKS_SO = os.path.join(OUT_DIR, "libmma_rate.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr"]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def build(verbose_ptxas: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    objs, procs = [], []
    for src in sources():
        obj = os.path.join(OUT_DIR, os.path.basename(src)[:-3] + ".o")
        cmd = [NVCC, *ARCH, *FLAGS, "-c", src, "-o", obj]
        if verbose_ptxas:
            cmd += ["-Xptxas", "-v"]
        objs.append(obj)
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    peaks = [NVCC, *ARCH, *FLAGS, "-shared", PEAKS_SRC, "-o", PEAKS_SO]
    procs.append((peaks, subprocess.Popen(peaks, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    errs, logs = [], []
    for cmd, p in procs:
        out, _ = p.communicate()
        logs.append(out.decode(errors="replace"))
        if p.returncode != 0:
            errs.append(" ".join(cmd) + "\n" + out.decode(errors="replace"))
    if errs:
        raise RuntimeError("moe_v41 build failed:\n" + "\n".join(errs))
    link = [NVCC, *ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", SO, "-lcudart"]
    p = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if p.returncode != 0:
        raise RuntimeError("moe_v41 link failed:\n" + p.stdout.decode(errors="replace"))
    return "\n".join(logs)


if __name__ == "__main__":
    import sys
    print(build(verbose_ptxas="-v" in sys.argv))
