"""What the sm_103a tensor cores accept, checked with the compiler (no GPU).

The prefill design question "int8 tcgen05 MMA tiles or fp16 ones" is settled
by the toolchain: ptxas refuses tcgen05.mma .kind::i8 for sm_103a (GB300) and
accepts the same instruction for sm_100a, while .kind::f16 is accepted for
sm_103a.  Only the compiler's answer is read here; no output is inspected."""
import os
import subprocess

import pytest

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

SRC = r'''
#include <stdint.h>
__global__ void k(uint32_t d, uint64_t a, uint64_t b, uint32_t id) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
               " tcgen05.mma.cta_group::1.kind::KIND [%0], %1, %2, %3, p;\n}\n"
               :: "r"(d), "l"(a), "l"(b), "r"(id), "r"(1) : "memory");
}
'''


def _compile(tmp_path, kind, arch):
    src = tmp_path / f"probe_{kind}_{arch}.cu"
    src.write_text(SRC.replace("KIND", kind))
    p = subprocess.run([NVCC, "-gencode", f"arch=compute_{arch},code=sm_{arch}", "-c", str(src), "-o",
                        str(tmp_path / "probe.o")], capture_output=True, text=True)
    return p.returncode, p.stdout + p.stderr


@pytest.fixture(scope="module", autouse=True)
def _nvcc():
    if not os.path.exists(NVCC):
        pytest.skip("nvcc not available")


def test_int8_mma_is_refused_for_sm103a(tmp_path):
    rc, out = _compile(tmp_path, "i8", "103a")
    assert rc != 0
    assert "not supported on .target 'sm_103a'" in out


def test_int8_mma_is_accepted_for_sm100a(tmp_path):
    rc, out = _compile(tmp_path, "i8", "100a")
    assert rc == 0, out


def test_f16_mma_is_accepted_for_sm103a(tmp_path):
    rc, out = _compile(tmp_path, "f16", "103a")
    assert rc == 0, out
