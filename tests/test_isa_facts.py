"""Facts about the sm_103a instruction set that the kernels' design rests on, checked with the
toolchain on the CPU: the fifth-generation tensor core has no int8 MMA kind on this target (so the
int8 products go through exact fp16 conversion), while the fp16 kind the tensor-memory arm uses
assembles."""
import os
import shutil
import subprocess
import tempfile

import pytest

NVCC = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"

SRC = r'''
#include <cstdint>
__global__ void k(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, int acc) {
  asm volatile("{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::KIND [%0], %1, %2, %3, p;\n}"
               :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
'''


def _assemble(kind):
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "k.cu")
        with open(src, "w") as f:
            f.write(SRC.replace("KIND", kind))
        return subprocess.run([NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-c", src, "-o", os.path.join(d, "k.o")],
                              capture_output=True, text=True)


@pytest.mark.skipif(not os.path.exists(NVCC), reason="nvcc not found")
def test_tcgen05_has_no_int8_kind_on_sm_103a():
    r = _assemble("i8")
    assert r.returncode != 0
    assert "kind::i8" in r.stderr and "not supported" in r.stderr


@pytest.mark.skipif(not os.path.exists(NVCC), reason="nvcc not found")
def test_tcgen05_fp16_kind_assembles_on_sm_103a():
    r = _assemble("f16")
    assert r.returncode == 0, r.stderr
