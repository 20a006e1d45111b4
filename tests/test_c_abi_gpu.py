"""The GEMM C ABI called from plain C (tests/c_abi/gemm_from_c.c): built with gcc against
include/gb300_gemm.h and the in-tree library, it owns its CUDA buffers and checks an
integer-valued problem exactly, plus two argument errors; then the host-operand entry point
with pageable buffers, equal to the device call and exact on a taller M-major problem."""
import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_gemm_from_plain_c(tmp_path):
    from layout_algebra_gb300 import build
    lib = build.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = tmp_path / "gemm_from_c"
    cmd = ["gcc", "-std=c11", "-O1", os.path.join(ROOT, "tests", "c_abi", "gemm_from_c.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           lib, "-L", os.path.join(cuda, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.dirname(lib),
           "-Wl,-rpath," + os.path.join(cuda, "lib64"), "-o", str(exe)]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "0 of 60000 outputs wrong" in r.stdout
    assert "host call: 0 of 60000 outputs differ from the device call" in r.stdout
    assert "host call, M-major A in 4 row blocks: 0 of 870400 outputs wrong" in r.stdout
