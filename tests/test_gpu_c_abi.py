"""The C ABI used from a C program (tests/c/flce_c_smoke.c): caller-owned
buffers, no Python in the loop, checked against the uniform-logit closed
form (W = 0: lse = log V, loss = log V, dx = 0, dW from the softmax at 1/V)."""
import os
import shutil
import subprocess

import pytest

from linear_cross_entropy_gemm_gb300 import build as B

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def test_c_program_against_closed_form(tmp_path):
    lib = B.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cc = shutil.which("gcc")
    assert cc, "gcc missing"
    exe = tmp_path / "flce_c_smoke"
    cmd = [cc, "-std=c99", "-O2", os.path.join(HERE, "c", "flce_c_smoke.c"), "-o", str(exe),
           "-I", os.path.join(B.ROOT, "include"), "-I", os.path.join(cuda, "include"),
           os.path.abspath(lib), "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm",
           "-Wl,-rpath," + os.path.dirname(os.path.abspath(lib)) + ":" + os.path.join(cuda, "lib64")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    lines = r.stdout.splitlines()
    assert len(lines) == 3 and all(l.startswith("ok") for l in lines), r.stdout
