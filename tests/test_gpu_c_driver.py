"""The C ABI from plain C: build tests/c_abi_driver.c against the headers and
the in-tree library (no PyTorch in the process) and run it on the GPU."""
import os
import subprocess

import pytest


pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_driver(tmp_path):
    from sequence_head_relayout_gb300 import _build
    lib = _build.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = tmp_path / "c_abi_driver"
    subprocess.run(["gcc", "-std=c99", "-O1", "-Wall", "-Werror",
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                    os.path.join(ROOT, "tests", "c_abi_driver.c"), "-o", str(exe),
                    "-L", os.path.dirname(lib), "-lvf_relayout",
                    "-L", os.path.join(cuda, "lib64"), "-lcudart",
                    "-Wl,-rpath," + os.path.dirname(lib) + ":" + os.path.join(cuda, "lib64")],
                   check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert "c driver ok" in out.stdout
