"""The CUDA-error path of the C ABI, without a fault: in a process that sees
no CUDA device, a call whose arguments pass every host check reaches the
pointer query, which fails, and the call returns VF_ERR_CUDA (nothing is
launched).  Runs the same way with or without a GPU on the machine."""
import os
import subprocess
import sys

import pytest

import sequence_head_relayout_gb300 as vf

pytestmark = pytest.mark.usefixtures("lib_built")

PROBE = r"""
import ctypes, sys
lib = ctypes.CDLL(sys.argv[1])
I64 = ctypes.c_int64
f = lib.vf_qkv_pack
f.argtypes = [ctypes.c_void_p, ctypes.POINTER(I64)] + [I64] * 5 + [ctypes.c_void_p] * 2
f.restype = ctypes.c_int
st = (I64 * 4)(96, 32, 8, 1)
rc = f(1 << 40, st, 4, 4, 8, 2, 1, 1 << 41, None)
g = lib.vf_status_string
g.argtypes = [ctypes.c_int]
g.restype = ctypes.c_char_p
print(rc, g(rc).decode())
"""


def test_no_visible_device_returns_cuda_error():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, "-c", PROBE, vf.LIB_PATH], env=env,
                         capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    rc, _, msg = out.stdout.strip().partition(" ")
    assert int(rc) == -4 and "CUDA" in msg
