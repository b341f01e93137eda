"""Build ``libvf_relayout.so`` in-tree with nvcc for sm_103a (GB300).

One translation unit, one ``-gencode``; the CUDA runtime is linked
statically so the library needs nothing but the driver at load time.
"""
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
SOURCES = [os.path.join(CSRC, "vf_relayout.cu")]
DEPS = SOURCES + [os.path.join(CSRC, "relayout_kernel.cuh"), os.path.join(CSRC, "launch.cuh"),
                  os.path.join(ROOT, "include", "vf_relayout.h")]
LIB = os.path.join(PKG, "libvf_relayout.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc():
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = os.path.join(home, "bin", "nvcc")
    return exe if os.path.exists(exe) else "nvcc"


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(d) > t for d in DEPS)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not stale():
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = [nvcc(), "-O3", "-std=c++17", "-lineinfo", *ARCH,
           "-Xcompiler", "-fPIC,-O2,-Wall", "-shared",
           "-I", os.path.join(ROOT, "include"), "-o", tmp, *SOURCES]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
