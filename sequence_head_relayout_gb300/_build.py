"""Build ``libvf_relayout.so`` in-tree with nvcc for sm_103a (GB300).

Two translation units (the exact relayouts with the host checks, and the
lossy-transport kernels) compiled in parallel, one ``-gencode``, then linked;
the CUDA runtime is linked statically so the library needs nothing but the
driver at load time.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
SOURCES = [os.path.join(CSRC, "vf_relayout.cu"), os.path.join(CSRC, "vf_quant.cu")]
DEPS = SOURCES + [os.path.join(CSRC, n) for n in ("relayout_kernel.cuh", "launch.cuh",
                                                  "tiled_kernel.cuh", "quant_kernel.cuh",
                                                  "quant.h")] \
    + [os.path.join(ROOT, "include", "vf_relayout.h")]
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
    tag = ".tmp.%d" % os.getpid()
    objs = [os.path.splitext(src)[0] + tag + ".o" for src in SOURCES]
    common = [nvcc(), "-O3", "-std=c++17", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC,-O2,-Wall",
              "-I", os.path.join(ROOT, "include")]
    if verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(pair):
        src, obj = pair
        subprocess.run(common + ["-c", "-o", obj, src], check=True)

    try:
        with ThreadPoolExecutor(len(SOURCES)) as ex:
            list(ex.map(compile_one, zip(SOURCES, objs)))
        tmp = LIB + tag
        subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs], check=True)
        os.replace(tmp, LIB)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
