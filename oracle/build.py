"""Compile the C oracle (``vf_oracle.c``) into ``oracle/_build/libvf_oracle.so``.

Test infrastructure: building the checker is not using it.  Plain gcc, no
architecture flags, so the same source builds on x86-64 and aarch64 hosts.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "vf_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libvf_oracle.so")


def build(force: bool = False) -> str:
    """Build the oracle library if missing or older than its source; return its path."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + ".tmp.%d" % os.getpid()
    # float32 arithmetic exactly as written: no contraction into fused
    # multiply-adds, no fast-math; libm for rintf/frexpf/ldexpf
    cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-Wall", "-Wextra", "-Werror",
           "-ffp-contract=off", "-fno-fast-math", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
