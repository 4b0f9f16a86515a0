"""Compile the scalar C oracle into oracle/_build/libmxq_oracle.so.

Test infrastructure: the oracle is the checker, not part of the product.
Plain gcc, no SIMD intrinsics, no -march flags, so the same source gives the
same results on x86-64 and aarch64 hosts.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "mxq_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libmxq_oracle.so")

CFLAGS = ["-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    os.makedirs(OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(LIB)
             or os.path.getmtime(LIB) < max(os.path.getmtime(SRC),
                                            os.path.getmtime(os.path.join(HERE, "mxq_oracle.h"))))
    if force or stale:
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", *CFLAGS, "-o", tmp, SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
