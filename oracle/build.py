"""Compile the CPU oracle (``lpcoll_oracle.c``) into ``liblpcoll_oracle.so``.

Test infrastructure: the oracle is the correctness reference for the CUDA
library and is never linked into it. Built single-threaded with
``-O2 -ffp-contract=off`` so that no multiply-add is fused (gcc fuses by
default on aarch64, which would change the rounded results).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "lpcoll_oracle.c")
LIB = os.path.join(HERE, "liblpcoll_oracle.so")

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
          "-fPIC", "-shared", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


def build_source(src_text: str, out_path: str) -> str:
    """Compile C source text (a modified copy of the oracle) to out_path."""
    src_path = out_path + ".c"
    with open(src_path, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", *CFLAGS, src_path, "-o", out_path, "-lm"],
                   check=True)
    return out_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
