"""Build liblpcoll.so in-tree with nvcc for sm_103a.

Each translation unit under ``csrc/`` is compiled in parallel to an object in
``_build/``, then linked (CUDA runtime static) into ``liblpcoll.so`` next to
this file. A stamp of the sources and flags skips the build when nothing
changed.
"""
import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "liblpcoll.so")
STAMP = os.path.join(BUILD, "stamp")

SOURCES = ["lpcoll_api.cu", "lpcoll_codec.cu", "lpcoll_dda_f32.cu",
           "lpcoll_dda_bf16.cu", "lpcoll_scatter_f32.cu", "lpcoll_scatter_bf16.cu",
           "lpcoll_gather.cu", "lpcoll_variants.cu", "lpcoll_host.cu",
           "lpcoll_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# -fmad=false / -prec-div=true / -ftz=false back up the explicit __f*_rn
# intrinsics: every float operation of the kernels is one IEEE operation.
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-fmad=false", "-prec-div=true", "-prec-sqrt=true",
                     "-ftz=false", "-I" + INCLUDE, "-I" + CSRC]


def nvcc():
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build liblpcoll")


def _digest(extra):
    h = hashlib.sha256()
    for d in (CSRC, INCLUDE):
        for name in sorted(os.listdir(d)):
            p = os.path.join(d, name)
            if os.path.isfile(p):
                h.update(name.encode())
                with open(p, "rb") as f:
                    h.update(f.read())
    h.update(" ".join(extra).encode())
    return h.hexdigest()


def build(force: bool = False, extra_flags=()) -> str:
    """Compile and link liblpcoll.so; returns its path."""
    flags = NVCC_FLAGS + list(extra_flags)
    digest = _digest(flags)
    if not force and os.path.exists(LIB) and os.path.exists(STAMP):
        with open(STAMP) as f:
            if f.read().strip() == digest:
                return LIB
    os.makedirs(BUILD, exist_ok=True)
    exe = nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        cmd = [exe, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s\n%s" % (src, r.stdout, r.stderr))
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [exe, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(digest)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
