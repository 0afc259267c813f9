"""Build liblpcoll.so in-tree with nvcc for sm_103a.

Each translation unit under ``csrc/`` is compiled in parallel to an object in
``_build/``, then linked (CUDA runtime static) into ``liblpcoll.so`` next to
this file. A stamp of the sources and flags skips the build when nothing
changed.
"""
import concurrent.futures as cf
import fcntl
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
# The bounds-checked build (-DLPCOLL_DEBUG_BOUNDS): every global access of the
# kernels is checked against the buffers its call passed; for tests only.
DEBUG_BUILD = os.path.join(BUILD, "debug_bounds")
DEBUG_LIB = os.path.join(PKG, "liblpcoll_debug_bounds.so")

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


def build(force: bool = False, extra_flags=(), debug_bounds: bool = False) -> str:
    """Compile and link liblpcoll.so (debug_bounds: the bounds-checked
    liblpcoll_debug_bounds.so); returns its path. Processes that build at
    the same time (the ranks of a torchrun launch) take turns on a lock
    file, and all but the first find the library up to date."""
    flags = NVCC_FLAGS + list(extra_flags) + (["-DLPCOLL_DEBUG_BOUNDS"] if debug_bounds else [])
    build_dir = DEBUG_BUILD if debug_bounds else BUILD
    lib = DEBUG_LIB if debug_bounds else LIB
    os.makedirs(build_dir, exist_ok=True)
    with open(os.path.join(build_dir, "lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        return _build_locked(force, flags, build_dir, lib)


def _build_locked(force, flags, build_dir, lib):
    stamp = os.path.join(build_dir, "stamp")
    digest = _digest(flags)
    if not force and os.path.exists(lib) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return lib
    exe = nvcc()

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [exe, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s\n%s" % (src, r.stdout, r.stderr))
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = [exe, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib)
    with open(stamp, "w") as f:
        f.write(digest)
    return lib


def build_all(force: bool = False) -> str:
    """Both libraries, compiled at once; returns the path of liblpcoll.so."""
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        main = ex.submit(build, force)
        dbg = ex.submit(build, force, (), True)
        dbg.result()
        return main.result()


if __name__ == "__main__":
    print(build_all(force="--force" in sys.argv))
