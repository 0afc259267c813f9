"""A plain C program against liblpcoll.so and include/lpcoll.h: it compiles
and links here (no GPU needed) and, on a GPU, runs the pages' torch.full
allreduce example through the C ABI alone."""
import os
import shutil
import subprocess

import pytest

from precision_collective_reduction_gb300 import build as lib_build

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "c", "lpcoll_c_example.c")


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def compile_example(out_path):
    lib = lib_build.build()
    cuda = _cuda_home()
    libdir = os.path.dirname(lib)
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra",
           "-I" + lib_build.INCLUDE, "-I" + os.path.join(cuda, "include"), SRC,
           "-o", out_path, "-L" + libdir, "-llpcoll",
           "-L" + os.path.join(cuda, "lib64"), "-lcudart", "-lm",
           "-Wl,-rpath," + libdir, "-Wl,-rpath," + os.path.join(cuda, "lib64")]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out_path


def test_c_program_compiles_and_links(tmp_path):
    exe = compile_example(str(tmp_path / "lpcoll_c_example"))
    assert os.path.exists(exe)


@pytest.mark.gpu
def test_c_program_runs(tmp_path):
    exe = compile_example(str(tmp_path / "lpcoll_c_example"))
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "ok"
