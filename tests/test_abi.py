"""The C ABI without a GPU: the library loads, exports every function that
include/lpcoll.h declares, and rejects bad arguments on the host before any
launch (every call below fails validation, so nothing reaches CUDA)."""
import ctypes
import os
import re

import pytest

import precision_collective_reduction_gb300 as pcr
from precision_collective_reduction_gb300 import _binding as B
from precision_collective_reduction_gb300 import build as lib_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "lpcoll.h")
OK, ARG, ALIGN, UNSUP, RANK = 0, 1, 2, 3, 4
A = 0x10000  # an aligned fake device address: never dereferenced in these calls


@pytest.fixture(scope="module")
def L():
    lib_build.build()
    return pcr.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)) -
                  {"if", "defined"})


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert {"lp_quantize", "lp_dequantize", "lp_reduce", "dda_flat_sim",
            "dda_tree_sim", "lpcoll_status_string"} <= set(names)
    for name in names:
        assert hasattr(L, name), name


def test_status_strings(L):
    for st, name in B.STATUS.items():
        assert L.lpcoll_status_string(st).decode().startswith(name)
    assert b"unknown" in L.lpcoll_status_string(99)
    assert L.lpcoll_version() == 100
    assert L.lpcoll_last_cuda_error() == 0


def arr(*ptrs):
    return B.ptr_array(ptrs)


def test_quantize_validation(L):
    assert L.lp_quantize(A, 7, 10, 128, A, A, None) == ARG
    assert L.lp_quantize(A, 0, 10, 64, A, A, None) == UNSUP
    assert L.lp_quantize(A, 0, 10, 0, A, A, None) == UNSUP
    assert L.lp_quantize(None, 0, 0, 128, None, None, None) == OK  # n == 0
    assert L.lp_quantize(None, 0, 10, 128, A, A, None) == ARG
    assert L.lp_quantize(A, 1, 10, 128, None, A, None) == ARG
    assert L.lp_quantize(A + 4, 0, 10, 128, A, A, None) == ALIGN
    assert L.lp_quantize(A, 0, 10, 128, A, A + 8, None) == ALIGN
    # NULL is reported before misalignment
    assert L.lp_quantize(A + 4, 0, 10, 128, None, A, None) == ARG


def test_dequantize_validation(L):
    assert L.lp_dequantize(A, A, 10, 128, A, 2, None) == ARG
    assert L.lp_dequantize(A, A, 10, 256, A, 0, None) == UNSUP
    assert L.lp_dequantize(A, A, 0, 128, None, 0, None) == OK
    assert L.lp_dequantize(A, None, 10, 128, A, 0, None) == ARG
    assert L.lp_dequantize(A, A, 10, 128, A + 2, 1, None) == ALIGN


def test_reduce_validation(L):
    two = arr(A, A)
    assert L.lp_reduce(two, two, 0, 10, 128, A, 0, None) == ARG
    assert L.lp_reduce(two, two, 17, 10, 128, A, 0, None) == ARG
    assert L.lp_reduce(two, two, 2, 10, 32, A, 0, None) == UNSUP
    assert L.lp_reduce(two, two, 2, 0, 128, None, 0, None) == OK
    assert L.lp_reduce(None, two, 2, 10, 128, A, 0, None) == ARG
    assert L.lp_reduce(arr(A, None), two, 2, 10, 128, A, 0, None) == RANK
    assert L.lp_reduce(two, arr(A, A + 4), 2, 10, 128, A, 0, None) == ALIGN
    assert L.lp_reduce(two, two, 2, 10, 128, None, 0, None) == ARG


@pytest.mark.parametrize("fn", ["dda_flat_sim", "dda_tree_sim"])
def test_allreduce_validation(L, fn):
    f = getattr(L, fn)
    tree = fn == "dda_tree_sim"

    def call(ins, outs, N, n, dt, block, wc, ws, sc=A, ss=A):
        if tree:
            return f(ins, outs, N, n, dt, block, wc, ws, sc, ss, None)
        return f(ins, outs, N, n, dt, block, wc, ws, None)

    two = arr(A, A)
    assert call(two, two, 2, 10, 5, 128, two, two) == ARG          # dtype
    assert call(two, two, 0, 10, 0, 128, two, two) == ARG          # N < 1
    assert call(two, two, 17, 10, 0, 128, two, two) == ARG         # N > 16
    assert call(two, two, 2, 10, 0, 64, two, two) == UNSUP         # block
    assert call(None, None, 2, 0, 0, 128, None, None) == OK        # n == 0
    assert call(None, two, 2, 10, 0, 0, None, None) == ARG
    assert call(arr(A, None), two, 2, 10, 0, 0, None, None) == RANK
    assert call(two, arr(None, A), 2, 10, 1, 0, None, None) == RANK
    assert call(two, two, 2, 10, 0, 128, None, two) == ARG         # LP needs wires
    assert call(two, two, 2, 10, 0, 128, two, arr(A, None)) == RANK
    assert call(arr(A, A + 8), two, 2, 10, 0, 0, None, None) == ALIGN
    assert call(two, two, 2, 10, 0, 128, arr(A + 1, A), two) == ALIGN
    # a NULL anywhere wins over a misaligned pointer anywhere
    assert call(arr(A + 8, A), arr(A, None), 2, 10, 0, 0, None, None) == RANK
    if tree:
        assert call(two, two, 2, 10, 0, 128, two, two, sc=None) == ARG
        assert call(two, two, 2, 10, 0, 128, two, two, ss=A + 4) == ALIGN


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(B, "_lib", None)
    with pytest.raises(RuntimeError, match="not found"):
        B.lib()


def test_library_is_built_for_sm103a():
    lib_build.build()
    assert "arch=compute_103a,code=sm_103a" in " ".join(lib_build.NVCC_FLAGS)
    assert os.path.getsize(lib_build.LIB) > 0
    ctypes.CDLL(lib_build.LIB)


@pytest.mark.parametrize("fn", ["reduce_scatter_sim", "all_gather_sim", "all_to_all_sim"])
def test_collective_validation(L, fn):
    f = getattr(L, fn)
    two = arr(A, A)
    assert f(two, two, 2, 10, 3, 128, two, two, None) == ARG        # dtype
    assert f(two, two, 0, 10, 0, 128, two, two, None) == ARG        # N < 1
    assert f(two, two, 17, 10, 0, 128, two, two, None) == ARG       # N > 16
    assert f(two, two, 2, 10, 0, 256, two, two, None) == UNSUP      # block
    assert f(None, None, 2, 0, 0, 128, None, None, None) == OK      # empty: no-op
    assert f(None, two, 2, 10, 0, 0, None, None, None) == ARG
    assert f(arr(A, None), two, 2, 10, 0, 0, None, None, None) == RANK
    assert f(two, None, 2, 10, 0, 0, None, None, None) == ARG
    assert f(two, two, 2, 10, 0, 128, None, two, None) == ARG       # LP needs wires
    assert f(two, two, 2, 10, 1, 128, two, arr(None, A), None) == RANK
    assert f(two, arr(A, A + 4), 2, 10, 0, 0, None, None, None) == ALIGN
    assert f(two, two, 2, 10, 0, 128, arr(A + 2, A), two, None) == ALIGN
    # a NULL anywhere outranks a misaligned pointer anywhere
    assert f(arr(A + 4, A), None, 2, 10, 0, 0, None, None, None) == ARG
    assert f(arr(A + 4, A), arr(A, None), 2, 10, 0, 0, None, None, None) == RANK
    assert f(two, arr(A + 4, A), 2, 10, 0, 128, arr(A, None), two, None) == RANK
    if fn == "reduce_scatter_sim":
        # n = 10 over 8 ranks: shards of 2 elements, ranks 5..7 empty. Their
        # outputs may be NULL: the call gets past the NULL checks and stops at
        # the misaligned out[0] (nothing is launched), while a NULL output of
        # a non-empty shard is refused.
        eight = arr(*([A] * 8))
        assert f(eight, arr(A + 4, A, A, A, A, None, None, None), 8, 10, 0, 0, None,
                 None, None) == ALIGN
        assert f(eight, arr(A + 4, None, A, A, A, A, A, A), 8, 10, 0, 0, None, None,
                 None) == RANK
        assert f(eight, arr(*([A] + [None] * 7)), 8, 10, 0, 128, None, None,
                 None) == ARG                                       # wires first
    else:
        assert f(two, arr(A, None), 2, 10, 0, 0, None, None, None) == RANK


def test_variant_validation(L):
    two = arr(A, A)
    assert L.lp_quantize_fmt(A, 0, 10, 128, 2, A, A, None) == ARG       # format
    assert L.lp_quantize_fmt(A, 2, 10, 128, 0, A, A, None) == ARG       # dtype
    for bad in (0, 16, 48, 512):
        assert L.lp_quantize_fmt(A, 0, 10, bad, 1, A, A, None) == UNSUP
    assert L.lp_quantize_fmt(None, 0, 0, 64, 1, None, None, None) == OK
    assert L.lp_quantize_fmt(A, 1, 10, 32, 1, None, A, None) == ARG
    assert L.lp_quantize_fmt(A, 1, 10, 256, 0, A, A + 4, None) == ALIGN
    assert L.lp_dequantize_fmt(A, A, 10, 64, 3, A, 0, None) == ARG
    assert L.lp_dequantize_fmt(A, A, 10, 100, 0, A, 0, None) == UNSUP
    assert L.lp_dequantize_fmt(A, A, 10, 64, 1, A + 2, 1, None) == ALIGN
    assert L.lp_reduce_fmt(two, two, 0, 10, 64, 1, A, 0, None) == ARG
    assert L.lp_reduce_fmt(two, two, 2, 10, 96, 1, A, 0, None) == UNSUP
    assert L.lp_reduce_fmt(arr(A, None), two, 2, 10, 64, 1, A, 0, None) == RANK
    assert L.lp_reduce_fmt(two, two, 2, 10, 64, 1, None, 0, None) == ARG


def test_host_allreduce_validation(L):
    # every call fails its checks before any copy, so the fake host and
    # device addresses are never touched
    two = arr(A, A)
    ws = L.lpcoll_host_workspace_bytes(2, 1024, 0, 128, 1, 1, 3)
    assert ws > 0 and L.lpcoll_host_workspace_bytes(2, 1024, 0, 128, 1, 1, 0) == 0
    assert L.lpcoll_host_workspace_bytes(2, 1024, 0, 128, 1, 1, 2) < ws
    f = L.lpcoll_host_allreduce
    assert f(two, two, two, 2, 10, 4, 128, 1024, 3, A, ws, None, None, None) == ARG   # dtype
    assert f(two, two, two, 0, 10, 0, 128, 1024, 3, A, ws, None, None, None) == ARG   # N
    assert f(two, two, two, 2, 10, 0, 128, 1024, 9, A, ws, None, None, None) == ARG   # slots
    assert f(two, two, two, 2, 10, 0, 64, 1024, 3, A, ws, None, None, None) == UNSUP  # block
    assert f(two, two, two, 2, 10, 0, 128, 1000, 3, A, ws, None, None, None) == ARG   # chunk
    assert f(two, two, two, 2, 0, 0, 128, 1024, 3, A, ws, None, None, None) == OK     # n == 0
    assert f(two, None, None, 2, 10, 0, 128, 1024, 3, A, ws, None, None, None) == ARG  # no output
    assert f(two, two, None, 2, 10, 0, 128, 1024, 3, None, ws, None, None, None) == ARG
    assert f(arr(A, None), two, None, 2, 10, 0, 128, 1024, 3, A, ws, None, None, None) == RANK
    assert f(two, two, arr(None, A), 2, 10, 0, 128, 1024, 3, A, ws, None, None, None) == RANK
    assert f(two, two, two, 2, 10, 0, 128, 1024, 3, A + 16, ws, None, None, None) == ALIGN
    assert f(two, two, two, 2, 10, 0, 128, 1024, 3, A, ws - 1, None, None, None) == ARG
