"""dda_flat_sim_noalloc, the allreduce entry point for callers that cannot
allocate device memory (plugins inside a framework that owns all device
memory, loops that must never enter cudaMalloc). Its wire payloads live in a
fixed array inside the library, so the caller passes only inputs and
outputs. It must give exactly what the CPU oracle gives, and what
dda_flat_sim gives with caller-provided wire buffers, call after call, since
every call reuses the same array.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from precision_collective_reduction_gb300 import _binding as B
from precision_collective_reduction_gb300 import build as lib_build
from precision_collective_reduction_gb300 import workloads as W

MAX_ELEMS = 64 * 1024 * 1024
A = 0x10000  # aligned fake device address, never dereferenced below


def _fn():
    lib_build.build()
    f = B.lib().dda_flat_sim_noalloc
    f.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p),
                  ctypes.c_int, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f


def test_rejects_messages_beyond_the_fixed_scratch():
    # every call here fails its argument checks before touching CUDA
    f = _fn()
    ptrs = B.ptr_array([A] * 16)
    assert f(ptrs, ptrs, 16, MAX_ELEMS // 16 + 1, 0, None) == 1     # LPCOLL_ERR_ARG
    assert f(ptrs, ptrs, 1, MAX_ELEMS + 1, 1, None) == 1
    assert f(ptrs, ptrs, 3, MAX_ELEMS // 3, 0, None) == 1           # 256-rounding
    assert f(ptrs, ptrs, 0, 10, 0, None) == 1
    assert f(ptrs, ptrs, 2, 10, 7, None) == 1
    assert f(ptrs, ptrs, 2, 0, 0, None) == 0                         # n == 0: no-op
    assert f(B.ptr_array([A, 0]), ptrs, 2, 10, 0, None) == 4        # LPCOLL_ERR_RANK
    assert f(B.ptr_array([A, A + 4]), ptrs, 2, 10, 0, None) == 2    # LPCOLL_ERR_ALIGN


SAMPLE_RANDOM_BLOCKS = 96


def _sample_blocks(n, seed):
    """The first and last 8 blocks (the ragged tail, if any, among them) and
    random blocks in between."""
    nb = (n + 127) // 128
    g = np.random.default_rng(seed)
    mid = g.choice(np.arange(8, max(nb - 8, 9)),
                   size=min(SAMPLE_RANDOM_BLOCKS, max(nb - 16, 1)), replace=False)
    return sorted(set(range(min(8, nb))) | set(int(b) for b in mid) |
                  set(range(max(nb - 8, 0), nb)))


def _gather(arr, blocks, n):
    return np.concatenate([arr[b * 128:min((b + 1) * 128, n)] for b in blocks])


def _host_bits(t):
    t = t.view(torch.int16) if t.dtype == torch.bfloat16 else t
    a = t.cpu().numpy()
    return a.view(np.uint16) if a.dtype == np.int16 else a


@pytest.mark.gpu
@pytest.mark.parametrize("dt,N,n", [(W.F32, 8, 128 * 1000 + 5), (W.BF16, 4, 32 * 8192),
                                    (W.BF16, 3, 777), (W.F32, 16, MAX_ELEMS // 16),
                                    (W.BF16, 8, MAX_ELEMS // 8)])
def test_matches_oracle_and_allocating_entry_point_twice(oracle, dt, N, n):
    # Two calls in a row with different inputs (the array keeps the first
    # call's payload when the second starts). Each call is checked against
    # the CPU oracle (every element of small messages; sampled 128-element
    # blocks of the large ones, which the oracle computes exactly, since
    # blocks are independent) and, every element, against dda_flat_sim
    # with caller-provided wire buffers. The last case is the documented
    # limit: 8 ranks x 8 Mi BF16, a 16 MiB message per rank.
    from precision_collective_reduction_gb300 import runner
    f = _fn()
    ref = runner.RankBuffers(N, n, dt, 128)
    outs = [torch.empty_like(t) for t in ref.ins]
    p_out = B.ptr_array([t.data_ptr() for t in outs])
    stream = torch.cuda.current_stream().cuda_stream
    full = N * n <= 4 << 20
    blocks = None if full else _sample_blocks(n, 7 + N)
    for call in range(2):
        ins = W.random_inputs(N, n, dt, 50 + 10 * call + N, scale_spread=3.0)
        ref.load(ins)
        ref.flat(stream)
        for t in outs:
            t.fill_(7)
        st = f(ref.a_in, p_out, N, n, dt, stream)
        assert st == 0, B.status_string(st)
        torch.cuda.synchronize()
        sub = ins if full else [_gather(x, blocks, n) for x in ins]
        want = oracle.flat(sub)[0]
        if not full:
            idx = torch.from_numpy(_gather(np.arange(n), blocks, n)).cuda()
        for r in range(N):
            got = _host_bits(outs[r] if full else outs[r][idx])
            assert np.array_equal(got.view(np.uint8), want[r].view(np.uint8)), \
                "call %d: rank %d output differs from the oracle" % (call, r)
            a = ref.outs[r].view(torch.uint8)
            b = outs[r].view(torch.uint8)
            assert torch.equal(a, b), "call %d: rank %d output differs from dda_flat_sim" % (
                call, r)
    del ref, outs
    torch.cuda.empty_cache()
