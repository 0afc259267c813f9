"""lpcoll_host_allreduce (host-resident buffers, chunked and overlapped,
through HostAllreduce and directly) gives the same bits as one launch over
the whole message, and as the oracle."""
import numpy as np
import pytest
import torch

from precision_collective_reduction_gb300 import runner, workloads as W
from precision_collective_reduction_gb300.host import HostAllreduce
from gpu_util import from_dev, same_bits

pytestmark = pytest.mark.gpu

TDT = {W.F32: torch.float32, W.BF16: torch.bfloat16}


def _host(a, dt):
    t = torch.from_numpy(a)
    if dt == W.BF16:
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.pin_memory()


def _np(t, dt):
    return t.view(torch.int16).numpy().view(np.uint16) if dt == W.BF16 else t.numpy()


@pytest.mark.parametrize("dt", [W.F32, W.BF16])
@pytest.mark.parametrize("block", [128, 0])
@pytest.mark.parametrize("chunk,slots", [(128 * 64, 2), (128 * 100, 3), (1 << 22, 3)])
def test_chunked_equals_single_launch(dt, block, chunk, slots):
    N, n = 4, 128 * 1000 + 37
    ins = W.random_inputs(N, n, dt, 77 + chunk % 7, scale_spread=3.0)
    ref = runner.RankBuffers(N, n, dt, block, separate_tree_out=True)
    ref.load(ins)
    s = torch.cuda.current_stream().cuda_stream
    ref.flat(s)
    ref.tree(s)
    torch.cuda.synchronize()
    h = HostAllreduce(N, n, dt, block, algos=("flat", "tree"), chunk=chunk, slots=slots)
    hin = [_host(x, dt) for x in ins]
    hout = {a: [torch.empty(n, dtype=TDT[dt]).pin_memory() for _ in range(N)]
            for a in ("flat", "tree")}
    for _ in range(2):  # a second run reuses the slots
        for a in hout:
            for t in hout[a]:
                t.fill_(0)
        h.run(hin, hout)
        for r in range(N):
            assert same_bits(_np(hout["flat"][r], dt), from_dev(ref.outs[r]))
            assert same_bits(_np(hout["tree"][r], dt), from_dev(ref.tree_outs[r]))


def test_matches_oracle(oracle):
    N, n = 3, 128 * 300 + 5
    ins = W.random_inputs(N, n, W.F32, 5, scale_spread=2.0)
    h = HostAllreduce(N, n, W.F32, 128, algos=("tree",), chunk=128 * 32)
    hout = {"tree": [torch.empty(n, dtype=torch.float32).pin_memory() for _ in range(N)]}
    h.run([_host(x, W.F32) for x in ins], hout)
    want = oracle.tree(ins)[0]
    for r in range(N):
        assert same_bits(hout["tree"][r].numpy(), want[r])


def test_direct_call_pageable_and_default_streams(oracle):
    # pageable host memory and one stream for all three roles: no overlap,
    # same results
    import precision_collective_reduction_gb300 as pcr
    N, n = 3, 128 * 77 + 9
    ins = W.random_inputs(N, n, W.BF16, 8, scale_spread=2.0)
    hin = [torch.from_numpy(x).view(torch.int16).view(torch.bfloat16) for x in ins]
    hflat = [torch.empty(n, dtype=torch.bfloat16) for _ in range(N)]
    pcr.lpcoll_host_allreduce(hin, host_out_flat=hflat, block=128, chunk=128 * 10, slots=2)
    want = oracle.flat(ins)[0]
    for r in range(N):
        assert same_bits(_np(hflat[r], W.BF16), want[r])
