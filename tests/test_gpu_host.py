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


@pytest.mark.parametrize("fail_step", [3, 10, 12, 25, 40, 61])
def test_error_return_waits_for_every_stream(fail_step):
    # A failure injected on the host at one enqueue step (no CUDA call
    # fails) must not let the call return while work it queued before the
    # failure still runs: on return, all three streams are idle, so the
    # caller may free its host buffers and the workspace at once.
    # 8 ranks x 16 Mi FP32 in chunks of 4 Mi: the copies of one chunk take
    # milliseconds, far longer than the host needs to reach the return.
    # Enqueue steps per chunk (flat only): 8 copies in, event record, wait,
    # launch, record, wait, 8 copies out, record (+1 wait once a slot is
    # reused), so the steps above land in the copy-in, launch, copy-out and
    # second-chunk phases.
    from precision_collective_reduction_gb300 import _binding as B
    N, n = 8, 16 << 20
    h = HostAllreduce(N, n, W.F32, 128, algos=("flat",), chunk=4 << 20, slots=2)
    hin = [torch.full((n,), float(r), dtype=torch.float32).pin_memory() for r in range(N)]
    hout = {"flat": [torch.empty(n, dtype=torch.float32).pin_memory() for _ in range(N)]}
    torch.cuda.synchronize()
    B.lib().lpcoll_debug_fail_host_enqueue(fail_step)
    with pytest.raises(B.LpcollError) as err:
        h.run(hin, hout)
    assert err.value.status == 5  # LPCOLL_ERR_CUDA
    idle = [s.query() for s in h.streams]
    assert idle == [True, True, True], idle
    assert B.lib().lpcoll_last_cuda_error() == 1  # cudaErrorInvalidValue, injected
    # the hook fired once: the next call runs normally and is correct
    h.run(hin, hout)
    want = float(N * (N - 1) // 2)
    assert all(bool((t == want).all()) for t in hout["flat"])
