"""The five reference workloads at full size, in the launch configuration the
benchmark times (``runner.RankBuffers``), checked against the oracle.

The small LP flat case (N=2, 1 Mi FP32 per rank) is compared in full. The
large cases are compared on sampled 128-element blocks (the first and last
blocks, the ragged tail if any, and random blocks): blocks are independent in
every stage, so the oracle run on the gathered blocks of every rank computes
exactly those blocks of the full result. On the whole message the test checks
properties that hold at any size: all N outputs identical, every scale finite
and non-negative.
"""
import numpy as np
import pytest
import torch

from precision_collective_reduction_gb300 import runner, workloads as W
from gpu_util import first_mismatch, from_dev, same_bits

pytestmark = pytest.mark.gpu

SAMPLE_RANDOM_BLOCKS = 96


def _gather_blocks(arr, blocks, n, block=128):
    return np.concatenate([arr[b * block:min((b + 1) * block, n)] for b in blocks])


def _sample_blocks(n, seed):
    nb = (n + 127) // 128
    g = np.random.default_rng(seed)
    mid = g.choice(np.arange(8, max(nb - 8, 9)), size=min(SAMPLE_RANDOM_BLOCKS, max(nb - 16, 1)),
                   replace=False)
    full = sorted(set(range(min(8, nb))) | set(int(b) for b in mid) |
                  set(range(max(nb - 8, 0), nb)))
    return full  # the ragged tail block, if any, is last


def _check(got, want, what):
    assert same_bits(got, want), "%s: first mismatch, count = %s" % (
        what, first_mismatch(got, want))


@pytest.mark.parametrize("w", W.WORKLOADS, ids=[w.name for w in W.WORKLOADS])
def test_workload(oracle, w):
    ins = W.draw_all(w)
    bufs = runner.RankBuffers(w.nranks, w.n, w.dtype, w.block,
                              separate_tree_out=True)
    bufs.load(ins)
    stream = torch.cuda.current_stream().cuda_stream
    full_compare = w.nranks * w.n <= 4 << 20
    blocks = None if full_compare else _sample_blocks(w.n, w.seed)
    for algo in w.algos:
        bufs.run(algo, stream)
        torch.cuda.synchronize()
        outs = bufs.tree_outs if algo == "tree" else bufs.outs
        i0 = outs[0].view(torch.int16 if outs[0].element_size() == 2 else torch.int32)
        for o in outs[1:]:
            assert torch.equal(o.view(i0.dtype), i0), "outputs differ across ranks"
        if w.block:
            for s in bufs.wire_scales:
                assert bool(torch.all(torch.isfinite(s) & (s >= 0)).item())
        if full_compare:
            sub_in = ins
        else:
            sub_in = [_gather_blocks(x, blocks, w.n) for x in ins]
        if algo == "tree":
            o_out, o_wc, o_ws, o_sc, o_ss = oracle.tree(sub_in, block=w.block)
        else:
            o_out, o_wc, o_ws = oracle.flat(sub_in, block=w.block)
        if full_compare:
            pick = pick_s = from_dev
        else:
            eidx = torch.from_numpy(_gather_blocks(np.arange(w.n), blocks, w.n)).cuda()
            bidx = torch.tensor(blocks, device="cuda")
            pick = lambda t: from_dev(t[eidx])  # noqa: E731
            pick_s = lambda t: from_dev(t[bidx])  # noqa: E731
        for r in range(w.nranks):
            _check(pick(outs[r]), o_out[r], "%s out[%d]" % (algo, r))
            if w.block:
                _check(pick(bufs.wire_codes[r]), o_wc[r],
                       "%s wire_codes[%d]" % (algo, r))
                _check(pick_s(bufs.wire_scales[r]), o_ws[r],
                       "%s wire_scales[%d]" % (algo, r))
        if w.block and algo == "tree":
            _check(pick(bufs.shard_codes), o_sc, "shard_codes")
            _check(pick_s(bufs.shard_scales), o_ss, "shard_scales")
    del bufs
    torch.cuda.empty_cache()
