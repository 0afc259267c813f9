"""ReduceScatter, AllGather and AlltoAll on the GPU against the CPU oracle,
bit for bit, through the C ABI: both dtypes, exact and low precision, rank
counts 1..16, ragged sizes and lengths that are not a multiple of 16 bytes
(element-wise path). Output buffers carry guard bands."""
import pytest
import torch

import precision_collective_reduction_gb300 as pcr
from precision_collective_reduction_gb300 import workloads as W
from gpu_util import Guarded, first_mismatch, from_dev, same_bits, to_dev

pytestmark = pytest.mark.gpu

TDT = {W.F32: torch.float32, W.BF16: torch.bfloat16}


def _same(got, want, what):
    assert same_bits(got, want), "%s: first mismatch, count = %s" % (
        what, first_mismatch(got, want))


def _wires(N, ncodes, nscales, block):
    if not block:
        return None, None
    wc = [Guarded(ncodes, torch.uint8) for _ in range(N)]
    ws = [Guarded(nscales, torch.float32) for _ in range(N)]
    return wc, ws


def _check_guards(*groups):
    for g in groups:
        for x in (g or []):
            assert x.intact(), "write past the end of a buffer"


@pytest.mark.parametrize("dt", [W.F32, W.BF16])
@pytest.mark.parametrize("block", [128, 0])
@pytest.mark.parametrize("N", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("n", [1, 127, 129, 1000, 128 * 300 + 5])
def test_reduce_scatter(oracle, dt, block, N, n):
    ins = W.random_inputs(N, n, dt, 9000 + 7 * N + n, scale_spread=3.0)
    per = pcr.shard_len(n, N, block)
    lens = [max(0, min(per, n - r * per)) for r in range(N)]
    outs = [Guarded(k, TDT[dt]) if k else None for k in lens]
    wc, ws = _wires(N, n, pcr.nblocks(n), block)
    kw = dict(wire_codes=[g.t for g in wc], wire_scales=[g.t for g in ws]) if block else {}
    pcr.reduce_scatter_sim([to_dev(x) for x in ins], [o.t if o else None for o in outs],
                           block=block, **kw)
    torch.cuda.synchronize()
    _check_guards([o for o in outs if o], wc, ws)
    want, owc, ows = oracle.reduce_scatter(ins, block=block)
    for r in range(N):
        if lens[r]:
            _same(from_dev(outs[r].t), want[r], "out[%d]" % r)
        if block:
            _same(from_dev(wc[r].t), owc[r], "wire_codes[%d]" % r)
            _same(from_dev(ws[r].t), ows[r], "wire_scales[%d]" % r)


@pytest.mark.parametrize("dt", [W.F32, W.BF16])
@pytest.mark.parametrize("block", [128, 0])
@pytest.mark.parametrize("N", [1, 3, 8, 16])
@pytest.mark.parametrize("m", [1, 3, 77, 128, 200, 1000, 4096 + 77, 32 * 8 * 20, 3 * 1024 + 264])
def test_all_gather(oracle, dt, block, N, m):
    ins = W.random_inputs(N, m, dt, 9500 + 11 * N + m, scale_spread=3.0)
    outs = [Guarded(N * m, TDT[dt]) for _ in range(N)]
    wc, ws = _wires(N, m, pcr.nblocks(m), block)
    kw = dict(wire_codes=[g.t for g in wc], wire_scales=[g.t for g in ws]) if block else {}
    pcr.all_gather_sim([to_dev(x) for x in ins], [o.t for o in outs], block=block, **kw)
    torch.cuda.synchronize()
    _check_guards(outs, wc, ws)
    want, owc, ows = oracle.all_gather(ins, block=block)
    for r in range(N):
        _same(from_dev(outs[r].t), want[r], "out[%d]" % r)
        if block:
            _same(from_dev(wc[r].t), owc[r], "wire_codes[%d]" % r)
            _same(from_dev(ws[r].t), ows[r], "wire_scales[%d]" % r)


@pytest.mark.parametrize("dt", [W.F32, W.BF16])
@pytest.mark.parametrize("block", [128, 0])
@pytest.mark.parametrize("N", [1, 2, 5, 8])
@pytest.mark.parametrize("c", [1, 3, 130, 200, 256, 1001, 32 * 8 * 9, 4096 + 8])
def test_all_to_all(oracle, dt, block, N, c):
    ins = W.random_inputs(N, N * c, dt, 9900 + 13 * N + c, scale_spread=3.0)
    outs = [Guarded(N * c, TDT[dt]) for _ in range(N)]
    wc, ws = _wires(N, N * c, N * pcr.nblocks(c), block)
    kw = dict(wire_codes=[g.t for g in wc], wire_scales=[g.t for g in ws]) if block else {}
    pcr.all_to_all_sim([to_dev(x) for x in ins], [o.t for o in outs], block=block, **kw)
    torch.cuda.synchronize()
    _check_guards(outs, wc, ws)
    want, owc, ows = oracle.all_to_all(ins, block=block)
    for r in range(N):
        _same(from_dev(outs[r].t), want[r], "out[%d]" % r)
        if block:
            _same(from_dev(wc[r].t), owc[r], "wire_codes[%d]" % r)
            _same(from_dev(ws[r].t), ows[r], "wire_scales[%d]" % r)


def test_reduce_scatter_is_a_slice_of_flat():
    # the LP reduce-scatter result is the owner's shard of the flat allreduce
    N, n = 8, 32 * 8192 + 640
    ins = [to_dev(x) for x in W.random_inputs(N, n, W.BF16, 31, scale_spread=2.0)]
    wc = [torch.empty(n, dtype=torch.uint8, device="cuda") for _ in range(N)]
    ws = [torch.empty(pcr.nblocks(n), dtype=torch.float32, device="cuda") for _ in range(N)]
    flat = [torch.empty_like(t) for t in ins]
    pcr.dda_flat_sim(ins, flat, wire_codes=wc, wire_scales=ws)
    per = pcr.shard_len(n, N)
    outs = [torch.empty(max(0, min(per, n - r * per)), dtype=torch.bfloat16, device="cuda")
            for r in range(N)]
    pcr.reduce_scatter_sim(ins, outs, wire_codes=wc, wire_scales=ws)
    torch.cuda.synchronize()
    for r in range(N):
        a = outs[r].view(torch.int16)
        b = flat[0][r * per:r * per + outs[r].numel()].view(torch.int16)
        assert torch.equal(a, b), r
