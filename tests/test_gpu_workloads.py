"""The five reference workloads at full size, in the launch configuration the
benchmark times (``runner.RankBuffers``), checked against the oracle.

The small LP flat case (N=2, 1 Mi FP32 per rank) is compared in full. The
large cases are compared on sampled 128-element blocks (the first and last
blocks, the ragged tail if any, and random blocks): blocks are independent in
every stage, so the oracle run on the gathered blocks of every rank computes
exactly those blocks of the full result. On the whole message the test checks
properties that hold at any size: all N outputs identical, every scale finite
and non-negative. With LPCOLL_FULL_ORACLE=1 every workload, the collectives
and the variants are also compared with the oracle run on the whole message,
element by element (about a minute of oracle time on one core).
"""
import os

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


@pytest.mark.skipif(os.environ.get("LPCOLL_FULL_ORACLE") != "1",
                    reason="whole-message oracle comparison: set LPCOLL_FULL_ORACLE=1 "
                           "(about a minute of CPU oracle time)")
@pytest.mark.parametrize("w", W.WORKLOADS, ids=[w.name for w in W.WORKLOADS])
def test_workload_full_oracle(oracle, w):
    """Every element of every output, wire payload and shard payload of the
    full-size workload against the oracle run on the whole message."""
    ins = W.draw_all(w)
    bufs = runner.RankBuffers(w.nranks, w.n, w.dtype, w.block, separate_tree_out=True)
    bufs.load(ins)
    stream = torch.cuda.current_stream().cuda_stream
    for algo in w.algos:
        bufs.run(algo, stream)
        torch.cuda.synchronize()
        if algo == "tree":
            o_out, o_wc, o_ws, o_sc, o_ss = oracle.tree(ins, block=w.block)
        else:
            o_out, o_wc, o_ws = oracle.flat(ins, block=w.block)
        outs = bufs.tree_outs if algo == "tree" else bufs.outs
        for r in range(w.nranks):
            _check(from_dev(outs[r]), o_out[r], "%s out[%d]" % (algo, r))
            if w.block:
                _check(from_dev(bufs.wire_codes[r]), o_wc[r], "%s wire_codes[%d]" % (algo, r))
                _check(from_dev(bufs.wire_scales[r]), o_ws[r], "%s wire_scales[%d]" % (algo, r))
        if w.block and algo == "tree":
            _check(from_dev(bufs.shard_codes), o_sc, "shard_codes")
            _check(from_dev(bufs.shard_scales), o_ss, "shard_scales")
        del o_out
    del bufs
    torch.cuda.empty_cache()


@pytest.mark.skipif(os.environ.get("LPCOLL_FULL_ORACLE") != "1",
                    reason="whole-message oracle comparison: set LPCOLL_FULL_ORACLE=1")
@pytest.mark.parametrize("kind", ["reduce_scatter", "all_gather", "all_to_all"])
def test_collectives_full_oracle(oracle, kind):
    """The collectives in the benchmark's configuration (8 ranks, 16 MiB BF16
    per rank, low precision): every element of every output, wire code and
    scale against the oracle run on the whole message."""
    import precision_collective_reduction_gb300 as pcr
    w = W.LP_FLAT_N8_16MB_BF16
    N, n = w.nranks, w.n
    ins = W.draw_all(w)
    dins = [torch.from_numpy(x).view(torch.int16).view(torch.bfloat16).cuda() for x in ins]
    nb = pcr.nblocks(n)
    wc = [torch.empty(n, dtype=torch.uint8, device="cuda") for _ in range(N)]
    ws = [torch.empty(N * nb, dtype=torch.float32, device="cuda") for _ in range(N)]
    if kind == "reduce_scatter":
        per = pcr.shard_len(n, N)
        outs = [torch.empty(max(1, min(per, n - r * per)), dtype=torch.bfloat16, device="cuda")
                for r in range(N)]
        pcr.reduce_scatter_sim(dins, outs, wire_codes=wc, wire_scales=[t[:nb] for t in ws])
        o_out, o_wc, o_ws = oracle.reduce_scatter(ins)
        ncode, nscale = n, nb
    elif kind == "all_gather":
        m = n // N
        outs = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
        pcr.all_gather_sim([t[:m] for t in dins], outs, wire_codes=[t[:m] for t in wc],
                           wire_scales=[t[:pcr.nblocks(m)] for t in ws])
        o_out, o_wc, o_ws = oracle.all_gather([x[:m] for x in ins])
        ncode, nscale = m, pcr.nblocks(m)
    else:
        c = n // N
        outs = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
        pcr.all_to_all_sim(dins, outs, wire_codes=wc, wire_scales=ws)
        o_out, o_wc, o_ws = oracle.all_to_all(ins)
        ncode, nscale = n, N * pcr.nblocks(c)
    torch.cuda.synchronize()
    for r in range(N):
        _check(from_dev(outs[r])[:o_out[r].size], o_out[r], "%s out[%d]" % (kind, r))
        _check(from_dev(wc[r][:ncode]), o_wc[r][:ncode], "%s wire_codes[%d]" % (kind, r))
        _check(from_dev(ws[r][:nscale]), o_ws[r][:nscale], "%s wire_scales[%d]" % (kind, r))
    del dins, wc, ws, outs
    torch.cuda.empty_cache()


def test_collectives_at_benchmark_size(oracle):
    """ReduceScatter, AllGather and AlltoAll in the benchmark's configuration
    (8 ranks, 16 MiB BF16 per rank, low precision), checked on sampled
    128-element blocks against the oracle (blocks are independent)."""
    import precision_collective_reduction_gb300 as pcr
    w = W.LP_FLAT_N8_16MB_BF16
    N, n = w.nranks, w.n
    ins = W.draw_all(w)
    dins = [torch.from_numpy(x).view(torch.int16).view(torch.bfloat16).cuda() for x in ins]
    nb = pcr.nblocks(n)
    wc = [torch.empty(n, dtype=torch.uint8, device="cuda") for _ in range(N)]
    ws = [torch.empty(nb, dtype=torch.float32, device="cuda") for _ in range(N)]
    g = np.random.default_rng(77)

    # reduce-scatter: shard r of the flat allreduce, on sampled blocks
    per = pcr.shard_len(n, N)
    rs = [torch.empty(max(1, min(per, n - r * per)), dtype=torch.bfloat16, device="cuda")
          for r in range(N)]
    pcr.reduce_scatter_sim(dins, rs, wire_codes=wc, wire_scales=ws)
    torch.cuda.synchronize()
    blocks = sorted(set(g.choice(nb, 64, replace=False).tolist()) | {0, nb - 1})
    sub = [_gather_blocks(x, blocks, n) for x in ins]
    want = oracle.flat(sub)[0][0]
    got = []
    for b in blocks:
        owner, off = divmod(b * 128, per)
        got.append(from_dev(rs[owner][off:off + 128]))
    _check(np.concatenate(got), want, "reduce_scatter sampled blocks")

    # all-gather of the first m elements of every rank
    m = n // N
    outs = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    pcr.all_gather_sim([t[:m] for t in dins], outs, wire_codes=wc, wire_scales=ws)
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    mb = m // 128
    for r in range(N):
        for b in g.choice(mb, 8, replace=False).tolist() + [mb - 1]:
            blk = ins[r][b * 128:(b + 1) * 128]
            c, s = oracle.quantize(blk)
            want = oracle.dequantize(c, s, dtype=np.uint16)
            at = r * m + b * 128
            _check(from_dev(outs[-1][at:at + 128]), want, "all_gather r=%d b=%d" % (r, b))

    # all-to-all with chunks of c = n / N
    c = n // N
    pcr.all_to_all_sim(dins, outs, wire_codes=wc, wire_scales=ws)
    torch.cuda.synchronize()
    cb = c // 128
    for r in range(N):
        for j in range(N):
            for b in g.choice(cb, 3, replace=False).tolist() + [cb - 1]:
                blk = ins[r][j * c + b * 128:j * c + (b + 1) * 128]
                cc, ss = oracle.quantize(blk)
                want = oracle.dequantize(cc, ss, dtype=np.uint16)
                at = r * c + b * 128
                _check(from_dev(outs[j][at:at + 128]), want,
                       "all_to_all r=%d j=%d b=%d" % (r, j, b))
    del dins, wc, ws, rs, outs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("block", [32, 64, 128, 256])
def test_variants_at_benchmark_size(oracle, fmt, block):
    """The format / block-size ablation's configuration (8 ranks x 4 Mi FP32,
    gradient recipe): quantize and reduce on the GPU, sampled blocks of the
    payload and of the reduced result against the oracle."""
    import precision_collective_reduction_gb300 as pcr
    w = W.LP_GRAD_N8_256MB_F32
    n = 1 << 22
    ins = W.draw_all(w, n)
    dins = [torch.from_numpy(x).cuda() for x in ins]
    codes = [torch.empty(n, dtype=torch.uint8, device="cuda") for _ in range(w.nranks)]
    scales = [torch.empty(pcr.nblocks(n, block), dtype=torch.float32, device="cuda")
              for _ in range(w.nranks)]
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    for r in range(w.nranks):
        pcr.lp_quantize_fmt(dins[r], codes[r], scales[r], block, fmt)
    pcr.lp_reduce_fmt(codes, scales, out, block, fmt)
    torch.cuda.synchronize()
    nb = n // block
    g = np.random.default_rng(block + fmt)
    for b in g.choice(nb, 32, replace=False).tolist() + [0, nb - 1]:
        lo, hi = b * block, (b + 1) * block
        pays = [oracle.quantize_fmt(x[lo:hi], block, fmt) for x in ins]
        for r in (0, w.nranks - 1):
            _check(from_dev(codes[r][lo:hi]), pays[r][0], "codes r=%d b=%d" % (r, b))
            _check(from_dev(scales[r][b:b + 1]), pays[r][1], "scale r=%d b=%d" % (r, b))
        want = oracle.reduce_fmt([c for c, _ in pays], [s for _, s in pays], block, fmt)
        _check(from_dev(out[lo:hi]), want, "reduced b=%d" % b)
    del dins, codes, scales, out
    torch.cuda.empty_cache()


@pytest.mark.skipif(os.environ.get("LPCOLL_FULL_ORACLE") != "1",
                    reason="whole-message oracle comparison: set LPCOLL_FULL_ORACLE=1")
@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("block", [32, 64, 128, 256])
def test_variants_full_oracle(oracle, fmt, block):
    """The format / block-size ablation's configuration (8 ranks x 4 Mi FP32):
    every code and scale of every rank's payload and every element of the
    reduced result against the oracle."""
    import precision_collective_reduction_gb300 as pcr
    w = W.LP_GRAD_N8_256MB_F32
    n = 1 << 22
    ins = W.draw_all(w, n)
    dins = [torch.from_numpy(x).cuda() for x in ins]
    codes = [torch.empty(n, dtype=torch.uint8, device="cuda") for _ in range(w.nranks)]
    scales = [torch.empty(pcr.nblocks(n, block), dtype=torch.float32, device="cuda")
              for _ in range(w.nranks)]
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    for r in range(w.nranks):
        pcr.lp_quantize_fmt(dins[r], codes[r], scales[r], block, fmt)
    pcr.lp_reduce_fmt(codes, scales, out, block, fmt)
    torch.cuda.synchronize()
    pays = [oracle.quantize_fmt(x, block, fmt) for x in ins]
    for r in range(w.nranks):
        _check(from_dev(codes[r]), pays[r][0], "codes[%d]" % r)
        _check(from_dev(scales[r]), pays[r][1], "scales[%d]" % r)
    want = oracle.reduce_fmt([c for c, _ in pays], [s for _, s in pays], block, fmt)
    _check(from_dev(out), want, "reduced")
    del dins, codes, scales, out
    torch.cuda.empty_cache()
