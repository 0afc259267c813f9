"""Seeded random configurations of every entry point against the oracle, bit
for bit: operation, rank count, length (including ragged and tiny), dtype,
exact or low precision, FP8 format and block size, in place or not.

LPCOLL_FUZZ_CONFIGS sets how many configurations run (default 300)."""
import os

import numpy as np
import pytest
import torch

import precision_collective_reduction_gb300 as pcr
from precision_collective_reduction_gb300 import workloads as W
from gpu_util import from_dev, same_bits, to_dev

pytestmark = pytest.mark.gpu

TDT = {W.F32: torch.float32, W.BF16: torch.bfloat16}
NP = {W.F32: np.float32, W.BF16: np.uint16}
OPS = ["flat", "tree", "rs", "ag", "a2a", "quant", "reduce", "fmt"]


def _configs(count=int(os.environ.get("LPCOLL_FUZZ_CONFIGS", "300")), seed=2026):
    g = np.random.default_rng(seed)
    for i in range(count):
        op = OPS[i % len(OPS)]
        N = int(g.integers(1, 17))
        n = int(g.choice([g.integers(1, 300), g.integers(300, 5000), g.integers(5000, 40000)]))
        dt = int(g.integers(0, 2))
        block = int(g.choice([0, 128])) if op in ("flat", "tree", "rs", "ag", "a2a") else 128
        spread = float(g.uniform(0, 6))
        yield i, op, N, n, dt, block, spread, bool(g.integers(0, 2))


def _wires(N, ncodes, nscales):
    return ([torch.empty(ncodes, dtype=torch.uint8, device="cuda") for _ in range(N)],
            [torch.empty(nscales, dtype=torch.float32, device="cuda") for _ in range(N)])


@pytest.mark.parametrize("cfg", list(_configs()), ids=lambda c: "%d-%s" % (c[0], c[1]))
def test_random_config(oracle, cfg):
    i, op, N, n, dt, block, spread, flag = cfg
    seed = 20000 + i
    if op in ("flat", "tree"):
        ins = W.random_inputs(N, n, dt, seed, scale_spread=spread)
        xd = [to_dev(x) for x in ins]
        outs = xd if flag else [torch.empty_like(t) for t in xd]   # flag: in place
        wc, ws = _wires(N, n, pcr.nblocks(n))
        sc = torch.empty(n, dtype=torch.uint8, device="cuda")
        ss = torch.empty(pcr.nblocks(n), dtype=torch.float32, device="cuda")
        if op == "flat":
            pcr.dda_flat_sim(xd, outs, block=block, wire_codes=wc, wire_scales=ws)
            want = oracle.flat(ins, block=block)[0]
        else:
            pcr.dda_tree_sim(xd, outs, block=block, wire_codes=wc, wire_scales=ws,
                             shard_codes=sc, shard_scales=ss)
            want = oracle.tree(ins, block=block)[0]
        torch.cuda.synchronize()
        for r in range(N):
            assert same_bits(from_dev(outs[r]), want[r]), r
    elif op == "rs":
        ins = W.random_inputs(N, n, dt, seed, scale_spread=spread)
        per = pcr.shard_len(n, N, block)
        lens = [max(0, min(per, n - r * per)) for r in range(N)]
        outs = [torch.empty(k, dtype=TDT[dt], device="cuda") if k else None for k in lens]
        wc, ws = _wires(N, n, pcr.nblocks(n))
        pcr.reduce_scatter_sim([to_dev(x) for x in ins], outs, block=block, wire_codes=wc,
                               wire_scales=ws)
        torch.cuda.synchronize()
        want = oracle.reduce_scatter(ins, block=block)[0]
        for r in range(N):
            if lens[r]:
                assert same_bits(from_dev(outs[r]), want[r]), r
    elif op == "ag":
        m = max(1, n // N)
        ins = W.random_inputs(N, m, dt, seed, scale_spread=spread)
        outs = [torch.empty(N * m, dtype=TDT[dt], device="cuda") for _ in range(N)]
        wc, ws = _wires(N, m, pcr.nblocks(m))
        pcr.all_gather_sim([to_dev(x) for x in ins], outs, block=block, wire_codes=wc,
                           wire_scales=ws)
        torch.cuda.synchronize()
        want = oracle.all_gather(ins, block=block)[0]
        for r in range(N):
            assert same_bits(from_dev(outs[r]), want[r]), r
    elif op == "a2a":
        c = max(1, n // N)
        ins = W.random_inputs(N, N * c, dt, seed, scale_spread=spread)
        outs = [torch.empty(N * c, dtype=TDT[dt], device="cuda") for _ in range(N)]
        wc, ws = _wires(N, N * c, N * pcr.nblocks(c))
        pcr.all_to_all_sim([to_dev(x) for x in ins], outs, block=block, wire_codes=wc,
                           wire_scales=ws)
        torch.cuda.synchronize()
        want = oracle.all_to_all(ins, block=block)[0]
        for r in range(N):
            assert same_bits(from_dev(outs[r]), want[r]), r
    elif op == "quant":
        x = W.random_inputs(1, n, dt, seed, scale_spread=spread)[0]
        c = torch.empty(n, dtype=torch.uint8, device="cuda")
        s = torch.empty(pcr.nblocks(n), dtype=torch.float32, device="cuda")
        pcr.lp_quantize(to_dev(x), c, s)
        out = torch.empty(n, dtype=TDT[dt], device="cuda")
        pcr.lp_dequantize(c, s, out)
        torch.cuda.synchronize()
        oc, os_ = oracle.quantize(x)
        assert same_bits(from_dev(c), oc) and same_bits(from_dev(s), os_)
        assert same_bits(from_dev(out), oracle.dequantize(oc, os_, dtype=NP[dt]))
    elif op == "reduce":
        ins = W.random_inputs(N, n, dt, seed, scale_spread=spread)
        pays = [oracle.quantize(x) for x in ins]
        out = torch.empty(n, dtype=TDT[dt], device="cuda")
        pcr.lp_reduce([to_dev(c) for c, _ in pays], [to_dev(s) for _, s in pays], out)
        torch.cuda.synchronize()
        want = oracle.reduce([c for c, _ in pays], [s for _, s in pays], dtype=NP[dt])
        assert same_bits(from_dev(out), want)
    else:  # format / block-size variant of quantize + reduce
        fmt = int(flag)
        vb = pcr.VARIANT_BLOCKS[i % 4]
        ins = W.random_inputs(min(N, 4), n, dt, seed, scale_spread=spread)
        codes, scales = [], []
        for x in ins:
            c = torch.empty(n, dtype=torch.uint8, device="cuda")
            s = torch.empty(pcr.nblocks(n, vb), dtype=torch.float32, device="cuda")
            pcr.lp_quantize_fmt(to_dev(x), c, s, vb, fmt)
            codes.append(c)
            scales.append(s)
        out = torch.empty(n, dtype=TDT[dt], device="cuda")
        pcr.lp_reduce_fmt(codes, scales, out, vb, fmt)
        torch.cuda.synchronize()
        pays = [oracle.quantize_fmt(x, vb, fmt) for x in ins]
        for c, s, (oc, os_) in zip(codes, scales, pays):
            assert same_bits(from_dev(c), oc) and same_bits(from_dev(s), os_)
        want = oracle.reduce_fmt([c for c, _ in pays], [s for _, s in pays], vb, fmt,
                                 dtype=NP[dt])
        assert same_bits(from_dev(out), want)
