"""Messages longer than 2^31 elements: every index and byte offset of the
kernels is 64-bit. Two ranks of 2^31 + 200 FP32 elements (8.6 GB each, about
40 GB on the device with outputs and wires), LP flat and tree; sampled
128-element blocks at the start, across element 2^31 and at the ragged end
are checked against the oracle. The inputs are drawn on the GPU by PyTorch's
seeded generator (not by this library) and the sampled blocks are copied to
the host for the oracle."""
import pytest
import torch

import precision_collective_reduction_gb300 as pcr
from gpu_util import from_dev, same_bits

pytestmark = pytest.mark.gpu

N = 2
n = (1 << 31) + 200


def test_flat_and_tree_beyond_2_31_elements(oracle):
    free, _ = torch.cuda.mem_get_info()
    if free < 48 * (1 << 30):
        pytest.skip("needs about 40 GB of free device memory")
    g = torch.Generator(device="cuda").manual_seed(2024)
    ins = [torch.randn(n, device="cuda", generator=g) for _ in range(N)]
    outs = [torch.empty(n, device="cuda") for _ in range(N)]
    wc = [torch.empty(n, dtype=torch.uint8, device="cuda") for _ in range(N)]
    ws = [torch.empty(pcr.nblocks(n), device="cuda") for _ in range(N)]
    sc = torch.empty(n, dtype=torch.uint8, device="cuda")
    ss = torch.empty(pcr.nblocks(n), device="cuda")
    nb = pcr.nblocks(n)
    mid = (1 << 31) // 128
    # sorted and unique, so the ragged last block is also last in the sample
    # (blocks keep their boundaries when the oracle sees the gathered sample)
    blocks = sorted({0, 1, mid - 2, mid - 1, mid, mid + 1, nb - 2, nb - 1})
    idx = torch.cat([torch.arange(b * 128, min((b + 1) * 128, n), device="cuda")
                     for b in blocks])
    sub = [from_dev(t[idx]) for t in ins]
    for algo in ("flat", "tree"):
        if algo == "flat":
            pcr.dda_flat_sim(ins, outs, wire_codes=wc, wire_scales=ws)
            want, owc, ows = oracle.flat(sub)
        else:
            pcr.dda_tree_sim(ins, outs, wire_codes=wc, wire_scales=ws,
                             shard_codes=sc, shard_scales=ss)
            want, owc, ows, osc, oss = oracle.tree(sub)
        torch.cuda.synchronize()
        bidx = torch.tensor(blocks, device="cuda")
        for r in range(N):
            assert same_bits(from_dev(outs[r][idx]), want[r]), (algo, r)
            assert same_bits(from_dev(wc[r][idx]), owc[r]), (algo, r)
            assert same_bits(from_dev(ws[r][bidx]), ows[r]), (algo, r)
        if algo == "tree":
            assert same_bits(from_dev(sc[idx]), osc)
            assert same_bits(from_dev(ss[bidx]), oss)
    del ins, outs, wc, ws, sc, ss
    torch.cuda.empty_cache()
