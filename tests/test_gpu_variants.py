"""Format / block-size variants (E4M3 and E5M2; blocks of 32, 64, 128, 256)
of quantize, dequantize and reduce on the GPU against the CPU oracle, bit for
bit, through the C ABI."""
import numpy as np
import pytest
import torch

import precision_collective_reduction_gb300 as pcr
from precision_collective_reduction_gb300 import workloads as W
from gpu_util import Guarded, first_mismatch, from_dev, same_bits, to_dev

pytestmark = pytest.mark.gpu

TDT = {W.F32: torch.float32, W.BF16: torch.bfloat16}
FMTS = [pcr.E4M3, pcr.E5M2]


def _same(got, want, what):
    assert same_bits(got, want), "%s: first mismatch, count = %s" % (
        what, first_mismatch(got, want))


def _quantize(x, block, fmt):
    n = x.size
    c = Guarded(n, torch.uint8)
    s = Guarded(pcr.nblocks(n, block), torch.float32)
    pcr.lp_quantize_fmt(to_dev(x), c.t, s.t, block, fmt)
    torch.cuda.synchronize()
    assert c.intact() and s.intact()
    return from_dev(c.t), from_dev(s.t)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("block", pcr.VARIANT_BLOCKS)
@pytest.mark.parametrize("dt", [W.F32, W.BF16])
@pytest.mark.parametrize("n", [1, 100, 257, 128 * 40 + 5, 256 * 33])
def test_quantize_dequantize(oracle, fmt, block, dt, n):
    x = W.random_inputs(1, n, dt, 12000 + block + n + 7 * fmt, scale_spread=5.0)[0]
    codes, scales = _quantize(x, block, fmt)
    oc, os_ = oracle.quantize_fmt(x, block, fmt)
    _same(codes, oc, "codes")
    _same(scales, os_, "scales")
    out = Guarded(n, TDT[dt])
    pcr.lp_dequantize_fmt(to_dev(oc), to_dev(os_), out.t, block, fmt)
    torch.cuda.synchronize()
    assert out.intact()
    want = oracle.dequantize_fmt(oc, os_, block, fmt,
                                 dtype=np.float32 if dt == W.F32 else np.uint16)
    _same(from_dev(out.t), want, "dequantized")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("block", pcr.VARIANT_BLOCKS)
@pytest.mark.parametrize("dt", [W.F32, W.BF16])
@pytest.mark.parametrize("N", [1, 3, 5, 8, 16])
def test_reduce(oracle, fmt, block, dt, N):
    n = 128 * 30 + 17
    ins = W.random_inputs(N, n, dt, 13000 + block + N + 5 * fmt, scale_spread=3.0)
    pays = [oracle.quantize_fmt(x, block, fmt) for x in ins]
    out = Guarded(n, TDT[dt])
    pcr.lp_reduce_fmt([to_dev(c) for c, _ in pays], [to_dev(s) for _, s in pays], out.t,
                      block, fmt)
    torch.cuda.synchronize()
    assert out.intact()
    want = oracle.reduce_fmt([c for c, _ in pays], [s for _, s in pays], block, fmt,
                             dtype=np.float32 if dt == W.F32 else np.uint16)
    _same(from_dev(out.t), want, "reduced")


def test_e4m3_128_variant_equals_main_path():
    n = 128 * 77 + 3
    for dt in (W.F32, W.BF16):
        x = to_dev(W.random_inputs(1, n, dt, 3, scale_spread=3.0)[0])
        c1 = torch.empty(n, dtype=torch.uint8, device="cuda")
        s1 = torch.empty(pcr.nblocks(n), dtype=torch.float32, device="cuda")
        c2, s2 = torch.empty_like(c1), torch.empty_like(s1)
        pcr.lp_quantize(x, c1, s1)
        pcr.lp_quantize_fmt(x, c2, s2, 128, pcr.E4M3)
        torch.cuda.synchronize()
        assert torch.equal(c1, c2) and torch.equal(s1.view(torch.int32), s2.view(torch.int32))


def test_all_e5m2_codes(oracle):
    # a block holding 57344 has scale 1 and multiplier 1: its other elements
    # reach the E5M2 encoder unchanged (every finite code, midpoints, and the
    # floats around them)
    table = oracle.e5m2_decode_all()
    fin = np.array([table[c] for c in range(256) if np.isfinite(table[c])], dtype=np.float32)
    pos = np.array([table[c] for c in range(0x7C)], dtype=np.float64)
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    body = np.concatenate([fin, mids, np.nextafter(mids, np.float32(np.inf)),
                           np.nextafter(mids, np.float32(0)), -mids, [np.nan]])
    blocks = []
    for i in range(0, body.size, 127):
        blk = np.zeros(128, dtype=np.float32)
        blk[0] = 57344.0
        chunk = body[i:i + 127]
        blk[1:1 + chunk.size] = chunk
        blocks.append(blk)
    x = np.concatenate(blocks).astype(np.float32)
    codes, scales = _quantize(x, 128, pcr.E5M2)
    oc, os_ = oracle.quantize_fmt(x, 128, pcr.E5M2)
    assert np.all(os_ == 1.0)
    _same(scales, os_, "scales")
    _same(codes, oc, "codes")
