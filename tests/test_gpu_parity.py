"""CUDA path against the CPU oracle, element by element, through the C ABI.

Bit-exact for FP8 codes, FP32 scales and the fixed-order FP32 sums (and their
BF16 casts), for every entry point, both dtypes, rank counts 1..16, sizes
from one element to several hundred blocks with ragged tails, degenerate
blocks, in-place operation and CUDA-graph replay. Every output buffer carries
a guard band that must be left untouched.
"""
import numpy as np
import pytest
import torch

import precision_collective_reduction_gb300 as pcr
from precision_collective_reduction_gb300 import workloads as W
from gpu_util import Guarded, first_mismatch, from_dev, same_bits, to_dev

pytestmark = pytest.mark.gpu

F32, BF16 = W.F32, W.BF16
SIZES = [1, 3, 7, 127, 128, 129, 200, 255, 256, 257, 1000, 4096 + 77,
         128 * 300 + 5, 32 * 8 * 64]
TORCH_DT = {F32: torch.float32, BF16: torch.bfloat16}


def _np_dt(dt):
    return np.float32 if dt == F32 else np.uint16


def gpu_quantize(x):
    n = x.size
    xd = to_dev(x)
    c = Guarded(n, torch.uint8)
    s = Guarded(pcr.nblocks(n), torch.float32)
    pcr.lp_quantize(xd, c.t, s.t)
    torch.cuda.synchronize()
    assert c.intact() and s.intact()
    return from_dev(c.t), from_dev(s.t)


def gpu_allreduce(ins, algo, block=128, in_place=False):
    N = len(ins)
    n = ins[0].size
    dt = TORCH_DT[F32 if ins[0].dtype == np.float32 else BF16]
    xd = [to_dev(x) for x in ins]
    if in_place:
        outs = None
        out_t = xd
    else:
        outs = [Guarded(n, dt) for _ in range(N)]
        out_t = [o.t for o in outs]
    kw = {}
    wc = ws = sc = ss = None
    if block:
        wc = [Guarded(n, torch.uint8) for _ in range(N)]
        ws = [Guarded(pcr.nblocks(n), torch.float32) for _ in range(N)]
        kw = dict(wire_codes=[g.t for g in wc], wire_scales=[g.t for g in ws])
        if algo == "tree":
            sc = Guarded(n, torch.uint8)
            ss = Guarded(pcr.nblocks(n), torch.float32)
            kw.update(shard_codes=sc.t, shard_scales=ss.t)
    fn = pcr.dda_tree_sim if algo == "tree" else pcr.dda_flat_sim
    fn(xd, out_t, block=block, **kw)
    torch.cuda.synchronize()
    for g in (outs or []) + (wc or []) + (ws or []) + [x for x in (sc, ss) if x]:
        assert g.intact(), "write past the end of a buffer"
    res = {"out": [from_dev(t) for t in out_t]}
    if block:
        res["wc"] = [from_dev(g.t) for g in wc]
        res["ws"] = [from_dev(g.t) for g in ws]
        if algo == "tree":
            res["sc"] = from_dev(sc.t)
            res["ss"] = from_dev(ss.t)
    return res


def assert_same(got, want, what):
    assert same_bits(got, want), "%s differs: first index, count = %s" % (
        what, first_mismatch(got, want))


def check_against_oracle(oracle, ins, algo, block, res):
    if algo == "tree":
        outs, wc, ws, sc, ss = oracle.tree(ins, block=block)
    else:
        outs, wc, ws = oracle.flat(ins, block=block)
        sc = ss = None
    for r in range(len(ins)):
        assert_same(res["out"][r], outs[r], "out[%d]" % r)
        if block:
            assert_same(res["wc"][r], wc[r], "wire_codes[%d]" % r)
            assert_same(res["ws"][r], ws[r], "wire_scales[%d]" % r)
    if block and algo == "tree":
        assert_same(res["sc"], sc, "shard_codes")
        assert_same(res["ss"], ss, "shard_scales")


# -- staged building blocks ---------------------------------------------------

@pytest.mark.parametrize("dt", [F32, BF16])
@pytest.mark.parametrize("n", SIZES)
def test_quantize(oracle, dt, n):
    x = W.random_inputs(1, n, dt, 1000 + n, scale_spread=6.0)[0]
    codes, scales = gpu_quantize(x)
    oc, os_ = oracle.quantize(x)
    assert_same(codes, oc, "codes")
    assert_same(scales, os_, "scales")


@pytest.mark.parametrize("dt", [F32, BF16])
@pytest.mark.parametrize("n", [1, 129, 1000, 128 * 300 + 5])
def test_dequantize(oracle, dt, n):
    x = W.random_inputs(1, n, dt, 2000 + n, scale_spread=6.0)[0]
    oc, os_ = oracle.quantize(x)
    out = Guarded(n, TORCH_DT[dt])
    pcr.lp_dequantize(to_dev(oc), to_dev(os_), out.t)
    torch.cuda.synchronize()
    assert out.intact()
    assert_same(from_dev(out.t), oracle.dequantize(oc, os_, dtype=_np_dt(dt)), "out")


@pytest.mark.parametrize("dt", [F32, BF16])
@pytest.mark.parametrize("N", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("n", [5, 200, 511, 513, 4096 + 77, 128 * 37 + 15])
def test_reduce(oracle, dt, N, n):
    ins = W.random_inputs(N, n, dt, 3000 + 31 * N + n, scale_spread=4.0)
    pays = [oracle.quantize(x) for x in ins]
    out = Guarded(n, TORCH_DT[dt])
    pcr.lp_reduce([to_dev(c) for c, _ in pays], [to_dev(s) for _, s in pays], out.t)
    torch.cuda.synchronize()
    assert out.intact()
    want = oracle.reduce([c for c, _ in pays], [s for _, s in pays], dtype=_np_dt(dt))
    assert_same(from_dev(out.t), want, "out")


@pytest.mark.parametrize("dt", [F32, BF16])
def test_staged_many_grid_passes(oracle, dt):
    """lp_quantize and lp_reduce over a message long enough that every warp of
    the launch takes several grid-stride passes, with a ragged tail inside one
    lane's elements."""
    N, n = 3, 11 * (1 << 20) + 333
    ins = W.random_inputs(N, n, dt, 7100 + dt, scale_spread=5.0)
    pays = [gpu_quantize(x) for x in ins]
    want = [oracle.quantize(x) for x in ins]
    for r in range(N):
        assert_same(pays[r][0], want[r][0], "codes[%d]" % r)
        assert_same(pays[r][1], want[r][1], "scales[%d]" % r)
    out = Guarded(n, TORCH_DT[dt])
    pcr.lp_reduce([to_dev(c) for c, _ in pays], [to_dev(s) for _, s in pays], out.t)
    torch.cuda.synchronize()
    assert out.intact()
    assert_same(from_dev(out.t), oracle.reduce([c for c, _ in want], [s for _, s in want],
                                               dtype=_np_dt(dt)), "out")


# -- fused allreduce ------------------------------------------------------------

@pytest.mark.parametrize("algo,in_place", [("flat", False), ("tree", False), ("tree", True)])
def test_tile_path_full_oracle(oracle, algo, in_place):
    """FP32 low-precision allreduces of 8 ranks and 1 GiB of input or more
    take the tile path (results staged in shared memory, written by bulk
    copies): every element, code and scale against the oracle, with full
    tiles, a few full units after them and a ragged last unit."""
    N, n = 8, (1 << 25) + 3 * 1024 + 77
    assert N * n * 4 >= 1 << 30
    ins = W.random_inputs(N, n, F32, 9100 + in_place, scale_spread=3.0)
    res = gpu_allreduce(ins, algo, block=128, in_place=in_place)
    check_against_oracle(oracle, ins, algo, 128, res)



@pytest.mark.parametrize("algo", ["flat", "tree"])
@pytest.mark.parametrize("block", [128, 0])
@pytest.mark.parametrize("dt", [F32, BF16])
@pytest.mark.parametrize("N", [1, 2, 3, 5, 8, 16])
@pytest.mark.parametrize("n", [1, 127, 129, 200, 1000, 128 * 300 + 5])
def test_allreduce(oracle, algo, block, dt, N, n):
    ins = W.random_inputs(N, n, dt, 4000 + 97 * N + n, scale_spread=4.0)
    res = gpu_allreduce(ins, algo, block)
    check_against_oracle(oracle, ins, algo, block, res)


@pytest.mark.parametrize("algo", ["flat", "tree"])
@pytest.mark.parametrize("N", [4, 9, 12, 16])
def test_allreduce_more_ranks(oracle, algo, N):
    for dt in (F32, BF16):
        ins = W.random_inputs(N, 32 * 8 * 40 + 100, dt, 5000 + N, scale_spread=2.0)
        check_against_oracle(oracle, ins, algo, 128, gpu_allreduce(ins, algo))


@pytest.mark.parametrize("algo", ["flat", "tree"])
@pytest.mark.parametrize("block", [128, 0])
@pytest.mark.parametrize("dt", [F32, BF16])
def test_in_place(oracle, algo, block, dt):
    ins = W.random_inputs(4, 128 * 77 + 9, dt, 6000 + block, scale_spread=3.0)
    res = gpu_allreduce(ins, algo, block, in_place=True)
    check_against_oracle(oracle, ins, algo, block, res)


@pytest.mark.parametrize("dt", [F32, BF16])
def test_degenerate_and_signed_zero_blocks(oracle, dt):
    n = 128 * 6 + 40
    ins = []
    for r in range(3):
        x = np.random.default_rng(r).standard_normal(n).astype(np.float32)
        x[:128] = 0.0
        x[1:128:3] = -0.0
        x[128:256] *= np.float32(1e-37)     # degenerate: 448/a overflows
        x[256:384] *= np.float32(1e-35)     # tiny but quantized normally
        x[384:512] *= np.float32(1e30)      # large values
        x[512:640] = np.float32(3.0)        # constant block
        if dt == BF16:
            x = W.to_bf16_bits(x)
        ins.append(x)
    for algo in ("flat", "tree"):
        check_against_oracle(oracle, ins, algo, 128, gpu_allreduce(ins, algo))


def test_all_codes_and_rounding_boundaries(oracle):
    # A block whose maximum is 448 has s = 1 and multiplier 1, so its other
    # elements reach the E4M3 encoder unchanged: every code value, every
    # midpoint between neighbours, and the floats just around each midpoint.
    table = oracle.e4m3_decode_all()
    vals = [table[c] for c in range(256) if c not in (0x7F, 0xFF)]
    pos = np.array([table[c] for c in range(127)], dtype=np.float64)
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    up = np.nextafter(mids, np.float32(np.inf))
    down = np.nextafter(mids, np.float32(0))
    body = np.concatenate([vals, mids, up, down, -mids, -up, -down,
                           [np.nan]]).astype(np.float32)
    per = 127
    blocks = []
    for i in range(0, body.size, per):
        chunk = body[i:i + per]
        blk = np.zeros(128, dtype=np.float32)
        blk[0] = 448.0
        blk[1:1 + chunk.size] = chunk
        blocks.append(blk)
    x = np.concatenate(blocks)
    codes, scales = gpu_quantize(x)
    oc, os_ = oracle.quantize(x)
    assert np.all(os_ == 1.0)
    assert_same(scales, os_, "scales")
    assert_same(codes, oc, "codes")
    # every one of the 256 codes except the negative NaN was produced
    assert set(range(256)) - set(codes.tolist()) <= {0xFF}


def test_staged_equals_fused(oracle):
    for dt in (F32, BF16):
        n = 128 * 50 + 3
        ins = W.random_inputs(5, n, dt, 7000 + dt, scale_spread=3.0)
        pays = [gpu_quantize(x) for x in ins]
        out = torch.empty(n, dtype=TORCH_DT[dt], device="cuda")
        pcr.lp_reduce([to_dev(c) for c, _ in pays], [to_dev(s) for _, s in pays], out)
        torch.cuda.synchronize()
        fused = gpu_allreduce(ins, "flat")
        assert_same(from_dev(out), fused["out"][0], "staged vs fused")


def test_torch_full_example_facade(oracle):
    from oracle_pins import read_torch_full_cases
    for N, rows, cols, want in read_torch_full_cases():
        ts = [torch.full((rows, cols), float(r), dtype=torch.float, device="cuda")
              for r in range(N)]
        algo, block = pcr.allreduce_sim(ts, low_precision=False)
        torch.cuda.synchronize()
        assert block == 0
        for t in ts:
            assert torch.all(t == want).item(), (N, want)
        # low precision forced on (threshold 0): equal to the oracle, bit for bit
        ins = [np.full(rows * cols, float(r), dtype=np.float32) for r in range(N)]
        for algo in ("flat", "tree"):
            check_against_oracle(oracle, ins, algo, 128, gpu_allreduce(ins, algo))


def test_zero_length_is_noop():
    x = torch.empty(0, dtype=torch.float32, device="cuda")
    pcr.dda_flat_sim([x, x], [x, x], block=0)
    c = torch.empty(0, dtype=torch.uint8, device="cuda")
    s = torch.empty(0, dtype=torch.float32, device="cuda")
    pcr.lp_quantize(x, c, s)
    torch.cuda.synchronize()


@pytest.mark.parametrize("block", [0, 128])
def test_cuda_graph_replay(oracle, block):
    N, n = 8, 32 * 8192
    ins = W.random_inputs(N, n, BF16, 8100 + block, scale_spread=1.0)
    xd = [to_dev(x) for x in ins]
    outs = [torch.empty_like(t) for t in xd]
    kw = {}
    if block:
        kw = dict(wire_codes=[torch.empty(n, dtype=torch.uint8, device="cuda")
                              for _ in range(N)],
                  wire_scales=[torch.empty(pcr.nblocks(n), dtype=torch.float32,
                                           device="cuda") for _ in range(N)])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pcr.dda_flat_sim(xd, outs, block=block, **kw)  # warm-up outside capture
    torch.cuda.synchronize()
    for o in outs:
        o.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pcr.dda_flat_sim(xd, outs, block=block, **kw)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    want = oracle.flat(ins, block=block)[0]
    for r in range(N):
        assert_same(from_dev(outs[r]), want[r], "out[%d]" % r)


@pytest.mark.parametrize("graph", [False, True])
def test_chained_launches_keep_stream_order(oracle, graph):
    """Back-to-back dependent calls on one stream with no synchronisation in
    between, each reading what the previous one wrote: in-place flat and tree
    allreduces (exact and low precision), then a staged quantize -> reduce.
    The kernels are launched with programmatic dependent launch; the result
    must be the oracle's chain of the same calls, eagerly and replayed from a
    CUDA graph."""
    N, n = 8, 32 * 8192 + 77
    ins = W.random_inputs(N, n, BF16, 8300, scale_spread=1.0)
    chain = [("flat", 0), ("flat", 128), ("tree", 128), ("flat", 128), ("tree", 0),
             ("flat", 128)]
    want = [x.copy() for x in ins]
    for algo, block in chain:
        res = (oracle.flat if algo == "flat" else oracle.tree)(want, block=block)[0]
        want = [r.copy() for r in res]
    pays = [oracle.quantize(x) for x in want]
    want_red = oracle.reduce([c for c, _ in pays], [s for _, s in pays], dtype=np.uint16)

    xd = [to_dev(x) for x in ins]
    wc = [torch.empty(n, dtype=torch.uint8, device="cuda") for _ in range(N)]
    ws = [torch.empty(pcr.nblocks(n), dtype=torch.float32, device="cuda") for _ in range(N)]
    sc = torch.empty(n, dtype=torch.uint8, device="cuda")
    ss = torch.empty(pcr.nblocks(n), dtype=torch.float32, device="cuda")
    red = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()

    def calls():
        for algo, block in chain:
            kw = dict(wire_codes=wc, wire_scales=ws) if block else {}
            if algo == "flat":
                pcr.dda_flat_sim(xd, xd, block=block, stream=s, **kw)
            else:
                if block:
                    kw.update(shard_codes=sc, shard_scales=ss)
                pcr.dda_tree_sim(xd, xd, block=block, stream=s, **kw)
        for r in range(N):
            pcr.lp_quantize(xd[r], wc[r], ws[r], stream=s)
        pcr.lp_reduce(wc, ws, red, stream=s)

    torch.cuda.synchronize()
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            calls()
        for t, x in zip(xd, ins):   # capture ran nothing; start from the inputs
            t.copy_(to_dev(x))
        torch.cuda.synchronize()
        g.replay()
    else:
        with torch.cuda.stream(s):
            calls()
    torch.cuda.synchronize()
    for r in range(N):
        assert_same(from_dev(xd[r]), want[r], "chained out[%d]" % r)
    assert_same(from_dev(red), want_red, "chained reduce")


def test_pages_example_with_host_tensors():
    # the example as the pages write it: torch.full on the host, SUM in place
    from oracle_pins import read_torch_full_cases
    for N, rows, cols, want in read_torch_full_cases():
        ts = [torch.full((rows, cols), float(r), dtype=torch.float) for r in range(N)]
        algo, block = pcr.allreduce_sim(ts)
        assert (algo, block) == ("flat", 0)
        for t in ts:
            assert not t.is_cuda and torch.all(t == want).item(), (N, want)
        ts = [torch.full((rows, cols), float(r), dtype=torch.bfloat16) for r in range(N)]
        pcr.allreduce_sim(ts, algo="tree")
        for t in ts:
            assert torch.all(t.float() == want).item(), (N, want)
