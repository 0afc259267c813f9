"""The bounds-checked build of the library (liblpcoll_debug_bounds.so) on the
ragged cases: every global load, store and bulk copy of every kernel must
stay inside the buffers its call passed, at the sizes the header gives them.

In that build an access outside the listed buffers is skipped and recorded
instead of made (nothing traps), so a stray read or write of any kernel shows
up here as a flag, with no fault. The guard bands of the parity tests catch
only stray writes just past a buffer's end; these checks also catch reads,
and writes anywhere outside the call's buffers.

The cases: the 300 seeded random configurations of every entry point (ragged
and unaligned lengths, 1 to 16 ranks, both dtypes, exact and low precision,
every FP8 format and block size, in place or not), each also compared with
the oracle, so the checks are known to have skipped nothing; the allreduces
at ragged sizes; the tile path at 8 x (32 Mi + 3149) FP32, compared with the
normal build; the host-buffer pipeline; the non-allocating entry point. A
last case lists every buffer a few bytes short and checks that the checks
fire, without any access leaving the real buffers.
"""
import numpy as np
import pytest
import torch

import precision_collective_reduction_gb300 as pcr
import test_gpu_fuzz as fuzz
from precision_collective_reduction_gb300 import _binding as B
from precision_collective_reduction_gb300 import build as lib_build
from precision_collective_reduction_gb300 import runner, workloads as W
from precision_collective_reduction_gb300.host import HostAllreduce
from gpu_util import from_dev, same_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def debug_lib():
    path = lib_build.build(debug_bounds=True)
    with B.using_library(path) as L:
        st, _ = B.debug_bounds_errors()
        assert st in (0, 1)  # a fresh record; clears anything left over
        yield L


def _no_bad_access(what):
    st, bad = B.debug_bounds_errors()
    assert st == 0, "%s: access outside the call's buffers (status %d, first at 0x%x)" % (
        what, st, bad)


@pytest.mark.parametrize("cfg", list(fuzz._configs()), ids=lambda c: "%d-%s" % (c[0], c[1]))
def test_random_config_in_bounds(oracle, debug_lib, cfg):
    fuzz.test_random_config(oracle, cfg)
    _no_bad_access("config %d (%s)" % (cfg[0], cfg[1]))


@pytest.mark.parametrize("algo", ["flat", "tree"])
@pytest.mark.parametrize("block", [128, 0])
@pytest.mark.parametrize("dt", [W.F32, W.BF16])
@pytest.mark.parametrize("N", [1, 3, 8, 16])
@pytest.mark.parametrize("n", [1, 127, 129, 200, 4096 + 77, 128 * 300 + 5])
def test_allreduce_in_bounds(oracle, debug_lib, algo, block, dt, N, n):
    ins = W.random_inputs(N, n, dt, 3000 + N + n, scale_spread=3.0)
    bufs = runner.RankBuffers(N, n, dt, block, separate_tree_out=True)
    bufs.load(ins)
    bufs.run(algo, torch.cuda.current_stream().cuda_stream)
    _no_bad_access("%s N=%d n=%d" % (algo, N, n))
    want = (oracle.tree if algo == "tree" else oracle.flat)(ins, block=block)[0]
    outs = bufs.tree_outs if algo == "tree" else bufs.outs
    for r in range(N):
        assert same_bits(from_dev(outs[r]), want[r]), r


@pytest.mark.parametrize("algo,in_place", [("flat", False), ("tree", True)])
def test_tile_path_in_bounds(debug_lib, algo, in_place):
    # 8 ranks x (32 Mi + 3149) FP32: 1 GiB of input, the tile path with a
    # ragged tail after the last tile. The normal build's result is the
    # reference (it equals the oracle's in the parity tests).
    N, n = 8, (32 << 20) + 3149
    g = torch.Generator(device="cuda").manual_seed(11)
    ins = [torch.randn(n, device="cuda", generator=g) for _ in range(N)]
    nb = pcr.nblocks(n)
    wc = [torch.empty(n, dtype=torch.uint8, device="cuda") for _ in range(N)]
    ws = [torch.empty(nb, dtype=torch.float32, device="cuda") for _ in range(N)]
    sc = torch.empty(n, dtype=torch.uint8, device="cuda")
    ss = torch.empty(nb, dtype=torch.float32, device="cuda")

    def run(outs_):
        if algo == "flat":
            pcr.dda_flat_sim(ins_, outs_, wire_codes=wc, wire_scales=ws)
        else:
            pcr.dda_tree_sim(ins_, outs_, wire_codes=wc, wire_scales=ws, shard_codes=sc,
                             shard_scales=ss)
    with B.using_library(lib_build.LIB):
        ins_ = [t.clone() for t in ins]
        want = [torch.empty_like(t) for t in ins]
        run(want)
        torch.cuda.synchronize()
    ins_ = [t.clone() for t in ins]
    outs = ins_ if in_place else [torch.empty_like(t) for t in ins]
    run(outs)
    _no_bad_access("tile path %s" % algo)
    for r in range(N):
        assert torch.equal(outs[r].view(torch.int32), want[r].view(torch.int32)), r
    del ins, ins_, outs, want, wc, ws, sc, ss
    torch.cuda.empty_cache()


@pytest.mark.parametrize("N,m", [(3, 1001), (8, 777), (5, 128 * 40 + 3)])
@pytest.mark.parametrize("block", [128, 0])
@pytest.mark.parametrize("dt", [W.F32, W.BF16])
def test_gather_and_alltoall_unaligned_in_bounds(oracle, debug_lib, N, m, block, dt):
    tdt = torch.float32 if dt == W.F32 else torch.bfloat16
    ins = W.random_inputs(N, m, dt, 4000 + N, scale_spread=2.0)
    outs = [torch.empty(N * m, dtype=tdt, device="cuda") for _ in range(N)]
    wc = [torch.empty(N * m, dtype=torch.uint8, device="cuda") for _ in range(N)]
    ws = [torch.empty(N * pcr.nblocks(m), dtype=torch.float32, device="cuda")
          for _ in range(N)]
    pcr.all_gather_sim([to_dev(x) for x in ins], outs, block=block,
                       wire_codes=[t[:m] for t in wc],
                       wire_scales=[t[:pcr.nblocks(m)] for t in ws])
    _no_bad_access("all-gather N=%d m=%d" % (N, m))
    want = oracle.all_gather(ins, block=block)[0]
    for r in range(N):
        assert same_bits(from_dev(outs[r]), want[r]), r
    a2a = W.random_inputs(N, N * m, dt, 5000 + N, scale_spread=2.0)
    pcr.all_to_all_sim([to_dev(x) for x in a2a], outs, block=block, wire_codes=wc,
                       wire_scales=ws)
    _no_bad_access("all-to-all N=%d c=%d" % (N, m))
    want = oracle.all_to_all(a2a, block=block)[0]
    for r in range(N):
        assert same_bits(from_dev(outs[r]), want[r]), r


def test_host_pipeline_in_bounds(oracle, debug_lib):
    N, n = 3, 128 * 100 + 37
    ins = W.random_inputs(N, n, W.F32, 6000, scale_spread=2.0)
    h = HostAllreduce(N, n, W.F32, 128, algos=("flat", "tree"), chunk=128 * 16, slots=2)
    hout = {a: [torch.empty(n, dtype=torch.float32).pin_memory() for _ in range(N)]
            for a in ("flat", "tree")}
    h.run([torch.from_numpy(x).pin_memory() for x in ins], hout)
    _no_bad_access("host pipeline")
    for a, fn in (("flat", oracle.flat), ("tree", oracle.tree)):
        want = fn(ins)[0]
        for r in range(N):
            assert same_bits(hout[a][r].numpy(), want[r]), (a, r)


@pytest.mark.parametrize("dt,N,n", [(W.F32, 3, 1001), (W.BF16, 8, 128 * 50 + 7)])
def test_noalloc_in_bounds(oracle, debug_lib, dt, N, n):
    ins = W.random_inputs(N, n, dt, 7000 + N, scale_spread=2.0)
    xd = [to_dev(x) for x in ins]
    outs = [torch.empty_like(t) for t in xd]
    pcr.dda_flat_sim_noalloc(xd, outs)
    _no_bad_access("noalloc N=%d n=%d" % (N, n))
    want = oracle.flat(ins)[0]
    for r in range(N):
        assert same_bits(from_dev(outs[r]), want[r]), r


def test_checks_fire_on_shrunk_buffers(debug_lib):
    # The next call lists every buffer 4 bytes short: the quantize kernel's
    # last input load, code store and scale store then fail their checks
    # and are skipped (no access leaves the real buffers), and the record
    # says so. The call after it is clean again.
    n = 1000
    x = torch.randn(n, device="cuda")
    c = torch.empty(n, dtype=torch.uint8, device="cuda")
    s = torch.empty(pcr.nblocks(n), dtype=torch.float32, device="cuda")
    B.lib().lpcoll_debug_bounds_shrink(4)
    pcr.lp_quantize(x, c, s)
    st, bad = B.debug_bounds_errors()
    assert st == 1
    spans = [(t.data_ptr(), t.data_ptr() + t.numel() * t.element_size()) for t in (x, c, s)]
    assert any(lo <= bad < hi for lo, hi in spans), hex(bad)
    pcr.lp_quantize(x, c, s)
    _no_bad_access("quantize after the shrunk call")
    assert np.isfinite(from_dev(s)).all()
