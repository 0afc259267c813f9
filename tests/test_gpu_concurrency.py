"""Calls from several host threads at once, each on its own CUDA stream and
buffers (ctypes releases the GIL during a library call, so the calls really
overlap): results equal the single-threaded ones, bit for bit."""
import threading

import pytest
import torch

from precision_collective_reduction_gb300 import runner, workloads as W

pytestmark = pytest.mark.gpu


def test_threads_on_separate_streams():
    cases = [(2, 128 * 500 + 3, W.F32, 128, "flat"), (8, 32 * 8192, W.BF16, 0, "flat"),
             (5, 128 * 999, W.BF16, 128, "tree"), (16, 4096 + 77, W.F32, 128, "tree")]
    bufs, refs = [], []
    base = torch.cuda.current_stream().cuda_stream
    for i, (N, n, dt, block, algo) in enumerate(cases):
        b = runner.RankBuffers(N, n, dt, block)
        b.load(W.random_inputs(N, n, dt, 600 + i, scale_spread=2.0))
        b.run(algo, base)
        torch.cuda.synchronize()
        refs.append([o.clone() for o in b.outs])
        for o in b.outs:
            o.zero_()
        bufs.append(b)
    errors = []

    def work(i):
        try:
            N, n, dt, block, algo = cases[i]
            s = torch.cuda.Stream()
            for _ in range(25):
                bufs[i].run(algo, s.cuda_stream)
            s.synchronize()
        except Exception as e:  # reported by the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    torch.cuda.synchronize()
    for b, ref in zip(bufs, refs):
        for o, r in zip(b.outs, ref):
            assert torch.equal(o.view(torch.uint8), r.view(torch.uint8))
