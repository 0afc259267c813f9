"""The two readings of the block-scale step, compared on the workloads' inputs.

The pages name FP8 quantization and FP32 arithmetic but not how an element is
scaled ("RCCLX: AMD GPU communication, Meta open source", code-journey.com,
"Funcionalidade Principal 2"). The library encodes fp8(x * fl(448 / a)), one
division per 128-element block; the other plain reading is fp8(x / fl(a /
448)), one division per element. Both give the same scale; their codes can
differ only where x * inv and x / s fall on opposite sides of a rounding
boundary of the E4M3 grid, and then by one step. The oracle carries the
divide reading behind a switch (off by default) for this comparison only.

Run as a script, it prints the counts on the five workloads at full size.
"""
import json
import os
import sys

import numpy as np

if __name__ == "__main__":
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
from precision_collective_reduction_gb300 import workloads as W  # noqa: E402

SAMPLE = 1 << 18  # elements per rank for the CPU test


def compare(oracle, w, n=None):
    """Codes that differ between the two readings over every rank's message
    of workload w (first n elements per rank): (differing, total, max code
    distance, scales identical)."""
    diff = total = 0
    dist = 0
    scales_same = True
    table = oracle.e4m3_decode_all()
    for x in W.draw_all(w, n):
        c_mul, s_mul = oracle.quantize(x)
        with oracle.divide_reading():
            c_div, s_div = oracle.quantize(x)
        scales_same &= np.array_equal(s_mul.view(np.uint32), s_div.view(np.uint32))
        d = c_mul != c_div
        diff += int(np.count_nonzero(d))
        total += x.size
        if d.any():
            # distance in grid steps: position of each value on the signed grid
            order = np.argsort(table[:127])
            rank = np.empty(127, dtype=np.int64)
            rank[order] = np.arange(127)
            a, b = c_mul[d], c_div[d]
            assert np.array_equal(a & 0x80, b & 0x80)
            dist = max(dist, int(np.max(np.abs(rank[a & 0x7F] - rank[b & 0x7F]))))
    return diff, total, dist, scales_same


def test_readings_differ_by_at_most_one_step(oracle):
    seen = 0
    for w in W.WORKLOADS:
        if not w.block:
            continue
        diff, total, dist, same = compare(oracle, w, SAMPLE)
        assert same, w.name
        assert dist <= 1, (w.name, dist)
        assert diff <= total // 1000, (w.name, diff, total)
        seen += diff
    # the readings are not identical on these inputs: the switch takes effect
    assert seen > 0


def test_switch_is_off_by_default(oracle):
    x = W.random_inputs(1, 128 * 50, W.F32, 3, scale_spread=2.0)[0]
    c0, s0 = oracle.quantize(x)
    with oracle.divide_reading():
        pass
    c1, s1 = oracle.quantize(x)
    assert np.array_equal(c0, c1) and np.array_equal(s0, s1)


if __name__ == "__main__":
    import oracle as orc
    for w in W.WORKLOADS:
        if w.block:
            diff, total, dist, same = compare(orc, w)
            print(json.dumps({"workload": w.name, "codes": total, "differing": diff,
                              "fraction": diff / total, "max_steps": dist,
                              "scales_identical": bool(same)}), flush=True)
