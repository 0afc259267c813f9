"""Pins for the CPU oracle.

Each ``pin_*`` function checks the oracle (passed in as the ``oracle`` module,
or that module routed through a modified build) against something that does
not come from the oracle itself:

- the OCP FP8 specification's E4M3 reference points (``golden/``);
- PyTorch's own ``float8_e4m3fn`` and ``bfloat16`` conversions, an
  independent implementation of the same round-to-nearest-even codecs;
- structural facts of the format (monotone grid, spacing per binade,
  midpoints that must round to the even code);
- IEEE binary32 arithmetic worked out by hand (fixed summation order);
- invariants of the method: exact round trip of representable blocks, the
  2^-4 relative error bound of a 3-bit mantissa, order independence of the
  block maximum, N = 1 equal to the round trip, identical outputs on every
  rank, reduce-scatter + all-gather equal to allreduce on the exact path;
- an FP64 brute-force sum with the error bound the quantization allows;
- the pages' torch.full / allreduce(SUM) example and their compression ratio.

A pin raises AssertionError when it fails. ``test_oracle_pins`` runs them all
against the oracle; ``test_oracle_mutants`` checks that planted mistakes in
the oracle make at least one of them fail.
"""
import math
import os

import numpy as np
import torch

from precision_collective_reduction_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
F32, BF16 = 0, 1


# -- independent helpers (PyTorch's codecs, numpy IEEE arithmetic) -----------

def torch_e4m3_table():
    """float32 value of each of the 256 codes, decoded by PyTorch."""
    return (torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn)
            .float().numpy())


def torch_e4m3_encode(y):
    """PyTorch's RNE float32 -> e4m3fn (valid for |y| <= 448)."""
    t = torch.from_numpy(np.ascontiguousarray(y, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def torch_bf16_bits(x):
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def widen(a):
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32)
    return a


def nextafter32(x, toward):
    return np.nextafter(np.float32(x), np.float32(toward), dtype=np.float32)


def same_bits(a, b):
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    return a.shape == b.shape and np.array_equal(a.view(np.uint8), b.view(np.uint8))


def read_spec_points():
    pts = []
    with open(os.path.join(GOLDEN, "ofp8_e4m3_spec_points.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                c, v = line.split()
                pts.append((int(c, 16), float(v)))
    return pts


def read_torch_full_cases():
    cases = []
    with open(os.path.join(GOLDEN, "torch_full_allreduce.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                nr, rows, cols, val = line.split()
                cases.append((int(nr), int(rows), int(cols), float(val)))
    return cases


# -- E4M3 codec -------------------------------------------------------------

def pin_spec_points(oracle):
    for code, value in read_spec_points():
        got = oracle.e4m3_decode(code)
        if math.isnan(value):
            assert math.isnan(got), (hex(code), got)
            continue
        assert got == value and math.copysign(1, got) == math.copysign(1, value), \
            (hex(code), got, value)
        assert oracle.e4m3_encode(value) == code, (value, hex(code))


def pin_decode_vs_library(oracle):
    ours = oracle.e4m3_decode_all()
    ref = torch_e4m3_table()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert same_bits(ours[~nan], ref[~nan])


def pin_decode_structure(oracle):
    v = oracle.e4m3_decode_all().astype(np.float64)
    pos = v[:127]
    assert np.all(np.diff(pos) > 0), "positive codes must increase"
    gaps = np.diff(pos)
    # spacing is constant inside each exponent group of 8 codes, equal in the
    # subnormal group and the first normal group, and doubles after that
    spacing = [gaps[g * 8] for g in range(15)]
    for g in range(15):
        hi = min(g * 8 + 7, 126)
        assert np.all(gaps[g * 8:hi] == spacing[g]), g
    assert spacing[0] == spacing[1]
    for g in range(2, 15):
        assert spacing[g] == 2 * spacing[g - 1], g
    neg = oracle.e4m3_decode_all()
    for c in range(127):
        a, b = neg[c], neg[c | 0x80]
        assert np.float32(-a).view(np.uint32) == np.float32(b).view(np.uint32), c


def pin_encode_roundtrip(oracle):
    table = torch_e4m3_table()
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_encode(table[c]) == c, hex(c)


def pin_encode_ties(oracle):
    table = torch_e4m3_table().astype(np.float64)
    for c in range(126):
        lo, hi = table[c], table[c + 1]
        mid = (lo + hi) / 2
        assert float(np.float32(mid)) == mid
        even = c if c % 2 == 0 else c + 1
        for sgn, mask in ((1.0, 0x00), (-1.0, 0x80)):
            m = np.float32(sgn * mid)
            assert oracle.e4m3_encode(m) == (even | mask), (c, sgn)
            up = nextafter32(m, sgn * np.inf)
            down = nextafter32(m, 0.0)
            assert oracle.e4m3_encode(up) == ((c + 1) | mask), (c, sgn, "above")
            assert oracle.e4m3_encode(down) == (c | mask), (c, sgn, "below")


def pin_encode_vs_library(oracle):
    g = np.random.default_rng(1234)
    mag = np.exp2(g.uniform(-14, math.log2(448), 20000)).astype(np.float32)
    y = np.concatenate([mag, -mag, g.uniform(-448, 448, 5000).astype(np.float32)])
    y = y[np.abs(y) <= 448]
    assert np.array_equal(oracle.e4m3_encode_array(y), torch_e4m3_encode(y))


def pin_saturation(oracle):
    big = [448.0, float(nextafter32(448, np.inf)), 450.0, 463.9, 464.0, 479.0,
           480.0, 1e30, float(np.finfo(np.float32).max), math.inf]
    for v in big:
        assert oracle.e4m3_encode(v) == 0x7E, v
        assert oracle.e4m3_encode(-v) == 0xFE, -v
    assert oracle.e4m3_encode(math.nan) == 0x7F


def pin_subnormal_boundary(oracle):
    cases = [(2.0 ** -10, 0x00), (float(nextafter32(2.0 ** -10, 1)), 0x01),
             (3 * 2.0 ** -10, 0x02), (5 * 2.0 ** -10, 0x02),
             (15 * 2.0 ** -10, 0x08), (-(2.0 ** -10), 0x80), (1e-30, 0x00),
             (-1e-30, 0x80), (0.0, 0x00), (-0.0, 0x80)]
    for v, code in cases:
        assert oracle.e4m3_encode(v) == code, (v, hex(code))


# -- BF16 codec -------------------------------------------------------------

def pin_bf16(oracle):
    g = np.random.default_rng(99)
    x = np.concatenate([
        g.standard_normal(4000).astype(np.float32),
        (g.standard_normal(2000) * 1e-30).astype(np.float32),
        (g.standard_normal(2000) * 1e30).astype(np.float32),
        # exact ties: low 16 bits 0x8000, both parities of bit 16
        (np.arange(1000, dtype=np.uint32) * 0x10000 + 0x3F808000).view(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 1e-45, -1e-45,
                  np.finfo(np.float32).max], dtype=np.float32),
    ])
    assert np.array_equal(oracle.f32_to_bf16_array(x), torch_bf16_bits(x))
    h = np.arange(0, 65536, 7, dtype=np.uint16)
    ref = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float().numpy()
    ours = np.array([oracle.bf16_to_f32(int(v)) for v in h], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert same_bits(ours[~nan], ref[~nan])


# -- block scale and quantization ------------------------------------------

def pin_scale_rule(oracle):
    g = np.random.default_rng(7)
    a = np.exp2(g.uniform(-100, 100, 2000)).astype(np.float32)
    for v in a:
        s, inv = oracle.block_scale(v)
        assert s == np.float32(v) / np.float32(448.0), v
        assert inv == np.float32(448.0) / np.float32(v), v
    for v in (0.0, 1e-37, 1e-36):
        assert oracle.block_scale(v) == (0.0, 0.0), v
    s, inv = oracle.block_scale(2e-36)
    assert s > 0 and np.isfinite(inv)


def pin_reciprocal_rule(oracle):
    # The element multiplier is the per-block reciprocal 448/a, not a division
    # by the stored scale s = a/448. Find elements where the two readings give
    # different codes (numpy IEEE binary32 arithmetic, PyTorch's encoder) and
    # check that the oracle follows the reciprocal.
    g = np.random.default_rng(21)
    table = torch_e4m3_table()
    mids = (table[56:125].astype(np.float64) + table[57:126]) / 2
    found = 0
    for a in np.exp2(g.uniform(-10, 10, 400)).astype(np.float32):
        inv = np.float32(448.0) / a
        s = a / np.float32(448.0)
        for m in g.choice(mids, 4):
            x0 = np.float32(np.float32(m) / inv)
            xs = x0 + np.arange(-3, 4, dtype=np.float32) * np.spacing(x0)
            xs = xs[np.abs(xs) < a]
            y_mul = (xs * inv).astype(np.float32)
            y_div = (xs / s).astype(np.float32)
            c_mul = torch_e4m3_encode(y_mul)
            diff = c_mul != torch_e4m3_encode(y_div)
            for x, c in zip(xs[diff], c_mul[diff]):
                blk = np.zeros(128, dtype=np.float32)
                blk[0], blk[1] = a, x
                codes, scales = oracle.quantize(blk)
                assert scales[0] == s and codes[1] == c, (a, x)
                found += 1
    assert found >= 10, found


def pin_representable_roundtrip(oracle):
    g = np.random.default_rng(11)
    table = torch_e4m3_table()
    valid = np.array([c for c in range(256) if c not in (0x7F, 0xFF)],
                     dtype=np.uint8)
    for j in range(-20, 21, 4):
        s = np.float32(2.0 ** j)
        codes = g.choice(valid, size=128 * 5)
        codes[::128] = g.choice([0x7E, 0xFE], size=5)
        x = (table[codes] * s).astype(np.float32)
        for dt in (F32, BF16):
            xin = torch_bf16_bits(x) if dt == BF16 else x
            if dt == BF16:
                assert same_bits(widen(xin), x)
            qc, qs = oracle.quantize(xin)
            assert np.array_equal(qc, codes), j
            assert np.all(qs == s), j
            back = oracle.dequantize(qc, qs, dtype=xin.dtype)
            assert same_bits(back, xin), j


def _error_bound_ok(x, back, scales, n):
    x64 = x.astype(np.float64)
    d = np.abs(back.astype(np.float64) - x64)
    s = np.repeat(scales.astype(np.float64), 128)[:n]
    with np.errstate(divide="ignore", invalid="ignore"):
        y = np.where(s > 0, np.abs(x64) / s, 0.0)
    normal = y >= 2.0 ** -6
    ok_n = d[normal] <= 2.0 ** -4 * np.abs(x64[normal])
    ok_s = d[~normal] <= 2.0 ** -10 * s[~normal] * (1 + 2.0 ** -20) + \
        2.0 ** -22 * np.abs(x64[~normal])
    return bool(np.all(ok_n) and np.all(ok_s))


def pin_error_bound(oracle):
    # 10^7 values per distribution (plus a ragged tail block)
    n = 10 ** 7 + 37
    g = np.random.default_rng(5)
    cases = [
        g.standard_normal(n).astype(np.float32),
        g.laplace(0, 1, n).astype(np.float32),
        W.random_inputs(1, n, F32, 17, scale_spread=30.0)[0],
        (g.standard_normal(n) * 1e-30).astype(np.float32),
        (g.standard_normal(n) * 1e30).astype(np.float32),
    ]
    for x in cases:
        codes, scales = oracle.quantize(x)
        back = oracle.dequantize(codes, scales)
        assert _error_bound_ok(x, back, scales, n)


def pin_degenerate_blocks(oracle):
    x = np.zeros(256, dtype=np.float32)
    x[1::2] = -0.0
    x[128:] = (np.random.default_rng(3).standard_normal(128) * 1e-37).astype(np.float32)
    codes, scales = oracle.quantize(x)
    assert np.all(scales == 0.0)
    expect = np.where(np.signbit(x), 0x80, 0x00).astype(np.uint8)
    assert np.array_equal(codes, expect)
    back = oracle.dequantize(codes, scales)
    assert np.all(back == 0.0) and np.array_equal(np.signbit(back), np.signbit(x))
    # a small but non-degenerate block is quantized normally
    y = np.full(128, 1e-35, dtype=np.float32)
    yc, ys = oracle.quantize(y)
    assert ys[0] > 0 and np.all(yc == 0x7E)


def pin_absmax_permutation(oracle):
    g = np.random.default_rng(8)
    x = g.standard_normal(128).astype(np.float32)
    codes, scales = oracle.quantize(x)
    for _ in range(5):
        p = g.permutation(128)
        pc, ps = oracle.quantize(x[p])
        assert ps[0] == scales[0]
        assert np.array_equal(pc, codes[p])


def pin_tail_block(oracle):
    g = np.random.default_rng(9)
    x = g.standard_normal(200).astype(np.float32)
    x[150] = 40.0  # the tail block's own maximum
    codes, scales = oracle.quantize(x)
    hc, hs = oracle.quantize(x[:128])
    tc, ts = oracle.quantize(x[128:])
    assert scales.size == 2
    assert np.array_equal(codes[:128], hc) and scales[0] == hs[0]
    assert np.array_equal(codes[128:], tc) and scales[1] == ts[0]
    assert scales[1] == np.float32(40.0) / np.float32(448.0)


def pin_constant_blocks(oracle):
    for j in (-30, -3, 0, 7, 60):
        for sgn in (1.0, -1.0):
            x = np.full(300, sgn * 448.0 * 2.0 ** j, dtype=np.float32)
            codes, scales = oracle.quantize(x)
            assert np.all(codes == (0x7E if sgn > 0 else 0xFE))
            assert np.all(scales == np.float32(2.0 ** j))
    x = np.full(128, 3.0, dtype=np.float32)
    codes, scales = oracle.quantize(x)
    assert np.all(codes == 0x7E)
    assert scales[0] == np.float32(3.0) / np.float32(448.0)


# -- reduction and allreduce -------------------------------------------------

def pin_n1_equals_roundtrip(oracle):
    g = np.random.default_rng(12)
    x = g.standard_normal(1000).astype(np.float32)
    x[:128] = 0.0
    x[3] = -0.0
    for xin in (x, torch_bf16_bits(x)):
        codes, scales = oracle.quantize(xin)
        rt = oracle.dequantize(codes, scales, dtype=xin.dtype)
        assert same_bits(oracle.reduce([codes], [scales], dtype=xin.dtype), rt)
        outs, _, _ = oracle.flat([xin])
        assert same_bits(outs[0], rt)
        ex, _, _ = oracle.flat([xin], block=0)
        assert same_bits(ex[0], xin)


def pin_fixed_order(oracle):
    # exact path, IEEE binary32 by hand: (1 + 2^-24) rounds to 1 (tie, even),
    # so rank order 0,1,2 gives 1.0; the reverse order would give 1 + 2^-23.
    e = 2.0 ** -24
    for vals, want in (((1.0, e, e), 1.0), ((e, e, 1.0), 1.0 + 2.0 ** -23)):
        ins = [np.array([v], dtype=np.float32) for v in vals]
        outs, _, _ = oracle.flat(ins, block=0)
        assert all(o[0] == np.float32(want) for o in outs), (vals, outs)
    # low precision with exactly representable payloads: rank 0 holds 2^24
    # in a block of scale 2^20, ranks 1 and 2 hold 1.0 in blocks of scale 1.
    # 2^24 + 1 ties to 2^24, so the fixed order gives 2^24 (not 2^24 + 2).
    ins = []
    for r in range(3):
        x = np.zeros(128, dtype=np.float32)
        x[0] = 448.0 * 2.0 ** 20 if r == 0 else 448.0
        x[5] = 2.0 ** 24 if r == 0 else 1.0
        ins.append(x)
    outs, _, _ = oracle.flat(ins)
    assert all(o[5] == np.float32(2.0 ** 24) for o in outs), outs[0][5]
    # the payload-level reductions, codes and scales written by hand: rank 0
    # decodes to 1.0 (the code of 1.0 with scale 1), ranks 1 and 2 to 2^-24
    # (the same code with scale 2^-24). Rank order gives 1.0, the reverse
    # order 1 + 2^-23: for the main reduce and for every format and block
    # size of the variants.
    one = {E4M3: 0x38, E5M2: 0x3C}  # sign 0, exponent = bias, mantissa 0
    for fmt, block in [(f, b) for f in (E4M3, E5M2) for b in (32, 64, 128, 256)] + [(None, 128)]:
        n = block + 3
        nb = -(-n // block)
        code = one[E4M3 if fmt is None else fmt]
        codes = [np.full(n, code, dtype=np.uint8) for _ in range(3)]
        scales = [np.full(nb, s, dtype=np.float32) for s in (1.0, e, e)]
        for order, want in ((slice(None), 1.0), (slice(None, None, -1), 1.0 + 2.0 ** -23)):
            cs, ss = codes[order], scales[order]
            out = (oracle.reduce(cs, ss) if fmt is None
                   else oracle.reduce_fmt(cs, ss, block, fmt))
            assert np.all(out == np.float32(want)), (fmt, block, want, out[:3])


def _bounds(ins, scales, out_dtype, tree_scales=None):
    """Per-element bound on |out - T| for T the FP64 sum of the inputs."""
    n = ins[0].size
    N = len(ins)
    xs = [widen(x).astype(np.float64) for x in ins]
    T = np.sum(xs, axis=0)
    A = np.sum([np.abs(x) for x in xs], axis=0)
    Eq = np.zeros(n)
    for x, s in zip(xs, scales):
        Eq += 2.0 ** -4 * np.abs(x) + 2.0 ** -10 * np.repeat(
            s.astype(np.float64), 128)[:n] * (1 + 2.0 ** -20)
    base = Eq + (N - 1) * 2.0 ** -24 * (A + Eq) * 1.0001
    u = 2.0 ** -8 if out_dtype == np.uint16 else 2.0 ** -24
    if tree_scales is not None:
        sp = np.repeat(tree_scales.astype(np.float64), 128)[:n]
        base = base + 2.0 ** -4 * (np.abs(T) + base) + 2.0 ** -10 * sp * (1 + 2.0 ** -20)
    return T, base + u * (np.abs(T) + base) + 1e-45


def pin_brute_force(oracle):
    seed = 100
    for N in (1, 2, 3, 8):
        for n in (1, 127, 128, 129, 200, 1000):
            for dt in (F32, BF16):
                seed += 1
                ins = W.random_inputs(N, n, dt, seed, scale_spread=3.0)
                outs, wc, ws = oracle.flat(ins)
                T, bound = _bounds(ins, ws, ins[0].dtype)
                for o in outs:
                    assert np.all(np.abs(widen(o).astype(np.float64) - T) <= bound), \
                        ("flat", N, n, dt)
                touts, twc, tws, sc, ss = oracle.tree(ins)
                T, bound = _bounds(ins, tws, ins[0].dtype, tree_scales=ss)
                for o in touts:
                    assert np.all(np.abs(widen(o).astype(np.float64) - T) <= bound), \
                        ("tree", N, n, dt)


def pin_outputs_identical(oracle):
    for dt in (F32, BF16):
        ins = W.random_inputs(3, 777, dt, 55, scale_spread=2.0)
        for fn in (oracle.flat, oracle.tree):
            outs = fn(ins)[0]
            for o in outs[1:]:
                assert same_bits(o, outs[0])


def pin_exact_tree_equals_flat(oracle):
    for dt in (F32, BF16):
        for N in (1, 3, 8):
            ins = W.random_inputs(N, 1031, dt, 70 + N)
            f = oracle.flat(ins, block=0)[0]
            t = oracle.tree(ins, block=0)[0]
            for a, b in zip(f, t):
                assert same_bits(a, b)


def _wire_sum(wc, ws, n):
    """The rank-ordered binary32 sum S of the dequantized wire payloads,
    from PyTorch's E4M3 decoding and numpy binary32 arithmetic (one rounded
    multiply per element, then one rounded add per rank)."""
    table = torch_e4m3_table()
    S = None
    for c, s in zip(wc, ws):
        v = (table[c] * np.repeat(s, 128)[:n]).astype(np.float32)
        S = v if S is None else (S + v).astype(np.float32)
    return S


def pin_tree_requant_grid(oracle):
    # The tree requantizes the binary32 sum S of the dequantized payloads
    # (for BF16 data too: the sum is cast to BF16 only at the output). Its
    # shard scale must be max|S|/448 (numpy IEEE division), its codes
    # PyTorch's encoding of S * (448/max|S|), and every output the cast of
    # PyTorch's decode of the shard code times the shard scale.
    for dt in (F32, BF16):
        ins = W.random_inputs(4, 128 * 9 + 50, dt, 91, scale_spread=2.0)
        n = ins[0].size
        outs, wc, ws, sc, ss = oracle.tree(ins)
        for r, x in enumerate(ins):  # the published payloads are each rank's own
            c, s = oracle.quantize(x)
            assert np.array_equal(wc[r], c) and same_bits(ws[r], s), (dt, r)
        S = _wire_sum(wc, ws, n)
        flat0 = oracle.flat(ins)[0][0]
        assert same_bits(flat0, S if dt == F32 else torch_bf16_bits(S)), dt
        for b in range(ss.size):
            blk = S[b * 128:(b + 1) * 128]
            a = np.float32(np.max(np.abs(blk)))
            assert ss[b] == a / np.float32(448.0), (dt, b)
            inv = np.float32(448.0) / a
            assert np.array_equal(sc[b * 128:(b + 1) * 128],
                                  torch_e4m3_encode((blk * inv).astype(np.float32))), (dt, b)
        grid = (torch_e4m3_table()[sc] * np.repeat(ss, 128)[:n]).astype(np.float32)
        want = grid if dt == F32 else torch_bf16_bits(grid)
        for o in outs:
            assert same_bits(o, want), dt
        assert np.count_nonzero(grid != S) > n // 2
        s = np.repeat(ss.astype(np.float64), 128)[:n]
        err = np.abs(grid.astype(np.float64) - S.astype(np.float64))
        assert np.all(err <= 2.0 ** -4 * np.abs(S) + 2.0 ** -10 * s * (1 + 2.0 ** -20))


def pin_torch_full_example(oracle):
    for N, rows, cols, want in read_torch_full_cases():
        ins32 = W.torch_full_example(N, (rows, cols))
        for ins in (ins32, [torch_bf16_bits(x) for x in ins32]):
            for fn in (oracle.flat, oracle.tree):
                outs = fn(ins, block=0)[0]
                for o in outs:
                    assert np.all(widen(o) == np.float32(want)), (N, fn.__name__)
            outs, wc, ws = oracle.flat(ins)
            T, bound = _bounds(ins, ws, ins[0].dtype)
            assert np.all(T == want)
            for r in range(N):
                assert np.all(wc[r] == (0x7E if r else 0x00)), r
                assert np.all(ws[r] == np.float32(r) / np.float32(448.0)), r
                assert np.all(np.abs(widen(outs[r]) - T) <= bound)
                assert same_bits(outs[r], outs[0])
            # Closed form of the low-precision results. Rank r's blocks hold
            # the constant r, so their scale is fl(r/448) and every code is
            # 448 (rank 0: a zero block, scale 0, code +0): rank r decodes to
            # v_r = fl(448 * fl(r/448)) and S is the rank-ordered binary32
            # sum of the v_r. Tree: S is constant in every block, so the
            # shard codes are 448 with scale fl(S/448) and every output is
            # the cast of fl(448 * fl(S/448)).
            f = np.float32
            S = f(0.0)
            for r in range(1, N):
                S = f(S + f(f(448.0) * f(f(r) / f(448.0))))

            def cast(v):
                full = np.full(rows * cols, v, dtype=np.float32)
                return torch_bf16_bits(full) if ins[0].dtype == np.uint16 else full
            for o in outs:
                assert same_bits(o, cast(S)), (N, "flat")
            touts, twc, tws, sc, ss = oracle.tree(ins)
            assert np.all(sc == (0x7E if S > 0 else 0x00)), (N, "tree codes")
            assert np.all(ss == f(S / f(448.0))), (N, "tree scales")
            for o in touts:
                assert same_bits(o, cast(f(f(448.0) * f(S / f(448.0))))), (N, "tree")


def pin_compression(oracle):
    n = 128 * 1000
    x = np.random.default_rng(4).standard_normal(n).astype(np.float32)
    for xin, ratio in ((x, 4.0), (torch_bf16_bits(x), 2.0)):
        codes, scales = oracle.quantize(xin)
        assert xin.nbytes / codes.nbytes == ratio
        assert math.isclose(xin.nbytes / (codes.nbytes + scales.nbytes),
                            ratio / (1 + 4 / 128), rel_tol=1e-12)


def pin_shard_len(oracle):
    cases = [(200, 8, 128, 128), (33554432, 8, 128, 4194304),
             (67108864, 8, 128, 8388608), (1000, 3, 128, 384), (1, 8, 128, 128),
             (10, 3, 0, 4), (1024, 8, 128, 128)]
    for n, N, block, want in cases:
        assert oracle.shard_len(n, N, block) == want, (n, N, block)


# -- ReduceScatter, AllGather, AlltoAll -------------------------------------

def _representable(n, seed, dt, j=0):
    """n elements that are E4M3 values times 2^j, with 448 * 2^j in every
    128-block (so every block's scale is exactly 2^j and the payload round
    trip is exact)."""
    g = np.random.default_rng(seed)
    table = torch_e4m3_table()
    valid = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    x = (table[g.choice(valid, size=n)] * np.float32(2.0 ** j)).astype(np.float32)
    x[::128] = np.float32(448.0 * 2.0 ** j)
    return torch_bf16_bits(x) if dt == BF16 else x


def pin_reduce_scatter(oracle):
    for dt in (F32, BF16):
        for N, n in ((1, 300), (3, 1000), (8, 129), (5, 128 * 40 + 1)):
            ins = W.random_inputs(N, n, dt, 300 + N + n, scale_spread=3.0)
            outs, wc, ws = oracle.reduce_scatter(ins)
            per = oracle.shard_len(n, N)
            T, bound = _bounds(ins, ws, ins[0].dtype)
            for r in range(N):
                lo, hi = r * per, min(n, (r + 1) * per)
                assert outs[r].size == max(0, hi - lo)
                if hi > lo:
                    err = np.abs(widen(outs[r]).astype(np.float64) - T[lo:hi])
                    assert np.all(err <= bound[lo:hi]), (N, n, r)
            flat = oracle.flat(ins)[0][0]
            for r in range(N):
                lo = r * per
                assert same_bits(outs[r], flat[lo:lo + outs[r].size])
            if N == 1:
                c, s = oracle.quantize(ins[0])
                assert same_bits(outs[0], oracle.dequantize(c, s, dtype=ins[0].dtype))
    for N, rows, cols, want in read_torch_full_cases():
        ins = W.torch_full_example(N, (rows, cols))
        outs = oracle.reduce_scatter(ins, block=0)[0]
        assert sum(o.size for o in outs) == rows * cols
        assert all(np.all(o == np.float32(want)) for o in outs)


def pin_all_gather(oracle):
    for dt in (F32, BF16):
        for N, m in ((1, 200), (3, 128), (4, 300), (8, 77)):
            # exactly representable contributions come back unchanged
            ins = [_representable(m, 400 + r, dt, j=3 * r - 4) for r in range(N)]
            outs, wc, ws = oracle.all_gather(ins)
            cat = np.concatenate(ins)
            for o in outs:
                assert same_bits(o, cat), (N, m)
            assert all(same_bits(o, cat) for o in oracle.all_gather(ins, block=0)[0])
            # general contributions: each segment within the quantization bound
            ins = W.random_inputs(N, m, dt, 500 + N, scale_spread=3.0)
            outs, wc, ws = oracle.all_gather(ins)
            for r in range(N):
                seg = outs[0][r * m:(r + 1) * m]
                x = widen(ins[r]).astype(np.float64)
                T, bound = _bounds([ins[r]], [ws[r]], ins[0].dtype)
                assert np.all(np.abs(widen(seg).astype(np.float64) - x) <= bound)
            for o in outs[1:]:
                assert same_bits(o, outs[0])


def pin_all_to_all(oracle):
    for dt in (F32, BF16):
        for N, c in ((1, 256), (2, 200), (4, 128), (3, 130)):
            ins = [np.concatenate([_representable(c, 600 + 10 * r + j, dt, j=r - j)
                                   for j in range(N)]) for r in range(N)]
            for block in (128, 0):
                outs = oracle.all_to_all(ins, block=block)[0]
                for j in range(N):
                    for r in range(N):
                        assert same_bits(outs[j][r * c:(r + 1) * c],
                                         ins[r][j * c:(j + 1) * c]), (N, c, j, r, block)
        # blocks restart at every chunk: chunk j's first scale is the largest
        # magnitude of its own first (up to) 128 elements over 448
        N, c = 3, 200
        ins = W.random_inputs(N, N * c, dt, 700, scale_spread=3.0)
        outs, wc, ws = oracle.all_to_all(ins)
        nbc = (c + 127) // 128
        for r in range(N):
            x = widen(ins[r])
            for j in range(N):
                first = x[j * c:j * c + 128]
                tail = x[j * c + 128:(j + 1) * c]
                assert ws[r][j * nbc] == np.float32(np.max(np.abs(first))) / np.float32(448.0)
                assert ws[r][j * nbc + 1] == np.float32(np.max(np.abs(tail))) / np.float32(448.0)
                T, bound = _bounds([ins[r][j * c:(j + 1) * c]], [ws[r][j * nbc:(j + 1) * nbc]],
                                   ins[0].dtype)
                got = widen(outs[j][r * c:(r + 1) * c]).astype(np.float64)
                assert np.all(np.abs(got - T) <= bound)


# -- format and block-size variants (E5M2; blocks of 32, 64, 128, 256) --------

E4M3, E5M2 = 0, 1
FP8_MAX = {E4M3: 448.0, E5M2: 57344.0}
VARIANT_BLOCKS = (32, 64, 128, 256)


def torch_e5m2_table():
    return (torch.arange(256, dtype=torch.uint8).view(torch.float8_e5m2)
            .float().numpy())


def torch_e5m2_encode(y):
    """PyTorch's RNE float32 -> e5m2 (valid for |y| <= 57344)."""
    t = torch.from_numpy(np.ascontiguousarray(y, dtype=np.float32))
    return t.to(torch.float8_e5m2).view(torch.uint8).numpy()


def pin_e5m2_decode(oracle):
    ours = oracle.e5m2_decode_all()
    ref = torch_e5m2_table()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert same_bits(ours[~nan], ref[~nan])
    # spec points: max finite 1.75 * 2^15, min normal 2^-14, min subnormal
    # 2^-16, +-Inf at S.11111.00
    assert ours[0x7B] == 57344.0 and ours[0x04] == 2.0 ** -14
    assert ours[0x01] == 2.0 ** -16 and ours[0x7C] == np.inf and ours[0xFC] == -np.inf
    pos = ours[:0x7C].astype(np.float64)
    gaps = np.diff(pos)
    assert np.all(gaps > 0)
    spacing = [gaps[g * 4] for g in range(31)]
    assert spacing[0] == spacing[1]
    for g in range(2, 31):
        assert spacing[g] == 2 * spacing[g - 1], g


def pin_e5m2_encode(oracle):
    table = torch_e5m2_table()
    for c in range(256):
        if np.isfinite(table[c]):
            assert oracle.e5m2_encode(table[c]) == c, hex(c)
    pos = table[:0x7C].astype(np.float64)
    for c in range(0x7A):
        mid = (pos[c] + pos[c + 1]) / 2
        assert float(np.float32(mid)) == mid
        even = c if c % 2 == 0 else c + 1
        for sgn, mask in ((1.0, 0x00), (-1.0, 0x80)):
            m = np.float32(sgn * mid)
            assert oracle.e5m2_encode(m) == (even | mask), (c, sgn)
            assert oracle.e5m2_encode(nextafter32(m, sgn * np.inf)) == ((c + 1) | mask)
            assert oracle.e5m2_encode(nextafter32(m, 0.0)) == (c | mask)
    g = np.random.default_rng(4321)
    mag = np.exp2(g.uniform(-20, math.log2(57344), 20000)).astype(np.float32)
    y = np.concatenate([mag, -mag])
    y = y[np.abs(y) <= 57344]
    assert np.array_equal(oracle.e5m2_encode_array(y), torch_e5m2_encode(y))
    for v in (57344.0, 57345.0, 61439.0, 61440.0, 1e30, math.inf):
        assert oracle.e5m2_encode(v) == 0x7B and oracle.e5m2_encode(-v) == 0xFB, v
    assert oracle.e5m2_encode(math.nan) == 0x7F
    for v, code in ((2.0 ** -17, 0x00), (float(nextafter32(2.0 ** -17, 1)), 0x01),
                    (3 * 2.0 ** -17, 0x02), (-0.0, 0x80), (-1e-30, 0x80)):
        assert oracle.e5m2_encode(v) == code, v


def pin_variant_scale_and_tail(oracle):
    g = np.random.default_rng(17)
    for fmt in (E4M3, E5M2):
        for a in np.exp2(g.uniform(-60, 60, 300)).astype(np.float32):
            s, inv = oracle.block_scale_fmt(a, fmt)
            assert s == a / np.float32(FP8_MAX[fmt])
            assert inv == np.float32(FP8_MAX[fmt]) / a
        for block in VARIANT_BLOCKS:
            n = 3 * block + block // 2 + 3
            x = g.standard_normal(n).astype(np.float32)
            codes, scales = oracle.quantize_fmt(x, block, fmt)
            assert scales.size == -(-n // block)
            for b in range(scales.size):
                blk = x[b * block:(b + 1) * block]
                assert scales[b] == np.float32(np.max(np.abs(blk))) / np.float32(FP8_MAX[fmt])
                one_c, one_s = oracle.quantize_fmt(blk, block, fmt)
                assert np.array_equal(codes[b * block:(b + 1) * block], one_c)
    # the E4M3 / 128 variant is the main path
    x = W.random_inputs(1, 1000, BF16, 3, scale_spread=2.0)[0]
    c1, s1 = oracle.quantize(x)
    c2, s2 = oracle.quantize_fmt(x, 128, E4M3)
    assert np.array_equal(c1, c2) and same_bits(s1, s2)


def pin_variant_roundtrip_and_bound(oracle):
    g = np.random.default_rng(23)
    tables = {E4M3: torch_e4m3_table(), E5M2: torch_e5m2_table()}
    for fmt in (E4M3, E5M2):
        table = tables[fmt]
        finite = np.array([c for c in range(256) if np.isfinite(table[c])], dtype=np.uint8)
        top = 0x7E if fmt == E4M3 else 0x7B
        for block in VARIANT_BLOCKS:
            for j in (-12, 0, 9):
                codes = g.choice(finite, size=block * 3)
                codes[::block] = top
                x = (table[codes] * np.float32(2.0 ** j)).astype(np.float32)
                qc, qs = oracle.quantize_fmt(x, block, fmt)
                assert np.array_equal(qc, codes) and np.all(qs == np.float32(2.0 ** j))
                assert same_bits(oracle.dequantize_fmt(qc, qs, block, fmt), x)
            # error bound: 2^-(m+1) relative for normals (m mantissa bits),
            # half a subnormal step times s below the normal range
            x = W.random_inputs(1, block * 20 + 7, F32, block + fmt, scale_spread=4.0)[0]
            qc, qs = oracle.quantize_fmt(x, block, fmt)
            back = oracle.dequantize_fmt(qc, qs, block, fmt).astype(np.float64)
            s = np.repeat(qs.astype(np.float64), block)[:x.size]
            x64 = x.astype(np.float64)
            y = np.where(s > 0, np.abs(x64) / np.where(s > 0, s, 1), 0)
            rel = 2.0 ** -4 if fmt == E4M3 else 2.0 ** -3
            min_normal = 2.0 ** -6 if fmt == E4M3 else 2.0 ** -14
            half_sub = 2.0 ** -10 if fmt == E4M3 else 2.0 ** -17
            err = np.abs(back - x64)
            normal = y >= min_normal
            assert np.all(err[normal] <= rel * np.abs(x64[normal]))
            assert np.all(err[~normal] <= half_sub * s[~normal] * (1 + 2.0 ** -20) +
                          2.0 ** -22 * np.abs(x64[~normal]))


def pin_variant_reduce(oracle):
    for fmt in (E4M3, E5M2):
        for block in VARIANT_BLOCKS:
            ins = W.random_inputs(4, block * 6 + 5, F32, 40 + block + fmt, scale_spread=3.0)
            pays = [oracle.quantize_fmt(x, block, fmt) for x in ins]
            out = oracle.reduce_fmt([c for c, _ in pays], [s for _, s in pays], block, fmt)
            T = np.sum([x.astype(np.float64) for x in ins], axis=0)
            # each dequantized value sums exactly as the dequantized payloads
            v = [oracle.dequantize_fmt(c, s, block, fmt).astype(np.float64) for c, s in pays]
            rel = 2.0 ** -4 if fmt == E4M3 else 2.0 ** -3
            half_sub = 2.0 ** -10 if fmt == E4M3 else 2.0 ** -17
            bound = np.zeros(T.size)
            for x, (c, s) in zip(ins, pays):
                bound += rel * np.abs(x) + half_sub * np.repeat(s.astype(np.float64),
                                                                block)[:x.size] * 1.000001
            bound += 3 * 2.0 ** -24 * np.sum(np.abs(v), axis=0) * 1.0001 + 1e-45
            assert np.all(np.abs(out.astype(np.float64) - T) <= bound), (fmt, block)


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
