"""Python handle on the CPU oracle (``lpcoll_oracle.c``).

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the library and its
binding never do. The functions below marshal numpy arrays into the C oracle
and back; all arithmetic happens in C.

Arrays: FP32 data is ``numpy.float32``; BF16 data is carried as its raw bits
in ``numpy.uint16``. Codes are ``numpy.uint8``, scales ``numpy.float32``.
"""
import contextlib
import ctypes

import numpy as np

from . import build as _build

F32 = 0
BF16 = 1
BLOCK = 128
E4M3 = 0
E5M2 = 1

_lib = None


def _load(path):
    L = ctypes.CDLL(path)
    c_sz = ctypes.c_size_t
    vp = ctypes.c_void_p
    pp = ctypes.POINTER(ctypes.c_void_p)
    L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
    L.orc_e4m3_decode.restype = ctypes.c_float
    L.orc_e4m3_encode.argtypes = [ctypes.c_float]
    L.orc_e4m3_encode.restype = ctypes.c_uint8
    L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
    L.orc_bf16_to_f32.restype = ctypes.c_float
    L.orc_f32_to_bf16.argtypes = [ctypes.c_float]
    L.orc_f32_to_bf16.restype = ctypes.c_uint16
    L.orc_block_scale.argtypes = [ctypes.c_float,
                                  ctypes.POINTER(ctypes.c_float),
                                  ctypes.POINTER(ctypes.c_float)]
    L.orc_block_scale.restype = None
    L.orc_quantize.argtypes = [vp, ctypes.c_int, c_sz, ctypes.c_int, vp, vp]
    L.orc_dequantize.argtypes = [vp, vp, c_sz, ctypes.c_int, vp, ctypes.c_int]
    L.orc_reduce.argtypes = [pp, pp, ctypes.c_int, c_sz, ctypes.c_int, vp,
                             ctypes.c_int]
    L.orc_flat.argtypes = [pp, pp, ctypes.c_int, c_sz, ctypes.c_int,
                           ctypes.c_int, pp, pp]
    L.orc_tree.argtypes = [pp, pp, ctypes.c_int, c_sz, ctypes.c_int,
                           ctypes.c_int, pp, pp, vp, vp]
    for f in ("orc_reduce_scatter", "orc_all_gather", "orc_all_to_all"):
        getattr(L, f).argtypes = [pp, pp, ctypes.c_int, c_sz, ctypes.c_int,
                                  ctypes.c_int, pp, pp]
        getattr(L, f).restype = ctypes.c_int
    L.orc_e5m2_decode.argtypes = [ctypes.c_uint8]
    L.orc_e5m2_decode.restype = ctypes.c_float
    L.orc_e5m2_encode.argtypes = [ctypes.c_float]
    L.orc_e5m2_encode.restype = ctypes.c_uint8
    L.orc_block_scale_fmt.argtypes = [ctypes.c_float, ctypes.c_int,
                                      ctypes.POINTER(ctypes.c_float),
                                      ctypes.POINTER(ctypes.c_float)]
    L.orc_block_scale_fmt.restype = None
    L.orc_quantize_fmt.argtypes = [vp, ctypes.c_int, c_sz, ctypes.c_int,
                                   ctypes.c_int, vp, vp]
    L.orc_dequantize_fmt.argtypes = [vp, vp, c_sz, ctypes.c_int, ctypes.c_int,
                                     vp, ctypes.c_int]
    L.orc_reduce_fmt.argtypes = [pp, pp, ctypes.c_int, c_sz, ctypes.c_int,
                                 ctypes.c_int, vp, ctypes.c_int]
    for f in ("orc_quantize_fmt", "orc_dequantize_fmt", "orc_reduce_fmt"):
        getattr(L, f).restype = ctypes.c_int
    L.orc_set_divide_reading.argtypes = [ctypes.c_int]
    L.orc_set_divide_reading.restype = None
    L.orc_shard_len.argtypes = [c_sz, ctypes.c_int, ctypes.c_int]
    L.orc_shard_len.restype = c_sz
    for f in ("orc_quantize", "orc_dequantize", "orc_reduce", "orc_flat",
              "orc_tree"):
        getattr(L, f).restype = ctypes.c_int
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = _load(_build.build())
    return _lib


@contextlib.contextmanager
def using(path):
    """Route every function of this module through another build of the
    oracle (the tests use this to check that planted mistakes are caught)."""
    global _lib
    saved = _lib
    _lib = _load(path)
    try:
        yield
    finally:
        _lib = saved


@contextlib.contextmanager
def divide_reading():
    """Inside the block, quantize elements as fp8(x / s) (one division per
    element) instead of fp8(x * (448 / a)): the other reading of the scale
    step, for comparing the two readings only."""
    L = lib()
    L.orc_set_divide_reading(1)
    try:
        yield
    finally:
        L.orc_set_divide_reading(0)


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else ctypes.c_void_p(0)


def _ptrs(arrs):
    return (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])


def _dtype_code(a):
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError("oracle data must be float32 or uint16 (bf16 bits), got %s"
                    % a.dtype)


def _check(status, what):
    if status != 0:
        raise ValueError("oracle %s returned status %d" % (what, status))


def nblocks(n, block=BLOCK):
    return (n + block - 1) // block


# -- scalar codecs ---------------------------------------------------------

def e4m3_decode(code):
    return lib().orc_e4m3_decode(int(code))


def e4m3_encode(y):
    return lib().orc_e4m3_encode(float(y))


def e4m3_decode_all():
    """Values of all 256 codes as float32 (index = code)."""
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float32)


def e4m3_encode_array(y):
    y = np.ascontiguousarray(y, dtype=np.float32).ravel()
    L = lib()
    return np.fromiter((L.orc_e4m3_encode(float(v)) for v in y), dtype=np.uint8,
                       count=y.size)


def bf16_to_f32(h):
    return lib().orc_bf16_to_f32(int(h))


def f32_to_bf16(f):
    return lib().orc_f32_to_bf16(float(f))


def f32_to_bf16_array(x):
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    L = lib()
    return np.fromiter((L.orc_f32_to_bf16(float(v)) for v in x), dtype=np.uint16,
                       count=x.size)


def block_scale(amax):
    s = ctypes.c_float()
    inv = ctypes.c_float()
    lib().orc_block_scale(float(amax), ctypes.byref(s), ctypes.byref(inv))
    return np.float32(s.value), np.float32(inv.value)


# -- array operations --------------------------------------------------------

def quantize(x, block=BLOCK):
    """One rank's payload: (codes uint8[n], scales float32[ceil(n/block)])."""
    x = np.ascontiguousarray(x)
    n = x.size
    codes = np.zeros(n, dtype=np.uint8)
    scales = np.zeros(max(nblocks(n, block), 1), dtype=np.float32)
    _check(lib().orc_quantize(_ptr(x), _dtype_code(x), n, block, _ptr(codes),
                              _ptr(scales)), "quantize")
    return codes, scales[:nblocks(n, block)]


def dequantize(codes, scales, dtype=np.float32, block=BLOCK):
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    out = np.zeros(codes.size, dtype=dtype)
    _check(lib().orc_dequantize(_ptr(codes), _ptr(scales), codes.size, block,
                                _ptr(out), _dtype_code(out)), "dequantize")
    return out


def reduce(codes_list, scales_list, dtype=np.float32, block=BLOCK):
    codes_list = [np.ascontiguousarray(c, dtype=np.uint8) for c in codes_list]
    scales_list = [np.ascontiguousarray(s, dtype=np.float32) for s in scales_list]
    n = codes_list[0].size
    out = np.zeros(n, dtype=dtype)
    _check(lib().orc_reduce(_ptrs(codes_list), _ptrs(scales_list),
                            len(codes_list), n, block, _ptr(out),
                            _dtype_code(out)), "reduce")
    return out


def _wires(nranks, n, block):
    if block == 0:
        return None, None
    codes = [np.zeros(max(n, 1), dtype=np.uint8) for _ in range(nranks)]
    scales = [np.zeros(max(nblocks(n, block), 1), dtype=np.float32)
              for _ in range(nranks)]
    return codes, scales


def flat(inputs, block=BLOCK):
    """DDA flat allreduce. Returns (outputs, wire_codes, wire_scales)."""
    inputs = [np.ascontiguousarray(x) for x in inputs]
    nranks = len(inputs)
    n = inputs[0].size
    outs = [np.zeros(n, dtype=inputs[0].dtype) for _ in range(nranks)]
    wc, ws = _wires(nranks, n, block)
    null = (ctypes.c_void_p * nranks)()
    _check(lib().orc_flat(_ptrs(inputs), _ptrs(outs), nranks, n,
                          _dtype_code(inputs[0]), block,
                          _ptrs(wc) if wc else null, _ptrs(ws) if ws else null),
           "flat")
    if wc is not None:
        wc = [c[:n] for c in wc]
        ws = [s[:nblocks(n, block)] for s in ws]
    return outs, wc, ws


def tree(inputs, block=BLOCK):
    """DDA tree allreduce. Returns (outputs, wire_codes, wire_scales,
    shard_codes, shard_scales)."""
    inputs = [np.ascontiguousarray(x) for x in inputs]
    nranks = len(inputs)
    n = inputs[0].size
    outs = [np.zeros(n, dtype=inputs[0].dtype) for _ in range(nranks)]
    wc, ws = _wires(nranks, n, block)
    null = (ctypes.c_void_p * nranks)()
    if block:
        sc = np.zeros(max(n, 1), dtype=np.uint8)
        ss = np.zeros(max(nblocks(n, block), 1), dtype=np.float32)
    else:
        sc = ss = None
    _check(lib().orc_tree(_ptrs(inputs), _ptrs(outs), nranks, n,
                          _dtype_code(inputs[0]), block,
                          _ptrs(wc) if wc else null, _ptrs(ws) if ws else null,
                          _ptr(sc), _ptr(ss)), "tree")
    if wc is not None:
        wc = [c[:n] for c in wc]
        ws = [s[:nblocks(n, block)] for s in ws]
        sc = sc[:n]
        ss = ss[:nblocks(n, block)]
    return outs, wc, ws, sc, ss


def reduce_scatter(inputs, block=BLOCK):
    """LP ReduceScatter. Returns (outputs, wire_codes, wire_scales); output r
    holds shard r (length min(L, n - r L), L = shard_len(n, N, block))."""
    inputs = [np.ascontiguousarray(x) for x in inputs]
    nranks = len(inputs)
    n = inputs[0].size
    per = shard_len(n, nranks, block) if n else 0
    lens = [max(0, min(per, n - r * per)) for r in range(nranks)]
    outs = [np.zeros(max(k, 1), dtype=inputs[0].dtype) for k in lens]
    wc, ws = _wires(nranks, n, block)
    null = (ctypes.c_void_p * nranks)()
    _check(lib().orc_reduce_scatter(_ptrs(inputs), _ptrs(outs), nranks, n,
                                    _dtype_code(inputs[0]), block,
                                    _ptrs(wc) if wc else null,
                                    _ptrs(ws) if ws else null), "reduce_scatter")
    outs = [o[:k] for o, k in zip(outs, lens)]
    if wc is not None:
        wc = [c[:n] for c in wc]
        ws = [s[:nblocks(n, block)] for s in ws]
    return outs, wc, ws


def all_gather(inputs, block=BLOCK):
    """LP AllGather of N contributions of m elements. Returns (outputs of
    N*m elements, wire_codes, wire_scales)."""
    inputs = [np.ascontiguousarray(x) for x in inputs]
    nranks = len(inputs)
    m = inputs[0].size
    outs = [np.zeros(max(nranks * m, 1), dtype=inputs[0].dtype) for _ in range(nranks)]
    wc, ws = _wires(nranks, m, block)
    null = (ctypes.c_void_p * nranks)()
    _check(lib().orc_all_gather(_ptrs(inputs), _ptrs(outs), nranks, m,
                                _dtype_code(inputs[0]), block,
                                _ptrs(wc) if wc else null,
                                _ptrs(ws) if ws else null), "all_gather")
    outs = [o[:nranks * m] for o in outs]
    if wc is not None:
        wc = [c[:m] for c in wc]
        ws = [s[:nblocks(m, block)] for s in ws]
    return outs, wc, ws


def all_to_all(inputs, block=BLOCK):
    """LP AlltoAll: input r is N chunks of c = size/N elements. Returns
    (outputs, wire_codes (N*c bytes each), wire_scales (N*ceil(c/128)))."""
    inputs = [np.ascontiguousarray(x) for x in inputs]
    nranks = len(inputs)
    if inputs[0].size % nranks:
        raise ValueError("all_to_all input length must be a multiple of N")
    c = inputs[0].size // nranks
    outs = [np.zeros(max(nranks * c, 1), dtype=inputs[0].dtype) for _ in range(nranks)]
    if block:
        nbc = nblocks(c, block)
        wc = [np.zeros(max(nranks * c, 1), dtype=np.uint8) for _ in range(nranks)]
        ws = [np.zeros(max(nranks * nbc, 1), dtype=np.float32) for _ in range(nranks)]
    else:
        wc = ws = None
    null = (ctypes.c_void_p * nranks)()
    _check(lib().orc_all_to_all(_ptrs(inputs), _ptrs(outs), nranks, c,
                                _dtype_code(inputs[0]), block,
                                _ptrs(wc) if wc else null,
                                _ptrs(ws) if ws else null), "all_to_all")
    outs = [o[:nranks * c] for o in outs]
    if wc is not None:
        wc = [x[:nranks * c] for x in wc]
        ws = [x[:nranks * nblocks(c, block)] for x in ws]
    return outs, wc, ws


# -- format / block-size variants ---------------------------------------------

def e5m2_decode(code):
    return lib().orc_e5m2_decode(int(code))


def e5m2_encode(y):
    return lib().orc_e5m2_encode(float(y))


def e5m2_decode_all():
    return np.array([e5m2_decode(c) for c in range(256)], dtype=np.float32)


def e5m2_encode_array(y):
    y = np.ascontiguousarray(y, dtype=np.float32).ravel()
    L = lib()
    return np.fromiter((L.orc_e5m2_encode(float(v)) for v in y), dtype=np.uint8,
                       count=y.size)


def block_scale_fmt(amax, fmt):
    s = ctypes.c_float()
    inv = ctypes.c_float()
    lib().orc_block_scale_fmt(float(amax), int(fmt), ctypes.byref(s), ctypes.byref(inv))
    return np.float32(s.value), np.float32(inv.value)


def quantize_fmt(x, block, fmt):
    x = np.ascontiguousarray(x)
    n = x.size
    codes = np.zeros(max(n, 1), dtype=np.uint8)
    scales = np.zeros(max(nblocks(n, block), 1), dtype=np.float32)
    _check(lib().orc_quantize_fmt(_ptr(x), _dtype_code(x), n, block, fmt, _ptr(codes),
                                  _ptr(scales)), "quantize_fmt")
    return codes[:n], scales[:nblocks(n, block)]


def dequantize_fmt(codes, scales, block, fmt, dtype=np.float32):
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    out = np.zeros(max(codes.size, 1), dtype=dtype)
    _check(lib().orc_dequantize_fmt(_ptr(codes), _ptr(scales), codes.size, block, fmt,
                                    _ptr(out), _dtype_code(out)), "dequantize_fmt")
    return out[:codes.size]


def reduce_fmt(codes_list, scales_list, block, fmt, dtype=np.float32):
    codes_list = [np.ascontiguousarray(c, dtype=np.uint8) for c in codes_list]
    scales_list = [np.ascontiguousarray(s, dtype=np.float32) for s in scales_list]
    n = codes_list[0].size
    out = np.zeros(max(n, 1), dtype=dtype)
    _check(lib().orc_reduce_fmt(_ptrs(codes_list), _ptrs(scales_list), len(codes_list),
                                n, block, fmt, _ptr(out), _dtype_code(out)), "reduce_fmt")
    return out[:n]


def shard_len(n, nranks, block=BLOCK):
    return lib().orc_shard_len(n, nranks, block)


def as_f32(a):
    """Widen oracle-format data (float32, or bf16 bits in uint16) to float32."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32)
    return a.astype(np.float32, copy=False)


