"""ctypes binding of liblpcoll.so, one Python function per C entry point.

Argument marshalling only: each function checks that the torch tensors it is
given are CUDA, contiguous, of the right dtype and large enough, then passes
their device pointers, the element count and the CUDA stream to the C call
of the same name, and raises ``LpcollError`` on a non-zero status. All the
arithmetic runs in the library's kernels. There is no fallback: if the
library is missing, every call raises.
"""
import contextlib
import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "liblpcoll.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "lpcoll.h")

F32 = 0
BF16 = 1
BLOCK = 128
E4M3 = 0
E5M2 = 1
VARIANT_BLOCKS = (32, 64, 128, 256)
MAX_RANKS = 16

STATUS = {0: "LPCOLL_OK", 1: "LPCOLL_ERR_ARG", 2: "LPCOLL_ERR_ALIGN",
          3: "LPCOLL_ERR_UNSUPPORTED", 4: "LPCOLL_ERR_RANK", 5: "LPCOLL_ERR_CUDA"}

_lib = None


class LpcollError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__("%s: %s" % (what, status_string(status)))


def lib():
    """The loaded liblpcoll.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "liblpcoll.so not found at %s; build it with "
                "precision_collective_reduction_gb300.build.build()" % LIB_PATH)
        _lib = _load(LIB_PATH)
    return _lib


@contextlib.contextmanager
def using_library(path):
    """Route every call of this module through another build of the library
    inside the block (the tests use the bounds-checked build this way)."""
    global _lib
    saved = _lib
    _lib = _load(path)
    try:
        yield _lib
    finally:
        _lib = saved


def _load(path):
    """Load one build of the library and declare its C signatures."""
    L = ctypes.CDLL(path)
    vp, sz, ci = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    pp = ctypes.POINTER(ctypes.c_void_p)
    L.lp_quantize.argtypes = [vp, ci, sz, ci, vp, vp, vp]
    L.lp_dequantize.argtypes = [vp, vp, sz, ci, vp, ci, vp]
    L.lp_reduce.argtypes = [pp, pp, ci, sz, ci, vp, ci, vp]
    L.dda_flat_sim.argtypes = [pp, pp, ci, sz, ci, ci, pp, pp, vp]
    L.dda_tree_sim.argtypes = [pp, pp, ci, sz, ci, ci, pp, pp, vp, vp, vp]
    for f in ("reduce_scatter_sim", "all_gather_sim", "all_to_all_sim"):
        getattr(L, f).argtypes = [pp, pp, ci, sz, ci, ci, pp, pp, vp]
    L.dda_flat_sim_noalloc.argtypes = [pp, pp, ci, sz, ci, vp]
    L.lp_quantize_fmt.argtypes = [vp, ci, sz, ci, ci, vp, vp, vp]
    L.lp_dequantize_fmt.argtypes = [vp, vp, sz, ci, ci, vp, ci, vp]
    L.lp_reduce_fmt.argtypes = [pp, pp, ci, sz, ci, ci, vp, ci, vp]
    L.lpcoll_host_workspace_bytes.argtypes = [ci, sz, ci, ci, ci, ci, ci]
    L.lpcoll_host_workspace_bytes.restype = sz
    L.lpcoll_host_allreduce.argtypes = [pp, pp, pp, ci, sz, ci, ci, sz, ci, vp, sz,
                                        vp, vp, vp]
    L.lpcoll_host_allreduce.restype = ci
    L.lpcoll_debug_fail_host_enqueue.argtypes = [ctypes.c_long]
    L.lpcoll_debug_fail_host_enqueue.restype = None
    for f in ("lp_quantize", "lp_dequantize", "lp_reduce", "dda_flat_sim",
              "dda_tree_sim", "reduce_scatter_sim", "all_gather_sim",
              "all_to_all_sim", "dda_flat_sim_noalloc", "lp_quantize_fmt",
              "lp_dequantize_fmt", "lp_reduce_fmt",
              "lpcoll_last_cuda_error", "lpcoll_version"):
        getattr(L, f).restype = ci
    L.lpcoll_status_string.argtypes = [ci]
    L.lpcoll_status_string.restype = ctypes.c_char_p
    L.lpcoll_debug_bounds_errors.argtypes = [ctypes.POINTER(ctypes.c_ulonglong)]
    L.lpcoll_debug_bounds_errors.restype = ci
    L.lpcoll_debug_bounds_shrink.argtypes = [sz]
    L.lpcoll_debug_bounds_shrink.restype = None
    return L


def debug_bounds_errors():
    """(status, first bad address) of the bounds-checked build: status 1 if
    a kernel access since the last call fell outside the buffers its call
    passed, 0 if none, -1 for the normal build. Synchronizes the device."""
    bad = ctypes.c_ulonglong(0)
    st = lib().lpcoll_debug_bounds_errors(ctypes.byref(bad))
    return st, bad.value


def status_string(status):
    s = lib().lpcoll_status_string(int(status)).decode()
    if status == 5:
        s += " (cudaError %d)" % lib().lpcoll_last_cuda_error()
    return s


def ptr_array(ptrs):
    """Host array of device pointers (ints) for a per-rank argument."""
    ptrs = list(ptrs)
    return (ctypes.c_void_p * max(len(ptrs), 1))(*ptrs)


def _rank_ptrs(ptrs, nranks, what, needed=True):
    """ptr_array of a per-rank argument, which the C call reads nranks
    entries of; an argument the call does not read (the wires of an exact
    call) may be shorter."""
    ptrs = list(ptrs) if ptrs is not None else []
    if needed and len(ptrs) < nranks:
        raise ValueError("%s lists %d pointers for %d ranks" % (what, len(ptrs), nranks))
    return ptr_array(ptrs)


def _check(st, what):
    if st != 0:
        raise LpcollError(st, what)


# -- raw calls: device pointers as ints ------------------------------------

def raw_lp_quantize(in_ptr, dtype, n, block, codes_ptr, scales_ptr, stream):
    _check(lib().lp_quantize(in_ptr, dtype, n, block, codes_ptr, scales_ptr, stream),
           "lp_quantize")


def raw_lp_dequantize(codes_ptr, scales_ptr, n, block, out_ptr, dtype, stream):
    _check(lib().lp_dequantize(codes_ptr, scales_ptr, n, block, out_ptr, dtype, stream),
           "lp_dequantize")


def raw_lp_reduce(codes_ptrs, scales_ptrs, nranks, n, block, out_ptr, dtype, stream):
    _check(lib().lp_reduce(_rank_ptrs(codes_ptrs, nranks, "codes"),
                           _rank_ptrs(scales_ptrs, nranks, "scales"), nranks, n, block,
                           out_ptr, dtype, stream), "lp_reduce")


def raw_dda_flat_sim(in_ptrs, out_ptrs, nranks, n, dtype, block, wc_ptrs, ws_ptrs,
                     stream):
    _check(lib().dda_flat_sim(_rank_ptrs(in_ptrs, nranks, "in"),
                              _rank_ptrs(out_ptrs, nranks, "out"), nranks, n, dtype, block,
                              _rank_ptrs(wc_ptrs, nranks, "wire_codes", block != 0),
                              _rank_ptrs(ws_ptrs, nranks, "wire_scales", block != 0),
                              stream), "dda_flat_sim")


def raw_dda_tree_sim(in_ptrs, out_ptrs, nranks, n, dtype, block, wc_ptrs, ws_ptrs,
                     sc_ptr, ss_ptr, stream):
    _check(lib().dda_tree_sim(_rank_ptrs(in_ptrs, nranks, "in"),
                              _rank_ptrs(out_ptrs, nranks, "out"), nranks, n, dtype, block,
                              _rank_ptrs(wc_ptrs, nranks, "wire_codes", block != 0),
                              _rank_ptrs(ws_ptrs, nranks, "wire_scales", block != 0),
                              sc_ptr, ss_ptr, stream), "dda_tree_sim")


def raw_collective(name, in_ptrs, out_ptrs, nranks, count, dtype, block, wc_ptrs,
                   ws_ptrs, stream):
    """reduce_scatter_sim / all_gather_sim / all_to_all_sim by name."""
    _check(getattr(lib(), name)(_rank_ptrs(in_ptrs, nranks, "in"),
                                _rank_ptrs(out_ptrs, nranks, "out"), nranks, count, dtype,
                                block, _rank_ptrs(wc_ptrs, nranks, "wire_codes", block != 0),
                                _rank_ptrs(ws_ptrs, nranks, "wire_scales", block != 0),
                                stream), name)


def raw_dda_flat_sim_noalloc(in_ptrs, out_ptrs, nranks, n, dtype, stream):
    _check(lib().dda_flat_sim_noalloc(_rank_ptrs(in_ptrs, nranks, "in"),
                                      _rank_ptrs(out_ptrs, nranks, "out"), nranks, n, dtype,
                                      stream), "dda_flat_sim_noalloc")


# -- torch-tensor calls -----------------------------------------------------

def _torch():
    import torch
    return torch


def dtype_code(t):
    torch = _torch()
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError("lpcoll data must be float32 or bfloat16, got %s" % t.dtype)


def nblocks(n, block=BLOCK):
    return (n + block - 1) // block


def _stream(stream):
    if stream is None:
        return _torch().cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _need(t, what, dtype=None, numel=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % what)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % what)
    if t.device.index != torch.cuda.current_device():
        # the library launches on the current device: a tensor of another
        # GPU would be dereferenced there
        raise ValueError("%s is on %s but the current CUDA device is cuda:%d"
                         % (what, t.device, torch.cuda.current_device()))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % what)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (what, dtype, t.dtype))
    if numel is not None and t.numel() < numel:
        raise ValueError("%s holds %d elements, needs %d" % (what, t.numel(), numel))
    return t.data_ptr()


def lp_quantize(x, codes, scales, block=BLOCK, stream=None):
    """One rank's message x -> FP8 payload (codes uint8[n], scales f32[ceil(n/128)])."""
    torch = _torch()
    n = x.numel()
    xp = _need(x, "x")
    cp = _need(codes, "codes", torch.uint8, n)
    sp = _need(scales, "scales", torch.float32, nblocks(n, block) if block else 0)
    raw_lp_quantize(xp, dtype_code(x), n, block, cp, sp, _stream(stream))
    return codes, scales


def lp_dequantize(codes, scales, out, block=BLOCK, stream=None):
    """FP8 payload -> out (float32 or bfloat16, n = out.numel())."""
    torch = _torch()
    n = out.numel()
    op = _need(out, "out")
    cp = _need(codes, "codes", torch.uint8, n)
    sp = _need(scales, "scales", torch.float32, nblocks(n, block) if block else 0)
    raw_lp_dequantize(cp, sp, n, block, op, dtype_code(out), _stream(stream))
    return out


def lp_reduce(codes, scales, out, block=BLOCK, stream=None):
    """Sum of the dequantized payloads codes[r]/scales[r] (rank order) -> out."""
    torch = _torch()
    n = out.numel()
    op = _need(out, "out")
    cps = [_need(c, "codes[%d]" % r, torch.uint8, n) for r, c in enumerate(codes)]
    sps = [_need(s, "scales[%d]" % r, torch.float32, nblocks(n, block) if block else 0)
           for r, s in enumerate(scales)]
    if len(cps) != len(sps):
        raise ValueError("codes and scales must list the same ranks")
    raw_lp_reduce(cps, sps, len(cps), n, block, op, dtype_code(out), _stream(stream))
    return out


def _rank_args(ins, outs, wire_codes, wire_scales, block):
    torch = _torch()
    _one_per_rank(ins, outs)
    n = ins[0].numel()
    dt = ins[0].dtype
    ip = [_need(t, "in[%d]" % r, dt, None) for r, t in enumerate(ins)]
    if any(t.numel() != n for t in ins):
        raise ValueError("every rank's message must have the same length")
    op = [_need(t, "out[%d]" % r, dt, n) for r, t in enumerate(outs)]
    if block:
        if wire_codes is None or wire_scales is None:
            raise ValueError("low precision (block=128) needs wire_codes and wire_scales")
        wc = [_need(t, "wire_codes[%d]" % r, torch.uint8, n)
              for r, t in enumerate(wire_codes)]
        ws = [_need(t, "wire_scales[%d]" % r, torch.float32, nblocks(n, block))
              for r, t in enumerate(wire_scales)]
        if len(wc) != len(ins) or len(ws) != len(ins):
            raise ValueError("one wire payload per rank")
    else:
        wc, ws = [], []
    return n, dtype_code(ins[0]), ip, op, wc, ws


def dda_flat_sim(ins, outs, block=BLOCK, wire_codes=None, wire_scales=None,
                 stream=None):
    """DDA flat allreduce of the N rank messages ``ins`` into ``outs``."""
    n, dt, ip, op, wc, ws = _rank_args(ins, outs, wire_codes, wire_scales, block)
    raw_dda_flat_sim(ip, op, len(ip), n, dt, block, wc, ws, _stream(stream))
    return outs


def dda_tree_sim(ins, outs, block=BLOCK, wire_codes=None, wire_scales=None,
                 shard_codes=None, shard_scales=None, stream=None):
    """DDA tree allreduce (reduce-scatter, requantize, all-gather)."""
    torch = _torch()
    n, dt, ip, op, wc, ws = _rank_args(ins, outs, wire_codes, wire_scales, block)
    sc = ss = 0
    if block:
        if shard_codes is None or shard_scales is None:
            raise ValueError("low precision tree needs shard_codes and shard_scales")
        sc = _need(shard_codes, "shard_codes", torch.uint8, n)
        ss = _need(shard_scales, "shard_scales", torch.float32, nblocks(n, block))
    raw_dda_tree_sim(ip, op, len(ip), n, dt, block, wc, ws, sc, ss, _stream(stream))
    return outs


def shard_len(n, nranks, block=BLOCK):
    """Elements per reduce-scatter shard (the last shard may be shorter)."""
    per = -(-n // nranks)
    return -(-per // block) * block if block else per


def _wire_args(ins, wire_codes, wire_scales, block, ncodes, nscales):
    torch = _torch()
    if not block:
        return [], []
    if wire_codes is None or wire_scales is None:
        raise ValueError("low precision (block=128) needs wire_codes and wire_scales")
    if len(wire_codes) != len(ins) or len(wire_scales) != len(ins):
        raise ValueError("one wire payload per rank")
    wc = [_need(t, "wire_codes[%d]" % r, torch.uint8, ncodes)
          for r, t in enumerate(wire_codes)]
    ws = [_need(t, "wire_scales[%d]" % r, torch.float32, nscales)
          for r, t in enumerate(wire_scales)]
    return wc, ws


def _one_per_rank(ins, outs):
    # the C call reads exactly N entries of every per-rank array
    if len(ins) == 0:
        raise ValueError("need at least one rank")
    if len(outs) != len(ins):
        raise ValueError("one output per input rank (%d inputs, %d outputs)"
                         % (len(ins), len(outs)))


def _inputs(ins, count):
    dt = ins[0].dtype
    ip = [_need(t, "in[%d]" % r, dt, None) for r, t in enumerate(ins)]
    if any(t.numel() != count for t in ins):
        raise ValueError("every rank's input must have %d elements" % count)
    return ip, dt


def reduce_scatter_sim(ins, outs, block=BLOCK, wire_codes=None, wire_scales=None,
                       stream=None):
    """ReduceScatter: outs[r] (shard_len elements, the last rank's fewer; may
    be None for an empty shard) receives shard r of the sum of ``ins``."""
    _one_per_rank(ins, outs)
    N = len(ins)
    n = ins[0].numel()
    ip, dt = _inputs(ins, n)
    per = shard_len(n, N, block) if n else 0
    op = []
    for r, t in enumerate(outs):
        k = max(0, min(per, n - r * per))
        op.append(0 if (t is None and k == 0) else _need(t, "out[%d]" % r, dt, k))
    wc, ws = _wire_args(ins, wire_codes, wire_scales, block, n, nblocks(n))
    raw_collective("reduce_scatter_sim", ip, op, N, n, dtype_code(ins[0]), block, wc, ws,
                   _stream(stream))
    return outs


def all_gather_sim(ins, outs, block=BLOCK, wire_codes=None, wire_scales=None,
                   stream=None):
    """AllGather: every outs[r] (N*m elements) receives all N contributions."""
    _one_per_rank(ins, outs)
    N = len(ins)
    m = ins[0].numel()
    ip, dt = _inputs(ins, m)
    op = [_need(t, "out[%d]" % r, dt, N * m) for r, t in enumerate(outs)]
    wc, ws = _wire_args(ins, wire_codes, wire_scales, block, m, nblocks(m))
    raw_collective("all_gather_sim", ip, op, N, m, dtype_code(ins[0]), block, wc, ws,
                   _stream(stream))
    return outs


def all_to_all_sim(ins, outs, block=BLOCK, wire_codes=None, wire_scales=None,
                   stream=None):
    """AlltoAll: ins[r] is N chunks of c elements; outs[j][r*c:(r+1)*c] receives
    chunk j of rank r."""
    _one_per_rank(ins, outs)
    N = len(ins)
    total = ins[0].numel()
    if total % N:
        raise ValueError("all_to_all input length must be a multiple of N")
    c = total // N
    ip, dt = _inputs(ins, total)
    op = [_need(t, "out[%d]" % r, dt, total) for r, t in enumerate(outs)]
    wc, ws = _wire_args(ins, wire_codes, wire_scales, block, total, N * nblocks(c))
    raw_collective("all_to_all_sim", ip, op, N, c, dtype_code(ins[0]), block, wc, ws,
                   _stream(stream))
    return outs


def dda_flat_sim_noalloc(ins, outs, stream=None):
    """dda_flat_sim with block=128 whose wires live in the library's own
    fixed device array (for callers that cannot allocate device memory)."""
    _one_per_rank(ins, outs)
    n = ins[0].numel()
    ip, dt = _inputs(ins, n)
    op = [_need(t, "out[%d]" % r, dt, n) for r, t in enumerate(outs)]
    raw_dda_flat_sim_noalloc(ip, op, len(ip), n, dtype_code(ins[0]), _stream(stream))
    return outs


def lp_quantize_fmt(x, codes, scales, block, fmt, stream=None):
    """Format / block-size variant of lp_quantize (fmt E4M3 or E5M2; block 32,
    64, 128 or 256)."""
    torch = _torch()
    n = x.numel()
    xp = _need(x, "x")
    cp = _need(codes, "codes", torch.uint8, n)
    sp = _need(scales, "scales", torch.float32, nblocks(n, block))
    _check(lib().lp_quantize_fmt(xp, dtype_code(x), n, block, fmt, cp, sp,
                                 _stream(stream)), "lp_quantize_fmt")
    return codes, scales


def lp_dequantize_fmt(codes, scales, out, block, fmt, stream=None):
    torch = _torch()
    n = out.numel()
    op = _need(out, "out")
    cp = _need(codes, "codes", torch.uint8, n)
    sp = _need(scales, "scales", torch.float32, nblocks(n, block))
    _check(lib().lp_dequantize_fmt(cp, sp, n, block, fmt, op, dtype_code(out),
                                   _stream(stream)), "lp_dequantize_fmt")
    return out


def lp_reduce_fmt(codes, scales, out, block, fmt, stream=None):
    torch = _torch()
    n = out.numel()
    op = _need(out, "out")
    cps = [_need(c, "codes[%d]" % r, torch.uint8, n) for r, c in enumerate(codes)]
    sps = [_need(s, "scales[%d]" % r, torch.float32, nblocks(n, block))
           for r, s in enumerate(scales)]
    if len(cps) != len(sps):
        raise ValueError("codes and scales must list the same ranks")
    _check(lib().lp_reduce_fmt(_rank_ptrs(cps, len(cps), "codes"),
                               _rank_ptrs(sps, len(cps), "scales"), len(cps), n, block, fmt,
                               op, dtype_code(out), _stream(stream)), "lp_reduce_fmt")
    return out


def lpcoll_host_workspace_bytes(nranks, chunk, dtype, block, flat, tree, slots):
    """Device workspace bytes lpcoll_host_allreduce needs (0 if invalid)."""
    return lib().lpcoll_host_workspace_bytes(nranks, chunk, dtype, block, int(bool(flat)),
                                             int(bool(tree)), slots)


def raw_host_allreduce(in_ptrs, flat_ptrs, tree_ptrs, nranks, n, dtype, block, chunk,
                       slots, ws_ptr, ws_bytes, s_in, s_cmp, s_out):
    """lpcoll_host_allreduce with host pointers as ints; flat_ptrs / tree_ptrs
    None to skip that allreduce."""
    _check(lib().lpcoll_host_allreduce(
        _rank_ptrs(in_ptrs, nranks, "host_in"),
        _rank_ptrs(flat_ptrs, nranks, "host_out_flat") if flat_ptrs is not None else None,
        _rank_ptrs(tree_ptrs, nranks, "host_out_tree") if tree_ptrs is not None else None,
        nranks, n, dtype, block, chunk, slots, ws_ptr, ws_bytes, s_in, s_cmp, s_out),
        "lpcoll_host_allreduce")


def _host(t, what, dtype, numel):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError("%s must be a host (CPU) torch.Tensor" % what)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % what)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (what, dtype, t.dtype))
    if t.numel() < numel:
        raise ValueError("%s holds %d elements, needs %d" % (what, t.numel(), numel))
    return t.data_ptr()


def lpcoll_host_allreduce(host_ins, host_out_flat=None, host_out_tree=None, block=BLOCK,
                          chunk=1 << 22, slots=3, workspace=None, streams=None):
    """Flat and / or tree allreduce of N host tensors into host tensors,
    chunked through a device workspace with copies and kernels overlapped.
    Returns when the results are in host memory. workspace: a CUDA uint8
    tensor of at least lpcoll_host_workspace_bytes(...) bytes; streams: three
    CUDA streams (copy in, compute, copy out)."""
    torch = _torch()
    for outs in (host_out_flat, host_out_tree):
        if outs is not None:
            _one_per_rank(host_ins, outs)
    N = len(host_ins)
    n = host_ins[0].numel()
    dt = host_ins[0].dtype
    ip = [_host(t, "host_in[%d]" % r, dt, n) for r, t in enumerate(host_ins)]
    fp = None if host_out_flat is None else [
        _host(t, "host_out_flat[%d]" % r, dt, n) for r, t in enumerate(host_out_flat)]
    tp = None if host_out_tree is None else [
        _host(t, "host_out_tree[%d]" % r, dt, n) for r, t in enumerate(host_out_tree)]
    need = lpcoll_host_workspace_bytes(N, chunk, dtype_code(host_ins[0]), block,
                                       fp is not None, tp is not None, slots)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device="cuda")
    wp = _need(workspace, "workspace", torch.uint8, need)
    if streams is None:
        streams = [torch.cuda.current_stream()] * 3
    sp = [_stream(x) for x in streams]
    raw_host_allreduce(ip, fp, tp, N, n, dtype_code(host_ins[0]), block, chunk, slots, wp,
                       workspace.numel(), *sp)
    return host_out_flat, host_out_tree
