"""In-place allreduce over N emulated ranks, the way the pages' example uses
an allreduce: every rank passes its tensor, SUM is the only operation, and
each tensor is overwritten with the result (code-journey.com "RCCLX: AMD GPU
communication, Meta open source", section "Guia Pratico e Perspectivas").

Algorithm choice (host logic only; the work runs in liblpcoll's kernels):
- Low precision is off unless asked for, as with the pages' environment
  switch (section "Funcionalidade Principal 2", table row "Ativacao"): the
  ``low_precision`` argument, else ``LPCOLL_LOW_PRECISION_ENABLE=1``.
- Even when asked for, it applies only to messages of at least
  ``LPCOLL_LP_MIN_BYTES`` bytes (default 16 MiB, the pages' threshold for the
  low-precision collectives); smaller messages are reduced exactly.
- ``algo``: "flat", "tree", or "auto". The pages place tree at
  somewhat larger messages than flat. Measured on one GB300 with 8 emulated
  ranks (BF16, 8 KiB to 256 MiB per rank), flat is never slower than tree:
  the exact tree is the same kernel, and the low-precision tree adds a
  requantization and a shard wire (equal up to 8 MiB, 2-3% slower from
  32 MiB up). So "auto" means flat unless ``LPCOLL_TREE_MIN_BYTES`` sets a
  message size from which to use tree.
"""
import os

from . import _binding as B

LP_ENV = "LPCOLL_LOW_PRECISION_ENABLE"
LP_MIN_BYTES_ENV = "LPCOLL_LP_MIN_BYTES"
TREE_MIN_BYTES_ENV = "LPCOLL_TREE_MIN_BYTES"
DEFAULT_LP_MIN_BYTES = 16 * (1 << 20)


def _flag(value):
    return str(value).strip().lower() in ("1", "true", "yes", "on")


def choose(message_bytes, low_precision=None, algo="auto", env=None):
    """(algorithm, block) for a message of ``message_bytes`` bytes per rank."""
    env = os.environ if env is None else env
    if algo not in ("auto", "flat", "tree"):
        raise ValueError("algo must be 'auto', 'flat' or 'tree', got %r" % (algo,))
    lp = _flag(env.get(LP_ENV, "0")) if low_precision is None else bool(low_precision)
    min_bytes = int(env.get(LP_MIN_BYTES_ENV, DEFAULT_LP_MIN_BYTES))
    block = B.BLOCK if (lp and message_bytes >= min_bytes) else 0
    if algo == "auto":
        tree_min = env.get(TREE_MIN_BYTES_ENV)
        algo = "tree" if (tree_min is not None and message_bytes >= int(tree_min)) \
            else "flat"
    return algo, block


class Workspace:
    """Device buffers for the FP8 payloads (wires), reused across calls with
    the same device, rank count and length."""

    def __init__(self):
        self._key = None
        self.wire_codes = self.wire_scales = None
        self.shard_codes = self.shard_scales = None

    def get(self, device, nranks, n):
        import torch
        key = (str(device), nranks, n)
        if key != self._key:
            nb = B.nblocks(n)
            self.wire_codes = [torch.empty(n, dtype=torch.uint8, device=device)
                               for _ in range(nranks)]
            self.wire_scales = [torch.empty(nb, dtype=torch.float32, device=device)
                                for _ in range(nranks)]
            self.shard_codes = torch.empty(n, dtype=torch.uint8, device=device)
            self.shard_scales = torch.empty(nb, dtype=torch.float32, device=device)
            self._key = key
        return self


_default_ws = Workspace()


def allreduce_sim(tensors, low_precision=None, algo="auto", stream=None,
                  workspace=None):
    """SUM-allreduce the N rank tensors in place; returns (algo, block) used.

    CUDA tensors are reduced by one fused launch. Host (CPU) tensors, as in
    the pages' example, go through the library's host-buffer pipeline
    (lpcoll_host_allreduce): copied to the GPU chunk by chunk, reduced, and
    written back in place; the call returns when they hold the result."""
    tensors = list(tensors)
    if not tensors:
        raise ValueError("need at least one rank tensor")
    n = tensors[0].numel()
    algo, block = choose(n * tensors[0].element_size(), low_precision, algo)
    if not tensors[0].is_cuda:
        chunk = 1 << 22
        outs = {"flat": None, "tree": None}
        outs[algo] = tensors
        B.lpcoll_host_allreduce(tensors, outs["flat"], outs["tree"], block=block,
                                chunk=chunk, slots=3)
        return algo, block
    ws = None
    if block:
        ws = (workspace or _default_ws).get(tensors[0].device, len(tensors), n)
    kw = {}
    if ws is not None:
        kw = dict(wire_codes=ws.wire_codes, wire_scales=ws.wire_scales)
    if algo == "tree":
        if ws is not None:
            kw.update(shard_codes=ws.shard_codes, shard_scales=ws.shard_scales)
        B.dda_tree_sim(tensors, tensors, block=block, stream=stream, **kw)
    else:
        B.dda_flat_sim(tensors, tensors, block=block, stream=stream, **kw)
    return algo, block
