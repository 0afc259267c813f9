"""Allreduce of N host-resident rank buffers through one GPU.

``HostAllreduce`` owns what the library's ``lpcoll_host_allreduce`` needs
for repeated calls on messages of one shape: a device workspace of a few
chunk slots and three CUDA streams (copy in, compute, copy out). Each
``run`` is one call of the native pipeline: the message is processed in
chunks of a multiple of 128 elements (same results as one launch over the
whole message, since every stage works on independent 128-element blocks),
with host->device copies, the flat and / or tree kernels and device->host
copies of different chunks overlapped; it returns when the results are in
host memory. Host buffers should be pinned (``torch.Tensor.pin_memory()``)
for the copies to overlap.
"""
import torch

from . import _binding as B


class HostAllreduce:
    """SUM-allreduce of N host buffers of n elements on the GPU.

    algos: "flat" and / or "tree"; each writes its own N host outputs.
    chunk: elements per chunk (rounded up to a multiple of 128). slots:
    chunks in flight (2 or more overlap copies and kernels).
    """

    def __init__(self, nranks, n, dtype, block=B.BLOCK, algos=("flat",),
                 chunk=1 << 22, slots=3, device="cuda"):
        if block not in (0, B.BLOCK):
            raise ValueError("block must be 0 or %d" % B.BLOCK)
        self.nranks, self.n, self.dtype, self.block = nranks, n, dtype, block
        self.algos = tuple(algos)
        if not set(self.algos) <= {"flat", "tree"} or not self.algos:
            raise ValueError("algos must name flat and / or tree")
        self.chunk = max(B.BLOCK, -(-min(chunk, max(n, 1)) // B.BLOCK) * B.BLOCK)
        self.slots = slots
        self.device = torch.device(device)
        need = B.lpcoll_host_workspace_bytes(nranks, self.chunk, dtype, block,
                                             "flat" in self.algos, "tree" in self.algos,
                                             slots)
        if need == 0:
            raise ValueError("invalid HostAllreduce configuration")
        self.workspace = torch.empty(need, dtype=torch.uint8, device=self.device)
        self.streams = [torch.cuda.Stream(self.device) for _ in range(3)]

    def run(self, host_ins, host_outs):
        """host_ins: N host tensors of n elements; host_outs: {algo: N host
        tensors}. Returns when the results are in host_outs."""
        if len(host_ins) != self.nranks:
            raise ValueError("one input per rank")
        B.lpcoll_host_allreduce(host_ins, host_outs.get("flat"), host_outs.get("tree"),
                                block=self.block, chunk=self.chunk, slots=self.slots,
                                workspace=self.workspace, streams=self.streams)

    def kernel_launches_per_run(self):
        return len(self.algos) * -(-self.n // self.chunk)
