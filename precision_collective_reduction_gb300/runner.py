"""Device buffers for one emulated collective and the calls that run it.

``RankBuffers`` holds, in one GPU's memory, the N rank messages, the N rank
results, the N FP8 wire payloads and the tree's shard payload of a message of
n elements, and launches the flat or tree allreduce over them through the C
ABI. The benchmark and the full-size tests both use it, so they time and
check the same launches.
"""
import torch

from . import _binding as B

TORCH_DT = {B.F32: torch.float32, B.BF16: torch.bfloat16}


class RankBuffers:
    def __init__(self, nranks, n, dtype, block=B.BLOCK, device="cuda",
                 separate_tree_out=False):
        self.nranks, self.n, self.dtype, self.block = nranks, n, dtype, block
        tdt = TORCH_DT[dtype]
        self.ins = [torch.empty(n, dtype=tdt, device=device) for _ in range(nranks)]
        self.outs = [torch.empty(n, dtype=tdt, device=device) for _ in range(nranks)]
        self.tree_outs = ([torch.empty(n, dtype=tdt, device=device)
                           for _ in range(nranks)] if separate_tree_out else self.outs)
        nb = B.nblocks(n)
        if block:
            self.wire_codes = [torch.empty(n, dtype=torch.uint8, device=device)
                               for _ in range(nranks)]
            self.wire_scales = [torch.empty(nb, dtype=torch.float32, device=device)
                                for _ in range(nranks)]
            self.shard_codes = torch.empty(n, dtype=torch.uint8, device=device)
            self.shard_scales = torch.empty(nb, dtype=torch.float32, device=device)
        else:
            self.wire_codes = self.wire_scales = None
            self.shard_codes = self.shard_scales = None
        self._ptrs()

    def _ptrs(self):
        self.p_in = [t.data_ptr() for t in self.ins]
        self.p_out = [t.data_ptr() for t in self.outs]
        self.p_tout = [t.data_ptr() for t in self.tree_outs]
        if self.block:
            self.p_wc = [t.data_ptr() for t in self.wire_codes]
            self.p_ws = [t.data_ptr() for t in self.wire_scales]
            self.p_sc = self.shard_codes.data_ptr()
            self.p_ss = self.shard_scales.data_ptr()
        else:
            self.p_wc = self.p_ws = []
            self.p_sc = self.p_ss = 0
        # prebuilt ctypes pointer arrays: a launch does no Python-side packing
        self.a_in = B.ptr_array(self.p_in)
        self.a_out = B.ptr_array(self.p_out)
        self.a_tout = B.ptr_array(self.p_tout)
        self.a_wc = B.ptr_array(self.p_wc)
        self.a_ws = B.ptr_array(self.p_ws)

    def load(self, host_arrays, non_blocking=False):
        """Copy N host arrays (float32, or bf16 bits as uint16) into the inputs."""
        for t, a in zip(self.ins, host_arrays):
            src = torch.from_numpy(a)
            if self.dtype == B.BF16:
                src = src.view(torch.int16).view(torch.bfloat16)
            t.copy_(src, non_blocking=non_blocking)

    def flat(self, stream):
        st = B.lib().dda_flat_sim(self.a_in, self.a_out, self.nranks, self.n,
                                  self.dtype, self.block, self.a_wc, self.a_ws, stream)
        if st:
            raise B.LpcollError(st, "dda_flat_sim")

    def tree(self, stream):
        st = B.lib().dda_tree_sim(self.a_in, self.a_tout, self.nranks, self.n,
                                  self.dtype, self.block, self.a_wc, self.a_ws,
                                  self.p_sc, self.p_ss, stream)
        if st:
            raise B.LpcollError(st, "dda_tree_sim")

    def run(self, algo, stream):
        (self.tree if algo == "tree" else self.flat)(stream)
