"""Allreduce of N host-resident rank buffers through one GPU, with transfers
and kernels overlapped.

The emulated collective is element-wise across ranks and every stage works
on independent 128-element blocks, so a message can be processed in chunks
whose boundaries are multiples of 128 elements with results identical to one
launch over the whole message. ``HostAllreduce`` streams the chunks through a
ring of device slots on three CUDA streams:

    h2d streams:    copy chunk k of every rank's input into slot k % S
    compute stream: run the requested allreduce(s) on slot k % S
    d2h streams:    copy chunk k of every result back to host memory

Events order the three stages of one chunk and keep a slot from being
refilled before its results have left the GPU, so copies in both directions
and the kernels of neighbouring chunks run at the same time. Host buffers
must be pinned (``torch.Tensor.pin_memory()``) for the copies to be
asynchronous. The kernels are the library's, called through the C ABI.
"""
import torch

from . import _binding as B

TORCH_DT = {B.F32: torch.float32, B.BF16: torch.bfloat16}


class _Slot:
    def __init__(self, nranks, chunk, dtype, block, algos, device, ncopy):
        tdt = TORCH_DT[dtype]
        nb = B.nblocks(chunk)
        self.ins = [torch.empty(chunk, dtype=tdt, device=device) for _ in range(nranks)]
        self.outs = {a: [torch.empty(chunk, dtype=tdt, device=device)
                         for _ in range(nranks)] for a in algos}
        if block:
            self.wc = [torch.empty(chunk, dtype=torch.uint8, device=device)
                       for _ in range(nranks)]
            self.ws = [torch.empty(nb, dtype=torch.float32, device=device)
                       for _ in range(nranks)]
            self.sc = torch.empty(chunk, dtype=torch.uint8, device=device)
            self.ss = torch.empty(nb, dtype=torch.float32, device=device)
            self.p_wc = [t.data_ptr() for t in self.wc]
            self.p_ws = [t.data_ptr() for t in self.ws]
            self.p_sc, self.p_ss = self.sc.data_ptr(), self.ss.data_ptr()
        else:
            self.p_wc = self.p_ws = []
            self.p_sc = self.p_ss = 0
        self.p_in = [t.data_ptr() for t in self.ins]
        self.p_out = {a: [t.data_ptr() for t in v] for a, v in self.outs.items()}
        self.h2d_done = [torch.cuda.Event() for _ in range(ncopy)]
        self.compute_done = torch.cuda.Event()
        self.d2h_done = [torch.cuda.Event() for _ in range(ncopy)]
        self.used = False


class HostAllreduce:
    """SUM-allreduce of N pinned host buffers (n elements each) on the GPU.

    algos: which allreduces to run on every chunk, "flat" and/or "tree"; each
    writes its own set of N host outputs. chunk: elements per chunk (rounded
    up to a multiple of 128). slots: device buffers in flight (>= 2).
    copy_streams: streams per copy direction; rank r's copies go on stream
    r % copy_streams, so several copy engines can work at once.
    """

    def __init__(self, nranks, n, dtype, block=B.BLOCK, algos=("flat",),
                 chunk=1 << 22, slots=3, copy_streams=1, device="cuda"):
        if block not in (0, B.BLOCK):
            raise ValueError("block must be 0 or %d" % B.BLOCK)
        if slots < 2:
            raise ValueError("need at least two slots to overlap")
        self.nranks, self.n, self.dtype, self.block = nranks, n, dtype, block
        self.algos = tuple(algos)
        chunk = max(B.BLOCK, (min(chunk, max(n, 1)) + B.BLOCK - 1) // B.BLOCK * B.BLOCK)
        self.chunk = chunk
        self.device = torch.device(device)
        self.ncopy = max(1, min(copy_streams, nranks))
        nslots = max(1, min(slots, -(-n // chunk)))
        self.slots = [_Slot(nranks, chunk, dtype, block, self.algos, self.device,
                            self.ncopy) for _ in range(nslots)]
        self.h2d = [torch.cuda.Stream(self.device) for _ in range(self.ncopy)]
        self.compute = torch.cuda.Stream(self.device)
        self.d2h = [torch.cuda.Stream(self.device) for _ in range(self.ncopy)]

    def chunks(self):
        for k, lo in enumerate(range(0, self.n, self.chunk)):
            yield k, lo, min(self.n, lo + self.chunk)

    def _launch(self, slot, algo, m):
        stream = self.compute.cuda_stream
        if algo == "tree":
            B.raw_dda_tree_sim(slot.p_in, slot.p_out[algo], self.nranks, m, self.dtype,
                               self.block, slot.p_wc, slot.p_ws, slot.p_sc, slot.p_ss,
                               stream)
        else:
            B.raw_dda_flat_sim(slot.p_in, slot.p_out[algo], self.nranks, m, self.dtype,
                               self.block, slot.p_wc, slot.p_ws, stream)

    def run(self, host_ins, host_outs):
        """host_ins: N host tensors of n elements; host_outs: {algo: N host
        tensors}. Enqueues everything and returns; call ``synchronize()``
        before reading host_outs."""
        if len(host_ins) != self.nranks:
            raise ValueError("one input per rank")
        S = len(self.slots)
        C = self.ncopy
        for k, lo, hi in self.chunks():
            m = hi - lo
            slot = self.slots[k % S]
            for i, st in enumerate(self.h2d):
                with torch.cuda.stream(st):
                    if slot.used:
                        for ev in slot.d2h_done:
                            st.wait_event(ev)
                    for r in range(i, self.nranks, C):
                        slot.ins[r][:m].copy_(host_ins[r][lo:hi], non_blocking=True)
                    slot.h2d_done[i].record(st)
            for ev in slot.h2d_done:
                self.compute.wait_event(ev)
            for a in self.algos:
                self._launch(slot, a, m)
            slot.compute_done.record(self.compute)
            for i, st in enumerate(self.d2h):
                with torch.cuda.stream(st):
                    st.wait_event(slot.compute_done)
                    for a in self.algos:
                        for r in range(i, self.nranks, C):
                            host_outs[a][r][lo:hi].copy_(slot.outs[a][r][:m],
                                                         non_blocking=True)
                    slot.d2h_done[i].record(st)
            slot.used = True

    def synchronize(self):
        for st in self.d2h:
            st.synchronize()

    def start_after(self, stream):
        """Make the next run's first copies wait for work queued on stream."""
        for st in self.h2d:
            st.wait_stream(stream)

    def finish_before(self, stream):
        """Make work queued on stream afterwards wait for the last results."""
        for st in self.d2h:
            stream.wait_stream(st)

    def kernel_launches_per_run(self):
        return len(self.algos) * len(list(self.chunks()))
