"""Helpers for the GPU tests: moving oracle-format arrays to and from torch
CUDA tensors, and guard-banded device buffers that detect stray writes."""
import numpy as np
import torch

GUARD = 64          # guard elements after every buffer
CANARY_U8 = 0xA5


def to_dev(a):
    """float32 -> torch.float32; uint16 (bf16 bits) -> torch.bfloat16."""
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def from_dev(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


class Guarded:
    """A device buffer of n elements followed by GUARD canary elements."""

    def __init__(self, n, dtype):
        self.n = n
        self.full = torch.empty(n + GUARD, dtype=dtype, device="cuda")
        self.full.view(torch.uint8).fill_(CANARY_U8)
        self.t = self.full[:n]

    def intact(self):
        tail = self.full[self.n:].contiguous().view(torch.uint8)
        return bool(torch.all(tail == CANARY_U8).item())


def same_bits(a, b):
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    return a.shape == b.shape and np.array_equal(a.view(np.uint8), b.view(np.uint8))


def first_mismatch(a, b):
    a = np.ascontiguousarray(a).view(np.uint8 if a.dtype == np.uint8 else
                                     (np.uint16 if a.itemsize == 2 else np.uint32))
    b = np.ascontiguousarray(b).view(a.dtype)
    idx = np.nonzero(a != b)[0]
    return None if idx.size == 0 else (int(idx[0]), int(idx.size))
