"""Seeded synthetic rank buffers for the five reference workloads.

This module only draws random numbers; it holds none of the reduction's
arithmetic, so both the CUDA path and the CPU oracle can take their inputs
from it. Each rank r of a workload draws from its own numpy ``Generator``
keyed by ``(seed, r)``. FP32 data is returned as ``numpy.float32``; BF16 data
as its raw bits in ``numpy.uint16`` (drawn in FP32, then rounded to nearest
even by PyTorch's own conversion).

The message sizes follow the two regimes of the pages ("RCCLX: AMD GPU
communication, Meta open source", code-journey.com): decode-size messages for
the DDA algorithms ("Funcionalidade Principal 1") and messages of 16 MB and
more for the low-precision collectives ("Funcionalidade Principal 2"). The
value distributions are synthetic stand-ins chosen per workload.
"""
from dataclasses import dataclass, field
from typing import List, Tuple

import numpy as np

F32 = 0
BF16 = 1
BLOCK = 128


@dataclass(frozen=True)
class Workload:
    name: str
    nranks: int
    n: int                 # elements per rank
    dtype: int             # F32 or BF16
    block: int             # 128 = low precision, 0 = exact precision
    algos: Tuple[str, ...]  # "flat" and/or "tree"
    dist: str              # generator recipe, see draw()
    seed: int
    params: dict = field(default_factory=dict)

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == F32 else 2

    @property
    def message_bytes(self) -> int:
        return self.n * self.elem_bytes


# The five reference workloads. The first is small enough for the oracle to
# finish in seconds; the others are the full-size cases.
LP_FLAT_N2_1M_F32 = Workload(
    "lp_flat_n2_1Mi_f32", 2, 1 << 20, F32, BLOCK, ("flat",), "normal", 0,
    {"sigma": 1.0})
DECODE_EXACT_FLAT_N8_BF16 = Workload(
    "decode_exact_flat_n8_32x8192_bf16", 8, 32 * 8192, BF16, 0, ("flat",),
    "normal_outliers", 1, {"sigma": 0.02, "p": 0.001, "factor": 50.0})
LP_FLAT_N8_16MB_BF16 = Workload(
    "lp_flat_n8_16MiB_bf16", 8, 8 * (1 << 20), BF16, BLOCK, ("flat",),
    "normal_rank_scaled", 2, {"lo": 0.5, "hi": 2.0})
LP_TREE_N8_64MB_BF16 = Workload(
    "lp_tree_n8_64MiB_bf16", 8, 32 * (1 << 20), BF16, BLOCK, ("tree",),
    "laplace", 3, {"b": 1.0})
LP_GRAD_N8_256MB_F32 = Workload(
    "lp_flat_tree_n8_256MiB_f32", 8, 64 * (1 << 20), F32, BLOCK,
    ("flat", "tree"), "normal_block_outliers", 4,
    {"sigma": 1e-3, "frac": 0.01, "factor": 1e3})

WORKLOADS = [LP_FLAT_N2_1M_F32, DECODE_EXACT_FLAT_N8_BF16, LP_FLAT_N8_16MB_BF16,
             LP_TREE_N8_64MB_BF16, LP_GRAD_N8_256MB_F32]
BY_NAME = {w.name: w for w in WORKLOADS}


def rank_rng(seed: int, rank: int) -> np.random.Generator:
    return np.random.default_rng([seed, rank])


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bits (uint16), rounded to nearest even by PyTorch."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def draw(w: Workload, rank: int, n: int = None) -> np.ndarray:
    """Rank ``rank``'s input for workload ``w``; ``n`` overrides the element
    count (a smaller case drawn with the same recipe and seed)."""
    n = w.n if n is None else n
    g = rank_rng(w.seed, rank)
    p = w.params
    if w.dist == "normal":
        x = g.standard_normal(n, dtype=np.float32) * np.float32(p["sigma"])
    elif w.dist == "normal_outliers":
        x = g.standard_normal(n, dtype=np.float32) * np.float32(p["sigma"])
        hit = g.random(n, dtype=np.float32) < p["p"]
        x[hit] *= np.float32(p["factor"])
    elif w.dist == "normal_rank_scaled":
        c = np.float32(g.uniform(p["lo"], p["hi"]))
        x = g.standard_normal(n, dtype=np.float32) * c
    elif w.dist == "laplace":
        x = g.laplace(0.0, p["b"], n).astype(np.float32)
    elif w.dist == "normal_block_outliers":
        x = g.standard_normal(n, dtype=np.float32) * np.float32(p["sigma"])
        nb = (n + BLOCK - 1) // BLOCK
        k = int(round(p["frac"] * nb))
        flag = np.zeros(nb, dtype=bool)
        flag[g.choice(nb, size=k, replace=False)] = True
        x[np.repeat(flag, BLOCK)[:n]] *= np.float32(p["factor"])
    else:
        raise ValueError("unknown recipe %r" % w.dist)
    x = np.ascontiguousarray(x, dtype=np.float32)
    return to_bf16_bits(x) if w.dtype == BF16 else x


def draw_all(w: Workload, n: int = None) -> List[np.ndarray]:
    return [draw(w, r, n) for r in range(w.nranks)]


def random_inputs(nranks: int, n: int, dtype: int, seed: int,
                  scale_spread: float = 0.0) -> List[np.ndarray]:
    """Generic N(0,1) rank buffers for parity tests of arbitrary sizes; with
    ``scale_spread`` > 0 each 128-block is multiplied by 10**u, u uniform in
    [-spread, spread], to exercise a wide range of block scales."""
    out = []
    for r in range(nranks):
        g = rank_rng(seed, r)
        x = g.standard_normal(n, dtype=np.float32)
        if scale_spread > 0 and n:
            nb = (n + BLOCK - 1) // BLOCK
            e = g.uniform(-scale_spread, scale_spread, nb).astype(np.float32)
            x *= np.repeat(np.float32(10.0) ** e, BLOCK)[:n]
        x = np.ascontiguousarray(x, dtype=np.float32)
        out.append(to_bf16_bits(x) if dtype == BF16 else x)
    return out


def torch_full_example(nranks: int, shape=(10, 20)) -> List[np.ndarray]:
    """The pages' usage example: rank r holds torch.full(shape, r) in FP32
    ("Guia Pratico e Perspectivas")."""
    return [np.full(int(np.prod(shape)), float(r), dtype=np.float32)
            for r in range(nranks)]
