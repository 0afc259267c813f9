"""GB300-native low-precision (FP8) collective reduction and DDA flat / tree
allreduce, with N ranks emulated as N buffers in one GPU's HBM.

The compute path is liblpcoll.so (hand-written CUDA for sm_103a behind the C
ABI in include/lpcoll.h); this package is its binding (``_binding``), an
in-place allreduce facade (``allreduce``), the build step (``build``) and the
seeded workload generators (``workloads``).
"""
from ._binding import (BF16, BLOCK, E4M3, E5M2, F32, MAX_RANKS, VARIANT_BLOCKS,
                       LpcollError, all_gather_sim, all_to_all_sim, dda_flat_sim,
                       dda_flat_sim_noalloc, dda_tree_sim, lib, lp_dequantize,
                       lp_dequantize_fmt, lp_quantize, lp_quantize_fmt, lp_reduce,
                       lp_reduce_fmt, lpcoll_host_allreduce,
                       lpcoll_host_workspace_bytes, nblocks, reduce_scatter_sim,
                       shard_len, status_string)
from .allreduce import Workspace, allreduce_sim, choose

__all__ = ["BF16", "BLOCK", "F32", "MAX_RANKS", "LpcollError", "Workspace",
           "all_gather_sim", "all_to_all_sim", "allreduce_sim", "choose",
           "dda_flat_sim", "dda_flat_sim_noalloc", "dda_tree_sim", "lib",
           "lp_dequantize", "lp_quantize", "lp_reduce", "nblocks", "E4M3", "E5M2",
           "VARIANT_BLOCKS", "lp_quantize_fmt", "lp_dequantize_fmt", "lp_reduce_fmt",
           "lpcoll_host_allreduce", "lpcoll_host_workspace_bytes",
           "reduce_scatter_sim", "shard_len", "status_string"]
