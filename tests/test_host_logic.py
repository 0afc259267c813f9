"""Host-side logic that needs no GPU: algorithm choice of the allreduce
facade, benchmark byte accounting, and the workload recipes."""
import numpy as np
import pytest

import bench
from precision_collective_reduction_gb300 import allreduce as AR
from precision_collective_reduction_gb300 import workloads as W

MiB = 1 << 20


def test_low_precision_off_by_default():
    assert AR.choose(64 * MiB, env={}) == ("flat", 0)


def test_env_switch_and_threshold():
    env = {AR.LP_ENV: "1"}
    assert AR.choose(16 * MiB, env=env) == ("flat", 128)       # at the threshold
    assert AR.choose(16 * MiB - 1, env=env) == ("flat", 0)     # below it
    env[AR.LP_MIN_BYTES_ENV] = "1024"
    assert AR.choose(4096, env=env) == ("flat", 128)


def test_argument_overrides_env():
    assert AR.choose(32 * MiB, low_precision=True, env={}) == ("flat", 128)
    assert AR.choose(32 * MiB, low_precision=False, env={AR.LP_ENV: "1"}) == ("flat", 0)


def test_algo_selection():
    assert AR.choose(1024, algo="tree", env={}) == ("tree", 0)
    env = {AR.TREE_MIN_BYTES_ENV: str(MiB)}
    assert AR.choose(MiB, env=env)[0] == "tree"
    assert AR.choose(MiB - 1, env=env)[0] == "flat"
    with pytest.raises(ValueError):
        AR.choose(1, algo="ring", env={})


def test_algorithmic_bytes_match_the_formulas():
    # N n (2 s + q) for flat, plus n q for the tree's shard wire, with
    # q = 1 + 4/128 bytes per element of FP8 payload
    w = W.LP_GRAD_N8_256MB_F32
    assert bench.bytes_alg(8, w.n, 4, 128, "flat") == 4_848_615_424
    assert bench.bytes_alg(8, w.n, 4, 128, "tree") == 4_917_821_440
    assert bench.bytes_alg(2, 1 << 20, 4, 128, "flat") == 18_939_904
    assert bench.bytes_alg(8, 32 * 8192, 2, 0, "flat") == 8_388_608
    assert bench.bytes_alg(8, 8 * MiB, 2, 128, "flat") == 337_641_472
    assert bench.bytes_alg(8, 32 * MiB, 2, 128, "tree") == 1_385_168_896


def test_workload_recipes():
    w = W.LP_GRAD_N8_256MB_F32
    x = W.draw(w, 0, n=128 * 1000)
    big = np.abs(x.reshape(-1, 128)).max(axis=1) > 0.05
    assert 3 <= big.sum() <= 30          # about 1% of blocks scaled by 1e3
    d = W.draw(W.DECODE_EXACT_FLAT_N8_BF16, 0)
    assert d.dtype == np.uint16 and d.size == 32 * 8192
    a = W.draw(W.LP_FLAT_N2_1M_F32, 1, n=1000)
    assert np.array_equal(a, W.draw(W.LP_FLAT_N2_1M_F32, 1, n=1000))   # seeded
    assert not np.array_equal(a, W.draw(W.LP_FLAT_N2_1M_F32, 0, n=1000))


def test_collective_bytes():
    n, N = 8 * MiB, 8
    q = n + 4 * (n // 128)
    assert bench.collective_bytes("reduce_scatter", N, n, 2, 128) == N * n * 2 + N * q + n * 2
    m = n // N
    assert bench.collective_bytes("all_gather", N, m, 2, 128) == \
        N * m * 2 + N * (m + 4 * m // 128) + N * N * m * 2
    assert bench.collective_bytes("all_to_all", N, m, 2, 0) == 2 * N * N * m * 2


def test_staged_bytes():
    n, N = 128 * 1000, 8
    q = n + 4 * 1000
    assert bench.staged_bytes("lp_quantize", N, n, 4) == 4 * n + q
    assert bench.staged_bytes("lp_dequantize", N, n, 2) == q + 2 * n
    assert bench.staged_bytes("lp_reduce", N, n, 4) == N * q + 4 * n
    # the staged chain of the 16 MiB BF16 workload: 8 quantizes (16 MiB read,
    # 8 Mi codes + 64 Ki scales written each), then the reduce of the 8
    # payloads into one 16 MiB output
    n = 8 * (1 << 20)
    chain = 8 * bench.staged_bytes("lp_quantize", 8, n, 2) + \
        bench.staged_bytes("lp_reduce", 8, n, 2)
    assert chain == 8 * (2 * n + n + 4 * (n // 128)) + 8 * (n + 4 * (n // 128)) + 2 * n
    assert chain == 289_406_976


def test_binding_refuses_short_rank_lists():
    # the C calls read N entries of every per-rank pointer array: the binding
    # must refuse a shorter list before it calls the library
    import torch
    from precision_collective_reduction_gb300 import _binding as B
    with pytest.raises(ValueError):
        B.raw_dda_flat_sim([16, 32], [16], 2, 10, B.F32, 0, [], [], 0)
    with pytest.raises(ValueError):
        B.raw_dda_tree_sim([16, 32], [16, 32], 2, 10, B.F32, 128, [16], [16, 32], 16, 16, 0)
    with pytest.raises(ValueError):
        B.raw_collective("all_gather_sim", [16], [16, 32], 2, 10, B.F32, 0, [], [], 0)
    with pytest.raises(ValueError):
        B.raw_lp_reduce([16, 32, 48], [16, 32], 3, 10, 128, 16, B.F32, 0)
    with pytest.raises(ValueError):
        B.raw_dda_flat_sim_noalloc([16], [16], 2, 10, B.F32, 0)
    with pytest.raises(ValueError):
        B.raw_host_allreduce([16, 32], [16], None, 2, 10, B.F32, 128, 128, 1, 16, 1 << 20,
                             0, 0, 0)
    # tensor-level calls check the list lengths before anything else
    t = [torch.zeros(4) for _ in range(3)]
    for fn in (B.dda_flat_sim, B.dda_tree_sim, B.reduce_scatter_sim, B.all_gather_sim,
               B.all_to_all_sim):
        with pytest.raises(ValueError):
            fn(t, t[:2], block=0)
    with pytest.raises(ValueError):
        B.dda_flat_sim_noalloc(t, t[:1])
    with pytest.raises(ValueError):
        B.lpcoll_host_allreduce(t, host_out_flat=t[:2])
    with pytest.raises(ValueError):
        B.dda_flat_sim([], [], block=0)
