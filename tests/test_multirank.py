"""Host logic of the multi-GPU benchmark run, on CPU with the gloo backend
and two ranks: each rank is an independent replica, the job time is the
slowest rank's, and the throughput counts the work of every rank."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        ms = 10.0 + 5.0 * r
        worst = bench.max_over_ranks(ms, dist, "cpu")
        dist.barrier()
        q.put((r, w, local, worst,
               bench.whole_job_gbps(1e9, 4, w, worst)))
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for r, (rank, w, local, worst, gbps) in enumerate(res):
        assert (rank, w, local) == (r, world, r)
        assert worst == 15.0                      # slowest rank's time
        assert gbps == pytest.approx(1e9 * 4 * 2 / 15e-3 / 1e9)


def test_single_rank_defaults(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5


def test_stdout_redirect_keeps_fd1_clean(capfd):
    with bench._StdoutToStderr():
        os.write(1, b"banner\n")
    os.write(1, b"json\n")
    out, err = capfd.readouterr()
    assert out == "json\n" and "banner" in err
