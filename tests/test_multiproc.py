"""The benchmark's multi-process path on CPU: two ranks over gloo (no GPU).

One process per GPU runs an independent replica of the round (the path has no
exchange step), so what is shared across ranks is the timing: the slowest rank's
time per step, and the whole-job throughput computed from it.
"""
import os
import socket
import sys

import pytest

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench

    ms = 10.0 + 2.5 * rank  # rank 1 is the slower one
    m = bench.ranks_max(ms, world)
    q.put((rank, m, bench.job_rounds_per_s(m, world)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = {}
    try:
        for _ in range(2):
            rank, m, v = q.get(timeout=120)
            got[rank] = (m, v)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [p.exitcode for p in procs] == [0, 0]
    for rank in (0, 1):
        m, v = got[rank]
        assert m == pytest.approx(12.5)
        assert v == pytest.approx(2 * 1000.0 / 12.5)  # both replicas' rounds in the slowest rank's time


def test_single_process_is_its_own_max():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.ranks_max(3.25, 1) == 3.25
    assert bench.job_rounds_per_s(4.0, 1) == pytest.approx(250.0)


def test_reference_arm_prints_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class A:
        config, seed, steps, warmup = "tiny", 0, 1, 0

    assert bench.reference_arm(A, rank=1, world=2) == 0
    assert capsys.readouterr().out == ""
