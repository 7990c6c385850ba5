"""The N > 1 path of bench.py on CPU: two gloo ranks, each a replica with its own sequences
and its own time; the job's time is the slowest rank's and its rate counts every rank's
units.  (No GPU: the collective is the only cross-rank step of the path.)"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist          # noqa: E402
import torch.multiprocessing as mp        # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, lr, w = bench.dist_env()
    local_ms = 100.0 + 50.0 * rank               # rank 1 is the slow one
    job_ms = bench.max_over_ranks(local_ms)
    rate = bench.whole_job_rate(w, 6, 10, job_ms)
    out.put((r, lr, w, job_ms, rate))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_replicas_report_the_slowest_time_and_all_units():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res.sort()
    assert [x[0] for x in res] == [0, 1] and all(x[2] == world for x in res)
    for r, lr, w, job_ms, rate in res:
        assert lr == r
        assert job_ms == 150.0                                   # the slowest rank
        assert rate == pytest.approx(world * 6 * 10 / 0.150)     # every rank's units


def test_single_process_is_its_own_max():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.whole_job_rate(1, 6, 100, 50.0) == pytest.approx(12000.0)
