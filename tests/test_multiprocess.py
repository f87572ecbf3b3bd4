"""The N > 1 path of bench.py on CPU with two gloo ranks: the job's time is
the slowest rank's, the throughput counts every rank's steps, and the
reference arm's other ranks exit without work.  (Every (b, h) is independent,
so N GPUs run replicas: the only cross-rank step is this reduction.)"""

import multiprocessing as mp
import os
import socket

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t = bench.reduce_max_time(0.5 + rank, torch.device("cpu"))
    v = bench.job_throughput(world, 10, 2e12, t)
    out.put((rank, t, v))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_all_steps():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, v in res:
        assert t == pytest.approx(1.5)                      # the slowest rank's time
        assert v == pytest.approx(2 * 10 * 2e12 / 1.5 / 1e12)  # both ranks' steps


def test_reference_arm_other_ranks_do_no_work(monkeypatch):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")

    class Args:
        steps, warmup, gpus = 2, 1, 2

    called = []
    monkeypatch.setattr(bench, "oracle_sample", lambda *a, **k: called.append(1) or (0.0, 0.0))
    assert bench.run_reference(Args(), None) is None
    assert not called
