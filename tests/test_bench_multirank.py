"""bench.py's multi-rank logic (replicas, no data-path collective) on CPU with
gloo, world size 2: the reported time is the slowest rank's, the value counts
every rank's work, and the reference arm runs on rank 0 only."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [3.0, 5.0][rank]
    got = bench.max_over_ranks(ms, world)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, got))


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get() for _ in range(2))
    assert res == {0: 5.0, 1: 5.0}


def test_whole_job_value_counts_all_ranks():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.whole_job_tflops(1e12, 10, 1, 100.0)
    two = bench.whole_job_tflops(1e12, 10, 2, 100.0)
    assert abs(one - 100.0) < 1e-9 and abs(two - 200.0) < 1e-9


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")

    class A:
        config = "latent"
        gpus = 2
    assert bench.run_reference(A()) == 0
