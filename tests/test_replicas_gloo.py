"""Host logic of bench.py's multi-GPU mode on CPU: world size 2 over gloo.

Each rank is a replica running the whole workload; the timed region's slowest rank sets
the time and the value is the units of all ranks over that time.  These tests run the
rank environment parsing, the barrier and the max-over-ranks reduction with two real
processes (no GPU)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    try:
        w, r, local = bench.dist_env()
        assert (w, r, local) == (world, rank, rank)
        bench.dist_init(w, "gloo")
        bench.dist_barrier(w)
        # rank 1 is the slow replica
        t = 1.5 if rank == 1 else 1.0
        tmax = bench.reduce_max(t, w, torch.device("cpu"))
        rate = bench.whole_job_rate(units_per_rank=100.0, world=w, max_seconds=tmax)
        q.put((rank, tmax, rate))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


def test_replica_timing_takes_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, tmax, rate in res:
        assert tmax == pytest.approx(1.5)
        assert rate == pytest.approx(200.0 / 1.5)


def test_single_process_needs_no_process_group():
    import bench
    assert bench.reduce_max(2.0, 1, torch.device("cpu")) == 2.0
    assert bench.whole_job_rate(10.0, 1, 2.0) == 5.0
