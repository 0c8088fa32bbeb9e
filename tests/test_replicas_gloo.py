"""The multi-process side of bench.py on CPU: with one process per GPU every
rank parses its own replica (no data-path collective), and the timing is the
maximum over ranks after a barrier.  Two gloo ranks check that host logic
without a GPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench._dist()
        assert (ws, r, local) == (world, rank, rank)
        bench._barrier(ws)
        # each rank's step time differs; every rank sees the slowest
        t = bench._max_over_ranks(10.0 + rank, ws, torch.device("cpu"))
        q.put((rank, t))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=5) for _ in range(world))
    assert got == [(0, 11.0), (1, 11.0)]


def test_single_process_needs_no_process_group():
    import bench
    assert bench._max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    bench._barrier(1)  # no-op without a process group
    assert not dist.is_initialized()
