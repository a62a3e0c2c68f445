"""Multi-process path of bench.py on CPU: two gloo ranks run the timing
barrier and the max-over-ranks reduction the GPU replicas use (the decode
step has no data-path exchange, so these are its only collectives)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, _ = bench.dist_env()
        assert (w, r) == (world, rank)
        bench.barrier(w)
        t = bench.max_over_ranks(1.0 + rank * 0.5, w)   # per-rank step time
        units = world * 100                              # weak scaling: every rank runs the same work
        q.put((rank, t, units / t))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert [r for r, _, _ in res] == [0, 1]
    assert all(t == 1.5 for _, t, _ in res)              # max over ranks, seen by every rank
    assert all(abs(v - 200 / 1.5) < 1e-9 for _, _, v in res)


def test_single_process_needs_no_collective():
    import bench
    assert bench.max_over_ranks(2.5, 1) == 2.5
    bench.barrier(1)
