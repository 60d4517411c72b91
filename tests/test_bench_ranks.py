"""Host logic of the benchmark's N-rank path, on CPU with two gloo ranks: the
barrier, the max-over-ranks step time, and the reference arm running on rank 0
only. The attention path itself has no collective (independent replicas)."""
import os
import socket
import sys
import types

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import io
    import contextlib
    import torch
    import torch.distributed as dist
    import bench

    w, r, local = bench.init_dist("gloo")
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    # each rank reports its own step time; every rank must see the slowest
    t = bench.max_over_ranks(1.5 + rank, w, torch.device("cpu"))
    # the reference arm prints only on rank 0; other ranks return without work
    printed = ""
    if rank != 0:
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            bench.run_reference(types.SimpleNamespace(steps=1, warmup=0))
        printed = buf.getvalue()
    bench.barrier(w)
    out.put((rank, t, printed))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_barrier_and_max_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=100) for _ in range(world))
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert [r for r, _, _ in res] == [0, 1]
    assert all(t == 2.5 for _, t, _ in res)     # max over ranks of 1.5 and 2.5
    assert res[1][2] == ""                       # rank 1 ran no reference work


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.0, 1, None) == 3.0
    bench.barrier(1)
