"""The multi-GPU bench path runs independent replicas (the decode path does
not shard): its only cross-rank work is a barrier and the max over ranks of
the timed region.  Checked here with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.distributed as td
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), MK_BENCH_BACKEND="gloo")
    import bench
    r, w, d = bench.dist()
    assert (r, w) == (rank, ws)
    bench.barrier(d)
    got = bench.max_over_ranks(10.0 + rank, d)
    q.put((rank, got))
    td.destroy_process_group()


def test_two_rank_max_of_timed_region():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res == {0: 11.0, 1: 11.0}


def test_single_process_needs_no_group():
    import bench
    os.environ.pop("WORLD_SIZE", None)
    assert bench.dist() == (0, 1, None)
    assert bench.max_over_ranks(3.5, None) == 3.5
