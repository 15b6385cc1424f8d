"""The benchmark's multi-rank plumbing (one replica per rank, barrier, max over
ranks) on two gloo ranks on the CPU, including a rank that dies before the
barrier: the survivor must get an error from its timed-out collective rather
than wait forever."""
import datetime
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, mode, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", timeout=datetime.timedelta(seconds=5))
    try:
        if mode == "ok":
            bench.barrier(world)
            q.put((rank, bench.max_over_ranks(10.0 + rank, world)))
        else:
            if rank == 1:
                os._exit(3)          # dies between steps, nothing in flight
            try:
                bench.barrier(world)
                q.put((rank, "no error"))
            except Exception as e:   # gloo reports the lost peer / timeout
                q.put((rank, "error:" + type(e).__name__))
    finally:
        if mode == "ok":
            dist.destroy_process_group()


def _run(mode):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, mode, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(60)
    out = {}
    while not q.empty():
        r, v = q.get()
        out[r] = v
    for p in procs:
        if p.is_alive():
            p.kill()
    return out, [p.exitcode for p in procs]


def test_two_ranks_take_the_max():
    out, codes = _run("ok")
    assert codes == [0, 0]
    assert out == {0: 11.0, 1: 11.0}


def test_lost_rank_is_reported_not_waited_for():
    out, codes = _run("lost")
    assert codes[1] == 3
    assert 0 in out and out[0].startswith("error:")
