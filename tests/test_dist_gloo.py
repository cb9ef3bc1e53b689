"""The multi-process path of bench.py on CPU: two gloo ranks (spawned, 127.0.0.1).

The library's path has no exchange step, so several GPUs run independent
replicas (weak scaling); what is shared between ranks is the barrier, the
max-over-ranks step time and the sum of the work, and the reference arm runs
on rank 0 alone.
"""
import multiprocessing as mp
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    d = bench.Dist()
    try:
        d.barrier()
        out = {"rank": d.rank, "world": d.world, "max": d.max(rank + 1.0),
               "sum": d.sum(rank + 1.0),
               # rank r did (r + 1) TFLOP per step at (2 + r) ms per step
               "agg": bench.aggregate(d, (rank + 1) * 1e12, 10, 2.0 + rank)}
        if rank != 0:  # the reference arm: only rank 0 works, the others exit 0
            class A:
                config, sweep, steps, warmup, reference_budget_s, gpus = 0, 0, 1, 1, 20.0, world
            out["reference_rc"] = bench.run_reference(A, d)
        d.barrier()
        q.put(out)
    finally:
        d.close()


@pytest.mark.parametrize("world", [2])
def test_gloo_ranks_share_max_time_and_summed_work(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    outs = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    outs.sort(key=lambda o: o["rank"])
    for o in outs:
        assert o["world"] == world
        assert o["max"] == world
        assert o["sum"] == world * (world + 1) / 2
        value, ms = o["agg"]
        assert ms == 2.0 + (world - 1)                  # the slowest rank
        assert value == pytest.approx(3e12 / (ms * 1e-3) / 1e12)  # all ranks' work / that time
    assert all(o["reference_rc"] == 0 for o in outs[1:])
