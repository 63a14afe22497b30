"""The N > 1 host path of bench.py on CPU: two gloo ranks on 127.0.0.1.

Replicas only (no data-path collective): each rank times its own steps, the
slowest rank's time is taken with one all-reduce(MAX), the whole-job value is
N x steps x work / that time, and the reference arm runs on rank 0 only."""
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


def _worker(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        import bench
        bench.barrier(ws)
        t = bench.max_over_ranks(ws, 10.0 + 5.0 * rank)           # rank 1 is the slow one
        value = bench.aggregate_value(ws, steps=4, step_work=2.5e9, t_max_ms=t)

        class Args:
            workload, steps, warmup = "llama7b_layer_decode", 1, 0
        ran = bench.run_reference(Args(), ws, rank) if rank != 0 else None  # non-zero ranks return at once
        out.put((rank, t, value, ran))
        bench.barrier(ws)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    [p.start() for p in procs]
    [p.join(120) for p in procs]
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, value, ran in res:
        assert t == 15.0                                       # max over ranks, seen by both
        assert value == pytest.approx(2 * 4 * 2.5e9 / 15e-3 / 1e9)
        assert ran is None


def test_single_rank_value():
    import bench
    assert bench.max_over_ranks(1, 3.0) == 3.0
    assert bench.aggregate_value(1, 10, 1e9, 1000.0) == pytest.approx(10.0)
