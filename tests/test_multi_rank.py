"""The multi-replica timing path of bench.py on CPU: two gloo ranks, each
with its own step time, combine into one whole-job throughput that counts
both ranks' tokens over the slowest rank's time.  (On GPUs each rank runs
an independent replica of the layer; the layer itself has no exchange.)"""
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
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)

    def reduce_max(v):
        t = torch.tensor([v], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    ms_local = 100.0 + 50.0 * rank          # rank 1 is the slow one
    value, ms = bench.aggregate(world, 4096, 10, ms_local, reduce_max)
    dist.barrier()
    q.put((rank, value, ms))
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_over_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    old = os.environ.get("PYTHONPATH", "")
    os.environ["PYTHONPATH"] = root + (os.pathsep + old if old else "")
    try:
        procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
    finally:
        os.environ["PYTHONPATH"] = old
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, value, ms in res:
        assert ms == pytest.approx(150.0)
        assert value == pytest.approx(2 * 4096 * 10 / 0.150)


def test_single_rank_aggregate_has_no_collective():
    import bench
    value, ms = bench.aggregate(1, 4096, 10, 80.0, reduce_max=None)
    assert ms == 80.0 and value == pytest.approx(4096 * 10 / 0.080)
