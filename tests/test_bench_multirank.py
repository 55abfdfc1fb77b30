"""The N > 1 path of bench.py on CPU: world_size 2 over gloo (the layer itself has no exchange
step, so ranks are independent replicas and only the timing reduction crosses ranks)."""
import importlib.util
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench = _bench()
        ws, r, local = bench.dist_setup(None)
        # rank r "timed" 10 + 5 r ms: every rank must see the slowest one
        ms = bench.max_over_ranks(10.0 + 5.0 * r, dist, "cpu")
        value = bench.job_throughput(1e9, 4, ms, ws)
        out.put((r, ws, local, ms, value))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, ws, local, ms, value) in enumerate(res):
        assert (rank, ws, local) == (r, world, r)
        assert ms == pytest.approx(15.0)  # max of 10 and 15
        # 2 replicas x 4 steps x 1 GB in 15 ms
        assert value == pytest.approx(2 * 4 * 1e9 / 15e-3 / 1e9)


def test_single_rank_is_identity():
    bench = _bench()
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_throughput(2e9, 10, 20.0, 1) == pytest.approx(2e9 * 10 / 0.02 / 1e9)
