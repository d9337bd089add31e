"""The N > 1 replica path of bench.py on CPU: two gloo ranks, the barrier,
the max over ranks of the timed region, the whole-job value, and the
reference arm, which only rank 0 runs."""
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


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        b.barrier(world)
        local_ms = [10.0, 12.5][rank]  # rank 1 is the slower replica
        worst = b.max_over_ranks(local_ms, world, device="cpu")
        value = b.job_tokens_per_s(world, 7168, 30, worst)
        # the reference arm: rank 1 returns at once, without work or output
        done = True
        if rank == 1:
            b.run_reference(None, world, rank, 0)
        out[rank] = (worst, value, done)
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_aggregate_like_the_bench():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(100)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0][0] == res[1][0] == 12.5
    expected = 2 * 7168 * 30 / 0.0125
    assert res[0][1] == pytest.approx(expected) and res[1][1] == pytest.approx(expected)
    assert res[1][2]


def test_single_rank_value():
    b = _bench()
    assert b.max_over_ranks(3.0, 1) == 3.0
    assert b.job_tokens_per_s(1, 100, 10, 1000.0) == pytest.approx(1000.0)
