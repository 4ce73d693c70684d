"""The benchmark's multi-rank aggregation on the CPU: two gloo ranks, each
with its own (different) timed seconds, must both report the whole job's
tokens over the slowest rank's time.  No GPU is used."""

import importlib.util
import os
import socket

import pytest
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


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        my_seconds = [0.5, 2.0][rank]
        value, t = b.whole_job_rate(my_seconds, tokens_per_step=64, steps=10, world=world, dist=dist, device="cpu")
        dist.barrier()
        out[rank] = (value, t)
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_and_all_tokens():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0] == res[1]
    value, t = res[0]
    assert t == 2.0
    assert value == pytest.approx(64 * 10 * 2 / 2.0)


def test_single_rank_is_its_own_time():
    b = _bench()
    value, t = b.whole_job_rate(0.25, tokens_per_step=64, steps=4, world=1)
    assert t == 0.25 and value == pytest.approx(64 * 4 / 0.25)
