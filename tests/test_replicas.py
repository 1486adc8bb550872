"""The bench's multi-GPU path: independent replicas, one per rank.

The decode shards by sequence with no exchange step, so ``bench.py`` under
torchrun runs one replica per rank; the only cross-rank operations are the
barriers around the timed region and the max over ranks of the elapsed time.
These tests run that host logic as two gloo ranks on the CPU.
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout
from types import SimpleNamespace

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, results):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist

    w, r, local = bench.dist_setup("gloo")
    try:
        bench.barrier(w)
        # rank r "took" 100 + 60 r ms for 10 steps of 64 sequences each
        ms_per_step, rate = bench.replica_rate(100.0 + 60.0 * r, w, 64, 10)
        # the reference arm runs on rank 0 alone; other ranks print nothing
        buf = io.StringIO()
        if r != 0:
            with redirect_stdout(buf):
                bench.run_reference(SimpleNamespace(steps=3, warmup=3), None, w, r)
        bench.barrier(w)
        results.put((r, w, local, ms_per_step, rate, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_replica_rate_single_rank():
    ms, rate = bench.replica_rate(250.0, 1, 32, 10)
    assert ms == pytest.approx(25.0)
    assert rate == pytest.approx(32 / 0.025)


def test_two_gloo_replicas_take_the_slowest_rank():
    world = 2
    ctx = mp.get_context("spawn")
    results = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    got = [results.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    got.sort()
    slowest_ms = 100.0 + 60.0 * (world - 1)
    for r, (rank, w, local, ms_per_step, rate, printed) in enumerate(got):
        assert (rank, w, local) == (r, world, r)
        # every rank agrees on the max over ranks ...
        assert ms_per_step == pytest.approx(slowest_ms / 10)
        # ... and the rate counts the sequences of all ranks
        assert rate == pytest.approx(world * 64 / (slowest_ms / 10 / 1e3))
        assert printed == ""
