"""Host-side logic of bench.py across ranks, on CPU with the gloo backend (world size 2):
the max-over-ranks timing, the weak-scaling aggregate and the rank-0-only reference arm."""

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


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        bench.barrier(world)
        t = bench.max_over_ranks(10.0 + 5.0 * rank, world, device="cpu")
        v = bench.weak_scaling_value(world, 4096, t)
        ref = bench.run_reference(type("A", (), {"steps": 1, "warmup": 0, "gpus": world})(), world, rank) \
            if rank == 1 else "skipped"
        results[rank] = (t, v, ref)
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_and_aggregate():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(results)
    for rank in range(world):
        t, v, _ = res[rank]
        assert t == 15.0                          # the slowest rank's time on every rank
        assert v == pytest.approx(2 * 4096 / 0.015)
    assert res[1][2] is None                      # the reference arm does no work off rank 0
