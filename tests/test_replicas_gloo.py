"""The multi-replica path of the benchmark on CPU: two gloo ranks.

On a node the benchmark runs one independent replica per GPU (tokens are
independent, so nothing is exchanged on the data path); the only collectives are the
barrier around the timed region and the maximum of the ranks' times.  Here two CPU
processes check that every rank gets the slowest rank's time, that the whole-job
throughput counts every replica's tokens over that time, and that the replicas draw
different activations from the same workload recipe.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from synth import CONFIGS, make_layer
    my_ms = [12.5, 30.25][rank]
    dist.barrier()
    got = bench.max_over_ranks(dist, my_ms, torch.device("cpu"))
    c = dict(CONFIGS["tiny"])
    L = make_layer(**{**c, "seed": c.get("seed", 0) + rank})
    q.put((rank, got, bench.job_tokens_per_s(L.T, 10, world, got), L.x[:2].copy()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_replicas_take_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = {}
    for _ in range(world):
        rank, got, value, x = q.get(timeout=120)
        out[rank] = (got, value, x)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in range(world):
        got, value, _ = out[rank]
        assert got == 30.25
        assert value == pytest.approx(64 * 10 * 2 / 0.03025)
    assert not np.array_equal(out[0][2], out[1][2])  # replicas draw their own activations

