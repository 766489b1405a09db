"""Replica sharding across processes, on the CPU with the gloo backend (world size 2): each
rank draws different canvases, the job time is the slowest rank's, and throughput counts every
rank's canvases."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from discrete_diffusion_text_gb300 import replicas


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle import dgoracle as O

        seed = replicas.replica_seed(4, rank, 0)
        canvas = torch.from_numpy(O.initial_canvas(2, 64, 4096, seed))
        gathered = [torch.zeros_like(canvas) for _ in range(world)]
        dist.all_gather(gathered, canvas)
        t = replicas.max_over_ranks(1.0 + rank)
        if rank == 0:
            q.put((bool(torch.equal(gathered[0], gathered[1])), t))
    finally:
        dist.destroy_process_group()


def test_replicas_draw_distinct_canvases_and_take_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    same, t = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert not same
    assert t == 2.0


def test_seeds_and_throughput():
    seeds = {replicas.replica_seed(1, r, s) for r in range(8) for s in range(100)}
    assert len(seeds) == 800
    assert replicas.job_throughput(4, 256, 2, 12, 0.01) == pytest.approx(4 * 256 * 2 * 12 / 0.01)
    assert replicas.max_over_ranks(3.5) == 3.5  # no process group: identity
