"""The N > 1 benchmark path on CPU with gloo, world size 2: replicas draw
their own seeded batches of identical shape, and the timing reduction takes
the slowest rank (no data-path collective exists to test)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from fp8_paged_kv_e4m3_gb300 import inputs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = bench.rank_workload(inputs.get("tiny"), rank)
        lay = inputs.page_layout(w)
        k = inputs.kv_tokens(w, 0, int(lay.lens.sum()), "k")
        slowest = bench.max_over_ranks(10.0 + rank, torch.device("cpu"), world)
        q.put((rank, float(k.float().sum()), lay.block_tables.shape, slowest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas():
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
    (r0, s0, shp0, m0), (r1, s1, shp1, m1) = res
    assert shp0 == shp1                 # same shapes on every rank
    assert s0 != s1                     # but each rank's own data
    assert m0 == m1 == 11.0             # both see the slowest rank's time


def test_aggregate_is_weak_scaling():
    g1, s1 = bench.aggregate(1_000_000_000, 32, 1, 10.0)
    g4, s4 = bench.aggregate(1_000_000_000, 32, 4, 10.0)
    assert g4 == pytest.approx(4 * g1) and s4 == pytest.approx(4 * s1)
    assert g1 == pytest.approx(100.0)
