"""Decode context parallelism on CPU: the page sharding, and the exchange
over two gloo ranks -- each rank's oracle partials of its own pages,
all-gathered into one workspace, combine to the single-rank attention.  The
same for MTP verify windows (q_len 4, causal inside the window), whose rows
are sharded as one-row sequences by `shard_window_rows`."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from fp8_paged_kv_e4m3_gb300 import build, dcp, inputs, kvq
from tests import _problems as P


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    kvq.load()


def _problem():
    w = inputs.Workload("dcp", 51, 1, 3, 1, 8, 2, 64, 0, "list:37,100,64", calib_tokens=64)
    return P.host_problem(w)


@pytest.mark.parametrize("world", [1, 2, 3, 4])
def test_shards_cover_every_page_once(world):
    pr = _problem()
    bt, lens = pr.layout.block_tables, pr.layout.lens
    shards = [dcp.shard_pages(bt, lens, world, r) for r in range(world)]
    for b in range(bt.shape[0]):
        n = (int(lens[b]) + 3) // 4
        pages = np.concatenate([s[0][b][s[0][b] >= 0] for s in shards])
        assert np.array_equal(pages, bt[b, :n])                  # in order, each once
        assert sum(int(s[1][b]) for s in shards) == int(lens[b])
        assert all(int(s[1][b]) > 0 for s in shards)


def test_shard_refuses_a_sequence_shorter_than_the_world():
    pr = _problem()
    with pytest.raises(ValueError):
        dcp.shard_pages(pr.layout.block_tables, pr.layout.lens, 11, 0)   # 37 tokens = 10 pages


def _rank_partials(pr, world, rank, S):
    kc, vc, ks, vs = P.oracle_pools(pr)
    bt, cl = dcp.shard_pages(pr.layout.block_tables, pr.layout.lens, world, rank)
    o, m, l, flags = oracle.attention_partials(pr.q, kc, vc, bt, cl, S, ks, vs)
    assert flags == 0
    p = kvq.AttnParams(pr.w.batch, 1, pr.w.num_q_heads, pr.w.num_kv_heads, pr.w.head_dim, S, bt.shape[1], 0,
                       0.0, 0, 0)
    ws = torch.zeros((kvq.workspace_bytes(p) + 3) // 4, dtype=torch.float32)
    vo, vm, vl = kvq.workspace_views(ws, p)
    vo.copy_(torch.from_numpy(o))
    vm.copy_(torch.from_numpy(m))
    vl.copy_(torch.from_numpy(l))
    return ws, p


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        kvq.load()
        pr = _problem()
        ws, p = _rank_partials(pr, world, rank, 2)
        ws_g, p_g = dcp.gather_partials(ws, p, world)
        go, gm, gl = kvq.workspace_views(ws_g, p_g)
        out = oracle.combine(go.double().numpy(), gm.double().numpy(), gl.double().numpy())
        q.put((rank, p_g.num_splits, out))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_exchange_partials():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=180) for _ in range(world)), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    pr = _problem()
    kc, vc, ks, vs = P.oracle_pools(pr)
    ref, _ = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, ks, vs)
    for rank, S_total, out in res:
        assert S_total == world * 2
        # out is [B][Hq][q_len][D]; the oracle's [B][q_len][Hq][D]
        np.testing.assert_allclose(out.transpose(0, 2, 1, 3), ref, rtol=1e-6, atol=1e-7)


def test_gather_without_a_group_is_rank_major():
    """One process holding every rank's workspace (the layout the combine reads)."""
    pr = _problem()
    parts, p = zip(*[_rank_partials(pr, 3, r, 2) for r in range(3)])
    ws_g, p_g = dcp.gather_partials(None, p[0], 3, parts=list(parts))
    assert p_g.num_splits == 6
    go, gm, gl = kvq.workspace_views(ws_g, p_g)
    for r in range(3):
        o, m, l = kvq.workspace_views(parts[r], p[0])
        assert torch.equal(go[:, :, :, 2 * r:2 * r + 2], o)
        assert torch.equal(gm[:, :, :, 2 * r:2 * r + 2], m)
    out = oracle.combine(go.double().numpy(), gm.double().numpy(), gl.double().numpy())
    kc, vc, ks, vs = P.oracle_pools(pr)
    ref, _ = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, ks, vs)
    np.testing.assert_allclose(out.transpose(0, 2, 1, 3), ref, rtol=1e-6, atol=1e-7)


def _verify_problem():
    w = inputs.Workload("dcp_verify", 53, 1, 3, 4, 8, 2, 64, 0, "list:37,100,64", calib_tokens=64)
    return P.host_problem(w)


@pytest.mark.parametrize("q_len", [1, 2, 4])
@pytest.mark.parametrize("world", [1, 2, 3])
def test_window_rows_see_each_key_of_their_row_once(world, q_len):
    """Row i of a window attends positions 0 .. L - q_len + i: over the ranks,
    each of them exactly once, and nothing past it."""
    pr = _problem()
    bt, lens = pr.layout.block_tables, pr.layout.lens
    page_shards = [dcp.shard_pages(bt, lens, world, r) for r in range(world)]
    rows = [dcp.shard_window_rows(bt, lens, q_len, world, r) for r in range(world)]
    for b in range(bt.shape[0]):
        L = int(lens[b])
        for i in range(q_len):
            seen, first = [], 0
            for r in range(world):
                rbt, rlen = rows[r]
                n = int(rlen[b * q_len + i])
                assert n >= 1
                assert np.array_equal(rbt[b * q_len + i], page_shards[r][0][b])   # the rank's pages of b
                seen.append(first + np.arange(n))
                first += int(page_shards[r][1][b])
            assert np.array_equal(np.concatenate(seen), np.arange(L - q_len + i + 1))


def test_window_rows_refuse_a_rank_past_the_window_start():
    pr = _problem()
    lens = np.array([5, 100, 64], dtype=np.int32)
    dcp.shard_pages(pr.layout.block_tables, lens, 2, 1)      # every rank holds a page ...
    with pytest.raises(ValueError, match="window row"):       # ... but rank 1 only position 4 of the first
        dcp.shard_window_rows(pr.layout.block_tables, lens, 4, 2, 1)


def _rank_window_partials(pr, world, rank, S):
    B, q_len, Hq, D = pr.q.shape
    kc, vc, ks, vs = P.oracle_pools(pr)
    bt, cl = dcp.shard_window_rows(pr.layout.block_tables, pr.layout.lens, q_len, world, rank)
    rows = np.ascontiguousarray(pr.q.reshape(B * q_len, 1, Hq, D))
    o, m, l, flags = oracle.attention_partials(rows, kc, vc, bt, cl, S, ks, vs)
    assert flags == 0
    p = kvq.AttnParams(B * q_len, 1, Hq, pr.w.num_kv_heads, D, S, bt.shape[1], 0, 0.0, 0, 0)
    ws = torch.zeros((kvq.workspace_bytes(p) + 3) // 4, dtype=torch.float32)
    vo, vm, vl = kvq.workspace_views(ws, p)
    vo.copy_(torch.from_numpy(o))
    vm.copy_(torch.from_numpy(m))
    vl.copy_(torch.from_numpy(l))
    return ws, p


def _verify_worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        kvq.load()
        pr = _verify_problem()
        ws, p = _rank_window_partials(pr, world, rank, 2)
        ws_g, p_g = dcp.gather_partials(ws, p, world)
        go, gm, gl = kvq.workspace_views(ws_g, p_g)
        out = oracle.combine(go.double().numpy(), gm.double().numpy(), gl.double().numpy())
        q.put((rank, out))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_exchange_verify_window_partials():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_verify_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=180) for _ in range(world)), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    pr = _verify_problem()
    B, q_len, Hq, D = pr.q.shape
    kc, vc, ks, vs = P.oracle_pools(pr)
    ref, _ = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, ks, vs)
    for rank, out in res:
        # out is [B * q_len][Hq][1][D] (one-row sequences); the oracle's [B][q_len][Hq][D]
        got = out.transpose(0, 2, 1, 3).reshape(B, q_len, Hq, D)
        np.testing.assert_allclose(got, ref, rtol=1e-6, atol=1e-7)

