"""Decode context parallelism on one GPU: every rank's share computed by the
library's partial call over the same pools, the partials gathered rank-major,
and the library's combine -- against the single-GPU oracle attention.  (The
exchange over a process group is the CPU gloo test's part.)"""
import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_e4m3_gb300 import build, dcp, inputs, kvq
from tests import _gpu as G
from tests import _problems as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    kvq.load()


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("shape", [("list:37,100,64", 8, 2, 64), ("list:4096,1000,2333", 32, 4, 128)])
def test_dcp_shares_combine_to_the_attention(world, shape):
    lens, Hq, Hkv, D = shape
    w = inputs.Workload("dcp_gpu", 52, 1, len(lens.split(",")), 1, Hq, Hkv, D, 0, lens, calib_tokens=128)
    pr = P.host_problem(w)
    dp = G.device_problem(pr, True)
    parts, p0 = [], None
    for r in range(world):
        bt, cl = dcp.shard_pages(pr.layout.block_tables, pr.layout.lens, world, r)
        p = kvq.attn_params(dp.q, Hkv, bt.shape[1], 2)
        ws = kvq.alloc_workspace(p, dp.q.device)
        kvq.paged_decode_attn_e4m3_partial(dp.q, dp.k_cache, dp.v_cache, G.to_dev(bt), G.to_dev(cl),
                                           dp.k_scale, dp.v_scale, ws, num_splits=2, err_flag=dp.err)
        parts.append(ws)
        p0 = p
    ws_g, p_g = dcp.gather_partials(None, p0, world, parts=parts)
    out = kvq.lse_combine(ws_g, torch.empty_like(dp.q), p_g)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    kc, vc, ks, vs = P.oracle_pools(pr, True, (dp.k_scale, dp.v_scale))
    ref, _ = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, ks, vs)
    G.assert_close(out.float().cpu().numpy(), ref, f"DCP x{world} {lens}")


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("shape", [("list:37,100,64", 8, 2, 64), ("list:4096,1000,2333", 32, 4, 128)])
def test_dcp_verify_window_rows_combine_to_the_attention(world, shape):
    """MTP verify (q_len 4, causal inside the window) over DCP: every rank's
    window rows as one-row sequences (`shard_window_rows`), the library's
    partial call, the rank-major gather and the library's combine, written
    straight into the [B][q_len][Hq][D] output."""
    lens, Hq, Hkv, D = shape
    w = inputs.Workload("dcp_gpu_verify", 54, 1, len(lens.split(",")), 4, Hq, Hkv, D, 0, lens, calib_tokens=128)
    pr = P.host_problem(w)
    dp = G.device_problem(pr, True)
    B, q_len = dp.q.shape[0], dp.q.shape[1]
    rows = dp.q.reshape(B * q_len, 1, Hq, D)
    parts, p0 = [], None
    for r in range(world):
        bt, cl = dcp.shard_window_rows(pr.layout.block_tables, pr.layout.lens, q_len, world, r)
        p = kvq.attn_params(rows, Hkv, bt.shape[1], 2)
        ws = kvq.alloc_workspace(p, dp.q.device)
        kvq.paged_decode_attn_e4m3_partial(rows, dp.k_cache, dp.v_cache, G.to_dev(bt), G.to_dev(cl),
                                           dp.k_scale, dp.v_scale, ws, num_splits=2, err_flag=dp.err)
        parts.append(ws)
        p0 = p
    ws_g, p_g = dcp.gather_partials(None, p0, world, parts=parts)
    out = torch.empty_like(dp.q)
    kvq.lse_combine(ws_g, out.view(B * q_len, 1, Hq, D), p_g)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    kc, vc, ks, vs = P.oracle_pools(pr, True, (dp.k_scale, dp.v_scale))
    ref, _ = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, ks, vs)
    G.assert_close(out.float().cpu().numpy(), ref, f"DCP verify x{world} {lens}")

