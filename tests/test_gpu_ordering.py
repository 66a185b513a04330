"""Ordering of decode attention behind this step's append in the same stream.

The attention kernels start under programmatic dependent launch while the
append still runs; without a top-k list the split kernel's producers copy the
cache pages of positions below L - q_len before waiting for the append, and
everything else (q, the pages holding this step's positions) after.  These
tests launch append and attention back to back, with no other work between
them, over many steps whose new keys dominate the scores and whose new values
change every step, so that a page read before the append had written it would
show in the output.  Contexts end at every offset inside a page, and the
window of a verify step spans two pages."""
import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_e4m3_gb300 import build, inputs, kvq
from tests import _gpu as G
from tests import _problems as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    kvq.load()


def _steps(lens, q_len, e4m3, S, strict, mma_sync=True, iters=12, topk=0, D=64):
    kw = dict(topk=topk, topk_fraction=1.0) if topk else {}
    w = inputs.Workload("order", 21, 1, len(lens), q_len, 8, 2, D, 0,
                        "list:" + ",".join(map(str, lens)), calib_tokens=64, **kw)
    pr = P.host_problem(w)
    dp = G.device_problem(pr, e4m3)
    rng = np.random.default_rng(4)
    B, Gq = len(lens), w.num_q_heads // w.num_kv_heads
    rows = pr.step_rows                                   # this step's tokens, (b, i) order
    slots = G.to_dev(pr.step_slots)
    p = kvq.AttnParams(B, q_len, w.num_q_heads, w.num_kv_heads, w.head_dim, S, dp.block_tables.shape[1],
                       0 if dp.topk_idx is None else dp.topk_idx.shape[2], 0.0, 0,
                       kvq._flags(False, mma_sync, False, strict))
    ws = kvq.alloc_workspace(p, dp.q.device)
    out = torch.empty_like(dp.q)
    ti, tl = (dp.topk_idx, dp.topk_lens) if topk else (None, None)
    for it in range(iters):
        # new keys along the query of the group's first head (they dominate), new values at random
        knew = np.empty((len(rows), w.num_kv_heads, w.head_dim), np.float16)
        for n, (b, i) in enumerate((b, i) for b in range(B) for i in range(q_len)):
            for g in range(w.num_kv_heads):
                knew[n, g] = (pr.q[b, i, g * Gq].astype(np.float32) * (2.0 + 0.1 * it)).astype(np.float16)
        vnew = (rng.standard_normal((len(rows), w.num_kv_heads, w.head_dim)) * 3).astype(np.float16)
        pr.k_tok[rows] = knew
        pr.v_tok[rows] = vnew
        kd, vd = G.to_dev(knew), G.to_dev(vnew)           # copies: fully ordered before the append
        if e4m3:
            kvq.kv_append_e4m3(kd, vd, slots, dp.k_cache, dp.v_cache, dp.k_scale, dp.v_scale, dp.err)
            kvq.paged_decode_attn_e4m3(dp.q, dp.k_cache, dp.v_cache, dp.block_tables, dp.context_lens,
                                       dp.k_scale, dp.v_scale, ws, out, ti, tl, S, err_flag=dp.err,
                                       mma_sync=mma_sync, strict_order=strict)
        else:
            kvq.kv_append_fp16(kd, vd, slots, dp.k_cache, dp.v_cache, dp.err)
            kvq.paged_decode_attn_fp16(dp.q, dp.k_cache, dp.v_cache, dp.block_tables, dp.context_lens,
                                       ws, out, ti, tl, S, err_flag=dp.err, mma_sync=mma_sync,
                                       strict_order=strict)
        got = out.float().cpu().numpy()
        assert dp.err.item() == 0
        kc, vc, ks, vs = P.oracle_pools(pr, e4m3, (dp.k_scale, dp.v_scale) if e4m3 else None)
        ref, _ = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, ks, vs,
                                  pr.topk_idx if topk else None, pr.topk_lens if topk else None)
        G.assert_close(got, ref, f"step {it} lens {lens} q_len {q_len} e4m3={e4m3} S={S} strict={strict}")


# contexts ending at each offset inside a page; long enough for several stages per split
LENS = [517, 518, 519, 520, 133]


@pytest.mark.parametrize("q_len", [1, 3, 4])
@pytest.mark.parametrize("S", [1, 3])
@pytest.mark.parametrize("e4m3", [True, False])
def test_append_then_attention_back_to_back(q_len, S, e4m3):
    _steps(LENS, q_len, e4m3, S, strict=False)


@pytest.mark.parametrize("q_len", [1, 4])
def test_strict_order_gives_the_same_results(q_len):
    _steps(LENS, q_len, True, 2, strict=True, iters=4)


def test_topk_calls_wait_for_the_preceding_kernel():
    _steps([300, 260], 1, True, 2, strict=False, iters=6, topk=200)


def test_tcgen05_kernel_behind_the_append():
    _steps([517, 300], 4, True, 2, strict=False, mma_sync=False, iters=6, D=128)
