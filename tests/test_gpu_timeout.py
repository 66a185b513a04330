"""The give-up path of the decode attention kernel's bounded waits, run on
the GPU without faulting or hanging it.

A pipeline wait that runs out (PR "[Model][SM70][FP8] Integrate calibrated
E4M3 QSA KV capacity path", sections Purpose and Validation boundary: the
path fails closed instead of producing a result it cannot vouch for) must
raise KVQ_DEV_TIMEOUT, let every bulk copy it issued land, mark its split
partials empty (m = -inf, l = 0) and return, leaving the context usable.

No real wait runs out on a healthy GPU, so a test-only build of the split
kernel's translation unit (define KVQ_TEST_STALL_CONSUMERS, never set in the
library's own build) makes the consumer warps first wait, with a 20 us
bound, on a barrier that only they could complete.  The wait therefore
always gives up; the producers, blocked on ring slots that are never
released, see the abort and stop; both drain their copies.  The case has
far more stages than the ring holds, so the producers do block.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_e4m3_gb300 import build, inputs, kvq
from tests import _gpu as G
from tests import _problems as P

pytestmark = pytest.mark.gpu

STALL_NS = 20000   # the consumers' bound on the stalled wait


@pytest.fixture(scope="module")
def stall_lib():
    build.build()
    kvq.load()
    path = build.build_variant("stall_consumers", {"KVQ_TEST_STALL_CONSUMERS": f"{STALL_NS}ull"})
    return kvq.load(path)


def _case():
    # head_dim 128, 8 query rows per kv head: the split kernel with 3 ring stages
    # of 16 pages; one split of 750 pages is 47 stages
    return inputs.Workload("timeout", 43, 1, 2, 1, 8, 2, 128, 1, "list:3000,517", calib_tokens=128)


def _call_partial(lib, dp, ws, p):
    return lib.paged_decode_attn_e4m3_partial(
        ctypes.c_void_p(dp.q.data_ptr()), ctypes.c_void_p(dp.k_cache.data_ptr()),
        ctypes.c_void_p(dp.v_cache.data_ptr()), dp.k_cache.shape[0],
        ctypes.c_void_p(dp.block_tables.data_ptr()), ctypes.c_void_p(dp.context_lens.data_ptr()),
        ctypes.c_float(dp.k_scale), ctypes.c_float(dp.v_scale), None, None,
        ctypes.c_void_p(ws.data_ptr()), ws.numel() * 4, ctypes.byref(p),
        ctypes.c_void_p(dp.err.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("num_splits", [1, 3])
def test_timeout_sets_flag_drains_and_empties_partials(stall_lib, num_splits):
    pr = P.host_problem(_case())
    dp = G.device_problem(pr)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    p = kvq.attn_params(dp.q, dp.k_cache.shape[1], dp.block_tables.shape[1], num_splits)
    ws = kvq.alloc_workspace(p, dp.q.device)
    ws.fill_(float("nan"))
    st = _call_partial(stall_lib, dp, ws, p)
    assert st == 0, "the launch itself must succeed"
    torch.cuda.synchronize()           # returns: nothing hung
    assert dp.err.item() & kvq.DEV_TIMEOUT, f"err_flag {dp.err.item()}: no timeout reported"
    o, m, l = kvq.workspace_views(ws, p)
    assert torch.isneginf(m).all(), "a split that gave up must write m = -inf"
    assert (l == 0).all(), "a split that gave up must write l = 0"
    # the combine gives such splits zero weight: every row without keys is 0
    out = torch.full_like(dp.q, float("nan"))
    stall_lib.kvq_lse_combine(ctypes.c_void_p(ws.data_ptr()), ws.numel() * 4, ctypes.c_void_p(out.data_ptr()),
                              ctypes.byref(p), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert (out == 0).all()


def test_context_usable_after_timeout(stall_lib):
    """After the give-up, the default library on the same context still gives
    the oracle's result."""
    pr = P.host_problem(_case())
    dp = G.device_problem(pr)
    p = kvq.attn_params(dp.q, dp.k_cache.shape[1], dp.block_tables.shape[1], 2)
    ws = kvq.alloc_workspace(p, dp.q.device)
    assert _call_partial(stall_lib, dp, ws, p) == 0
    torch.cuda.synchronize()
    assert dp.err.item() & kvq.DEV_TIMEOUT
    dp.err.zero_()
    got = G.run_attention(dp, num_splits=2).float().cpu().numpy()
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    kc, vc, ks, vs = P.oracle_pools(pr)
    assert np.array_equal(kc, dp.k_cache.cpu().numpy()) and np.array_equal(vc, dp.v_cache.cpu().numpy())
    ref, _ = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, ks, vs)
    G.assert_close(got, ref, "after timeout")


@pytest.fixture(scope="module")
def stall_cluster_lib():
    build.build()
    kvq.load()
    path = build.build_variant("stall_consumers_cluster", {"KVQ_TEST_STALL_CONSUMERS": f"{STALL_NS}ull"},
                               sources=("kvq_attn.cu", "kvq_attn_cm.cu"))
    return kvq.load(path)


def test_timeout_in_the_cluster_merge(stall_cluster_lib):
    """The full call's cluster-merging instances (here 3 splits of each of the 2
    x 2 (sequence, kv head) groups, one cluster each): every CTA gives up, marks
    its partials empty, and still passes its cluster's barrier exactly once, so
    the call returns, and the merge gives every row 0."""
    pr = P.host_problem(_case())
    dp = G.device_problem(pr)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    p = kvq.attn_params(dp.q, dp.k_cache.shape[1], dp.block_tables.shape[1], 3)
    assert kvq.attn_launches(p, True) == 1, "this shape takes the cluster merge"
    ws = kvq.alloc_workspace(p, dp.q.device)
    ws.fill_(float("nan"))
    out = torch.full_like(dp.q, float("nan"))
    st = stall_cluster_lib.paged_decode_attn_e4m3(
        ctypes.c_void_p(dp.q.data_ptr()), ctypes.c_void_p(dp.k_cache.data_ptr()),
        ctypes.c_void_p(dp.v_cache.data_ptr()), dp.k_cache.shape[0],
        ctypes.c_void_p(dp.block_tables.data_ptr()), ctypes.c_void_p(dp.context_lens.data_ptr()),
        ctypes.c_float(dp.k_scale), ctypes.c_float(dp.v_scale), None, None,
        ctypes.c_void_p(ws.data_ptr()), ws.numel() * 4, ctypes.c_void_p(out.data_ptr()), ctypes.byref(p),
        ctypes.c_void_p(dp.err.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, "the launch itself must succeed"
    torch.cuda.synchronize()           # returns: no CTA was left waiting at its cluster barrier
    assert dp.err.item() & kvq.DEV_TIMEOUT, f"err_flag {dp.err.item()}: no timeout reported"
    o, m, l = kvq.workspace_views(ws, p)
    assert torch.isneginf(m).all() and (l == 0).all()
    assert (out == 0).all()

