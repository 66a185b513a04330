"""The allocation-free attention entry point (for callers that cannot
allocate device memory: code under another framework's memory pool, plugins
that do not own the process allocator, paths that ban allocation after
start-up) against the regular entry point that takes a caller-owned
workspace, and against the oracle.

paged_decode_attn_e4m3_noalloc runs the same kernels with the same split
count; only the partials' buffer differs (the library's own scratch array
instead of the caller's workspace), so its output must be bit-identical to
paged_decode_attn_e4m3's, on two calls in a row (the second reuses the
scratch the first left behind).  Shapes cover the split (mma.sync) kernel,
the tcgen05 verify kernel (32 query rows per kv head at head_dim 128, with
fp16 and with FP8 scores) and a top-k list.

The file is named so that pytest collects it last; it also runs on its own
in a fresh process.  It calls the library through the C ABI with ctypes.
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

MAX_SCRATCH = 16 * 1024 * 1024   # KVQ_NOALLOC_SCRATCH_BYTES in include/kvq.h

# (workload, split count, FP8 scores)
CASES = {
    "tiny": (inputs.get("tiny"), 2, False),
    "tiny_verify": (inputs.get("tiny_verify"), 3, False),
    "decode": (inputs.get("decode"), 4, False),
    # MTP3 verify shape on the tcgen05 kernel: q_len 4 x 8 heads per kv head, head_dim 128
    "verify_tc": (inputs.Workload("noalloc_verify", 44, 1, 4, 4, 32, 4, 128, 0, "list:700,1500,93,2048",
                                  heavy_channels=4, calib_tokens=256), 0, False),
    "verify_tc_fp8": (inputs.Workload("noalloc_verify", 44, 1, 4, 4, 32, 4, 128, 0, "list:700,1500,93,2048",
                                      heavy_channels=4, calib_tokens=256), 0, True),
    # half of the sequences over a sorted top-256 list per (sequence, kv head)
    "topk": (inputs.Workload("noalloc_topk", 45, 1, 4, 1, 32, 4, 128, 0, "list:3000,700,1500,2100",
                             topk=256, topk_fraction=0.5, calib_tokens=256), 0, False),
}


@pytest.fixture(scope="module")
def lib():
    build.build()
    lib = kvq.load()
    V, Pp, i64, f32 = ctypes.c_void_p, ctypes.POINTER(kvq.AttnParams), ctypes.c_int64, ctypes.c_float
    lib.paged_decode_attn_e4m3_noalloc.argtypes = [V, V, V, i64, V, V, f32, f32, V, V, V, Pp, V, V]
    lib.paged_decode_attn_e4m3_noalloc.restype = ctypes.c_int
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _params(dp, num_splits, fp8_qk=False):
    return kvq.attn_params(dp.q, dp.k_cache.shape[1], dp.block_tables.shape[1], num_splits,
                           0 if dp.topk_idx is None else dp.topk_idx.shape[2], fp8_qk=fp8_qk)


def _noalloc(lib, dp, out, num_splits, fp8_qk=False):
    p = _params(dp, num_splits, fp8_qk)
    st = lib.paged_decode_attn_e4m3_noalloc(
        _ptr(dp.q), _ptr(dp.k_cache), _ptr(dp.v_cache), dp.k_cache.shape[0], _ptr(dp.block_tables),
        _ptr(dp.context_lens), ctypes.c_float(dp.k_scale), ctypes.c_float(dp.v_scale),
        _ptr(dp.topk_idx), _ptr(dp.topk_lens), _ptr(out), ctypes.byref(p), _ptr(dp.err),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, p


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_bit_identical_to_workspace_entry_point_twice(lib, name):
    w, S, fp8 = CASES[name]
    pr = P.host_problem(w)
    dp = G.device_problem(pr)
    p = _params(dp, S, fp8)
    assert kvq.workspace_bytes(p) <= MAX_SCRATCH
    if name.startswith("verify_tc"):    # the tcgen05 kernel's shape: head_dim 128, 9..64 rows per kv head
        assert w.head_dim == 128 and 8 < w.group * w.q_len <= 64
    ref = G.run_attention(dp, num_splits=S, fp8_qk=fp8)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    for _ in range(2):          # two calls in a row share (and reuse) the scratch buffer
        out = torch.full_like(dp.q, float("nan"))
        st, _ = _noalloc(lib, dp, out, S, fp8)
        assert st == 0
        torch.cuda.synchronize()
        assert dp.err.item() == 0
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"noalloc {name}: not bit-identical"
    # and against the oracle directly, from its own pools
    if name != "decode":        # the decode case's oracle run is covered by the full-size tests
        kc, vc, ks, vs = P.oracle_pools(pr)
        assert (ks, vs) == (dp.k_scale, dp.v_scale)
        want, flags = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, ks, vs,
                                       pr.topk_idx, pr.topk_lens, fp8_q=fp8)
        assert flags == 0
        G.assert_close(out.float().cpu().numpy(), want, f"noalloc {name} vs oracle")


def test_noalloc_refuses_problems_larger_than_its_scratch(lib):
    dp = G.device_problem(P.host_problem("tiny"))
    S = 100_000                 # workspace ~ 2*8*100000*64*4 bytes > 16 MiB
    p = kvq.attn_params(dp.q, 2, dp.block_tables.shape[1], S)
    assert kvq.workspace_bytes(p) > MAX_SCRATCH
    out = torch.zeros_like(dp.q)
    st, _ = _noalloc(lib, dp, out, S)
    assert st == -3             # KVQ_ERR_WORKSPACE, before any launch
    torch.cuda.synchronize()
    assert (out == 0).all()
