"""The allocation-free attention entry point (for callers that cannot
allocate device memory) against the regular entry point that takes a
caller-owned workspace.

The file is named so that pytest collects it last; it also runs on its own
in a fresh process.  It calls the library through the C ABI with ctypes.
"""
import ctypes

import numpy as np
import pytest
import torch

from fp8_paged_kv_e4m3_gb300 import build, kvq
from tests import _gpu as G
from tests import _problems as P

pytestmark = pytest.mark.gpu

MAX_SCRATCH = 16 * 1024 * 1024   # KVQ_NOALLOC_SCRATCH_BYTES in include/kvq.h


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


def _noalloc(lib, dp, out, num_splits):
    p = kvq.attn_params(dp.q, dp.k_cache.shape[1], dp.block_tables.shape[1], num_splits,
                        0 if dp.topk_idx is None else dp.topk_idx.shape[2])
    st = lib.paged_decode_attn_e4m3_noalloc(
        _ptr(dp.q), _ptr(dp.k_cache), _ptr(dp.v_cache), dp.k_cache.shape[0], _ptr(dp.block_tables),
        _ptr(dp.context_lens), ctypes.c_float(dp.k_scale), ctypes.c_float(dp.v_scale),
        _ptr(dp.topk_idx), _ptr(dp.topk_lens), _ptr(out), ctypes.byref(p), _ptr(dp.err),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, p


@pytest.mark.parametrize("name,S", [("tiny", 2), ("tiny_verify", 3), ("decode", 4)])
def test_noalloc_matches_workspace_entry_point_twice(lib, name, S):
    from fp8_paged_kv_e4m3_gb300 import inputs
    w = inputs.get(name)
    dp = G.device_problem(P.host_problem(w))
    ref = G.run_attention(dp, num_splits=S).float().cpu().numpy().astype(np.float64)
    for _ in range(2):          # two calls in a row share (and reuse) the scratch buffer
        out = torch.full_like(dp.q, float("nan"))
        st, p = _noalloc(lib, dp, out, S)
        assert st == 0
        torch.cuda.synchronize()
        assert dp.err.item() == 0
        G.assert_close(out.float().cpu().numpy(), ref, f"noalloc {name}")


def test_noalloc_refuses_problems_larger_than_its_scratch(lib):
    dp = G.device_problem(P.host_problem("tiny"))
    S = 100_000                 # workspace ~ 2*8*100000*64*4 bytes > 16 MiB
    p = kvq.attn_params(dp.q, 2, dp.block_tables.shape[1], S)
    assert kvq.workspace_bytes(p) > MAX_SCRATCH
    out = torch.zeros_like(dp.q)
    st, _ = _noalloc(lib, dp, out, S)
    assert st == -3             # KVQ_ERR_WORKSPACE, before any launch
    assert (out == 0).all()
