"""The full attention call's cluster merge: with up to 8 query rows per kv
head and up to 8 splits, the splits of each (sequence, kv head) run as one
thread-block cluster and merge their partials into the output themselves,
instead of a combine launch.  The merge is the combine kernel's own function
over the same workspace partials, so the output must be bit-identical to the
partial call followed by kvq_lse_combine, and match the oracle.  The split-K
partials and their log-sum-exp combine are PR "[Model][SM70] Calibrated E4M3
KV cache for Qwen4Exp QSA with MTP", section Status and history (the FP32
temporary output of the page-4 route)."""
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


def _oracle_out(dp):
    pr = dp.host
    kc, vc, ks, vs = P.oracle_pools(pr, dp.e4m3, (dp.k_scale, dp.v_scale) if dp.e4m3 else None)
    ref, _ = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, ks, vs,
                              pr.topk_idx, pr.topk_lens)
    return ref


def _check(dp, S, what):
    full = G.run_attention(dp, num_splits=S)
    ws, p = G.run_attention(dp, num_splits=S, partial=True)
    merged = kvq.lse_combine(ws, torch.empty_like(dp.q), p)
    torch.cuda.synchronize()
    assert dp.err.item() == 0, what
    assert torch.equal(full.view(torch.int16), merged.view(torch.int16)), what
    G.assert_close(full.float().cpu().numpy(), _oracle_out(dp), what)


# lengths with splits that hold no page (short sequences at 8 splits), contexts ending
# at every offset inside a page, and one sequence of several stages per split
LENS = "list:4,5,6,7,41,300,1029"


@pytest.mark.parametrize("e4m3", [True, False])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("q_len,Hq", [(1, 8), (4, 4), (3, 4)])
def test_cluster_merge_equals_partial_then_combine(e4m3, D, q_len, Hq):
    # Hq / Hkv * q_len <= 8 rows per kv head: the split kernel's cluster-merge instances
    w = inputs.Workload("cm", 51, 1, 7, q_len, Hq, 2, D, 0, LENS, outlier_channels=2, calib_tokens=64)
    dp = G.device_problem(P.host_problem(w), e4m3)
    for S in (1, 2, 3, 5, 8):
        _check(dp, S, f"e4m3={e4m3} D={D} q_len={q_len} S={S}")


def test_cluster_merge_with_topk_lists_and_the_combine_past_8_splits():
    w = inputs.Workload("cm", 52, 1, 6, 1, 8, 2, 128, 0, "list:700,33,512,9,260,1500", calib_tokens=64,
                        topk=96, topk_fraction=0.5)
    dp = G.device_problem(P.host_problem(w), True)
    for S in (4, 8, 9):   # 9 splits: the combine kernel
        _check(dp, S, f"top-k S={S}")


def test_cluster_merge_at_the_decode_shape():
    # 32 q / 4 kv heads, head_dim 128, q_len 1, split-K 4: the decode workload's shape
    w = inputs.Workload("cm", 53, 1, 6, 1, 32, 4, 128, 4, "list:4096,4093,517,1,2048,3333",
                        calib_tokens=128)
    dp = G.device_problem(P.host_problem(w), True)
    _check(dp, 4, "decode shape")
