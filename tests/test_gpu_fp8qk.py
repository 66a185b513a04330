"""GPU parity of the FP8 score variant (flag KVQ_ATTN_FP8_QK): the tcgen05
kernel with the query quantised to E4M3 per (sequence, kv head) and q k^T on
E4M3 tensor-core instructions, against the oracle's reading of the same
variant (oracle.attention(..., fp8_q=True)), which quantises the query in the
same binary32 steps; the scores then differ only by the order of the fp32
accumulation.  Outputs, FP32 split partials, top-k lists with NaN-filled
slots, scores that move the softmax reference, and ragged tails."""
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


def _oracle_out(dp, topk=True, fp8_q=True):
    pr = dp.host
    kc, vc, ks, vs = P.oracle_pools(pr, True, (dp.k_scale, dp.v_scale))
    out, _ = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, ks, vs,
                              pr.topk_idx if topk else None, pr.topk_lens if topk else None, fp8_q=fp8_q)
    return out


def _problem(lens, q_len, group, sentinel=P.SENTINEL, **kw):
    w = inputs.Workload("tc", 12, 1, len(lens), q_len, 2 * group, 2, 128, 0,
                        "list:" + ",".join(map(str, lens)), calib_tokens=64, heavy_channels=4, **kw)
    return G.device_problem(P.host_problem(w), True, sentinel=sentinel)


SHAPES = [
    ([300, 17, 129, 64], 4, 4),      # 16 rows; one-token tiles, exact 64/128 boundaries
    ([1000, 236, 33, 127], 4, 8),    # 32 rows (the verify shape), ragged tails
    ([70, 130, 300], 4, 16),         # 64 rows
    ([45, 200, 513], 3, 5),          # 15 rows: odd group and window (padding rows in the Q tile)
    ([5, 9, 4], 4, 8),               # window covering the whole context
]


@pytest.mark.parametrize("lens,q_len,group", SHAPES)
def test_fp8_scores_match_oracle(lens, q_len, group):
    dp = _problem(lens, q_len, group)
    ref = _oracle_out(dp)
    for S in (1, 3, 0):
        out = G.run_attention(dp, num_splits=S, fp8_qk=True)
        torch.cuda.synchronize()
        assert dp.err.item() == 0
        G.assert_close(out.float().cpu().numpy(), ref, f"fp8 scores {lens} q{q_len} G{group} S={S}")


def test_fp8_partials_match_oracle():
    dp = _problem([1000, 236, 33, 127], 4, 8)
    S = 3
    ws, p = G.run_attention(dp, num_splits=S, partial=True, fp8_qk=True)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    o, m, l = [x.cpu().numpy() for x in kvq.workspace_views(ws, p)]
    pr = dp.host
    kc, vc, ks, vs = P.oracle_pools(pr, True, (dp.k_scale, dp.v_scale))
    ro, rm, rl, _ = oracle.attention_partials(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens,
                                              S, ks, vs, fp8_q=True)
    nonempty = rl > 0
    assert np.array_equal(l > 0, nonempty)
    assert np.isneginf(m[~nonempty]).all()
    G.assert_close(m[nonempty], rm[nonempty], "tmp_max", atol=1e-4, rtol=1e-5)
    G.assert_close(l[nonempty], rl[nonempty], "tmp_sum", atol=1e-4, rtol=2e-3)
    G.assert_close(o[nonempty], ro[nonempty], "tmp_out")


def test_fp8_topk_and_nan_slots():
    dp = _problem([700, 300, 90], 4, 8, sentinel=0x7F, topk=160, topk_fraction=0.67)
    assert dp.topk_lens is not None
    ref = _oracle_out(dp)
    for S in (1, 2):
        out = G.run_attention(dp, num_splits=S, fp8_qk=True)
        torch.cuda.synchronize()
        assert dp.err.item() == 0
        G.assert_close(out.float().cpu().numpy(), ref, f"fp8 scores top-k S={S}")


def test_fp8_large_scores_move_the_reference():
    w = inputs.Workload("tc", 12, 1, 2, 4, 16, 2, 128, 0, "list:900,700", calib_tokens=64)
    pr = P.host_problem(w)
    ramp = np.linspace(0.2, 6.0, pr.k_tok.shape[0], dtype=np.float32)[:, None, None]
    pr.k_tok = (pr.k_tok.astype(np.float32) * ramp).astype(np.float16)
    pr.k_calib = (pr.k_calib.astype(np.float32) * 6.0).astype(np.float16)
    pr.q = (pr.q.astype(np.float32) * 3.0).astype(np.float16)
    dp = G.device_problem(pr, True)
    ref = _oracle_out(dp)
    for S in (1, 2):
        out = G.run_attention(dp, num_splits=S, fp8_qk=True)
        torch.cuda.synchronize()
        assert dp.err.item() == 0
        G.assert_close(out.float().cpu().numpy(), ref, f"fp8 scores, growing S={S}")


def test_fp8_zero_group_and_exact_grid_query():
    """A group whose query is all zero (scale 1, codes 0: the mean of V), and a
    query already on a power-of-two-scaled E4M3 grid, whose FP8 scores are the
    fp16 scores (the kernel's result then agrees with the plain oracle too)."""
    dp = _problem([300, 129], 4, 8)
    pr = dp.host
    rng = np.random.default_rng(5)
    G_ = pr.w.num_q_heads // pr.w.num_kv_heads
    codes = rng.integers(0, 0x7E, size=pr.q.shape).astype(np.uint8) | \
        (rng.integers(0, 2, size=pr.q.shape).astype(np.uint8) << 7)
    codes[(codes & 0x7F) > 0x5F] &= 0xDF                      # magnitudes up to 30
    for b in range(pr.q.shape[0]):                             # one +-448 per group: scale 2^-6 exactly
        for g in range(pr.w.num_kv_heads):
            codes[b, 0, g * G_, 0] = 0x7E | ((b + g) % 2) << 7
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    q = (vals * 2.0 ** -6).astype(np.float16)                  # exact in fp16
    q[0, :, 0:G_, :] = 0                                       # (b 0, kv head 0): all zero
    pr.q = q
    dp.q.copy_(torch.from_numpy(q).to(dp.q.device))
    ref8 = _oracle_out(dp)
    ref16 = _oracle_out(dp, fp8_q=False)
    for S in (1, 2):
        out = G.run_attention(dp, num_splits=S, fp8_qk=True).float().cpu().numpy()
        torch.cuda.synchronize()
        assert dp.err.item() == 0
        G.assert_close(out, ref8, f"grid query S={S}")
        G.assert_close(out, ref16, f"grid query vs fp16 scores S={S}")


def test_fp8_flag_refused_outside_its_shapes():
    dp = _problem([300, 17], 1, 4)       # 4 rows per kv head: the mma.sync kernel's shape
    with pytest.raises(kvq.KvqError):
        G.run_attention(dp, fp8_qk=True)
    dp = _problem([300, 17], 4, 4)
    with pytest.raises(kvq.KvqError):
        G.run_attention(dp, fp8_qk=True, bitcast_decode=True)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
