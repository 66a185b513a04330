"""GPU parity of the tcgen05 kernel, the default for more than 8 query rows per
kv head at head_dim 128 (MTP verify): outputs and FP32 split partials against
the oracle, and outputs beside the mma.sync kernel (flag KVQ_ATTN_MMA_SYNC), on
ragged lengths that leave partial 128-token tiles and odd staging stages."""
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


def _oracle_out(dp, topk=True):
    pr = dp.host
    kc, vc, ks, vs = P.oracle_pools(pr, dp.e4m3, (dp.k_scale, dp.v_scale) if dp.e4m3 else None)
    out, _ = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, ks, vs,
                              pr.topk_idx if topk else None, pr.topk_lens if topk else None)
    return out


def _problem(lens, q_len, group, e4m3, sentinel=P.SENTINEL, **kw):
    w = inputs.Workload("tc", 12, 1, len(lens), q_len, 2 * group, 2, 128, 0,
                        "list:" + ",".join(map(str, lens)), calib_tokens=64, heavy_channels=4, **kw)
    return G.device_problem(P.host_problem(w), e4m3, sentinel=sentinel)


SHAPES = [
    ([300, 17, 129, 64], 4, 4),      # 16 rows; one-token tiles, exact 64/128 boundaries
    ([1000, 236, 33, 127], 4, 8),    # 32 rows (the verify shape), ragged tails
    ([70, 130, 300], 4, 16),         # 64 rows
    ([45, 200, 513], 3, 5),          # 15 rows: odd group and window
    ([5, 9, 4], 4, 8),               # window covering the whole context
]


@pytest.mark.parametrize("lens,q_len,group", SHAPES)
@pytest.mark.parametrize("e4m3", [True, False])
def test_tc_matches_oracle_and_mma_sync(lens, q_len, group, e4m3):
    dp = _problem(lens, q_len, group, e4m3)
    ref = _oracle_out(dp)
    for S in (1, 3, 0):
        tc = G.run_attention(dp, num_splits=S)
        ms = G.run_attention(dp, num_splits=S, mma_sync=True)
        torch.cuda.synchronize()
        assert dp.err.item() == 0
        what = f"{lens} q{q_len} G{group} e4m3={e4m3} S={S}"
        G.assert_close(tc.float().cpu().numpy(), ref, "tcgen05 " + what)
        G.assert_close(ms.float().cpu().numpy(), ref, "mma.sync " + what)


@pytest.mark.parametrize("e4m3", [True, False])
def test_tc_partials_match_oracle(e4m3):
    dp = _problem([1000, 236, 33, 127], 4, 8, e4m3)
    S = 3
    ws, p = G.run_attention(dp, num_splits=S, partial=True)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    o, m, l = [x.cpu().numpy() for x in kvq.workspace_views(ws, p)]
    pr = dp.host
    kc, vc, ks, vs = P.oracle_pools(pr, e4m3, (dp.k_scale, dp.v_scale) if e4m3 else None)
    ro, rm, rl, _ = oracle.attention_partials(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens,
                                              S, ks, vs)
    nonempty = rl > 0
    assert np.array_equal(l > 0, nonempty)
    assert np.isneginf(m[~nonempty]).all()
    G.assert_close(m[nonempty], rm[nonempty], "tmp_max", atol=1e-4, rtol=1e-5)
    G.assert_close(l[nonempty], rl[nonempty], "tmp_sum", atol=1e-4, rtol=2e-3)
    G.assert_close(o[nonempty], ro[nonempty], "tmp_out")


@pytest.mark.parametrize("e4m3", [True, False])
def test_tc_topk_and_nan_slots(e4m3):
    dp = _problem([700, 300, 90], 4, 8, e4m3, sentinel=0x7F, topk=160, topk_fraction=0.67)
    assert dp.topk_lens is not None
    ref = _oracle_out(dp)
    for S in (1, 2):
        out = G.run_attention(dp, num_splits=S)
        torch.cuda.synchronize()
        assert dp.err.item() == 0
        G.assert_close(out.float().cpu().numpy(), ref, f"tcgen05 top-k e4m3={e4m3} S={S}")


def test_tc_large_scores_move_the_reference():
    """Scores that grow along the sequence force the running maximum past the
    2^8 reference band several times (tensor-memory rescale of O^T)."""
    w = inputs.Workload("tc", 12, 1, 2, 4, 16, 2, 128, 0, "list:900,700", calib_tokens=64)
    pr = P.host_problem(w)
    # keys grow in magnitude along the positions: later tokens dominate
    ramp = np.linspace(0.2, 6.0, pr.k_tok.shape[0], dtype=np.float32)[:, None, None]
    pr.k_tok = (pr.k_tok.astype(np.float32) * ramp).astype(np.float16)
    pr.k_calib = (pr.k_calib.astype(np.float32) * 6.0).astype(np.float16)
    pr.q = (pr.q.astype(np.float32) * 3.0).astype(np.float16)
    dp = G.device_problem(pr, True)
    ref = _oracle_out(dp)
    for S in (1, 2):
        out = G.run_attention(dp, num_splits=S)
        torch.cuda.synchronize()
        assert dp.err.item() == 0
        G.assert_close(out.float().cpu().numpy(), ref, f"growing scores S={S}")


@pytest.mark.parametrize("lens,q_len,group", SHAPES)
def test_tc_bitcast_decoder_matches_oracle_and_hardware_conversion(lens, q_len, group):
    """The pages' bitcast decoder on the tcgen05 kernel (flag
    KVQ_ATTN_BITCAST_DECODE on a verify shape): every K and V byte becomes its
    value times 2^-8 with the channels of each group of four in the order 0, 2,
    1, 3 (the query tile takes the same order, the output undoes it) and the
    2^8 folded into the hoisted scales.  Against the oracle, and against the
    hardware conversion within the path's tolerance (the Q K^T sums run over
    the channels in another order)."""
    dp = _problem(lens, q_len, group, True)
    ref = _oracle_out(dp)
    for S in (1, 3, 0):
        bc = G.run_attention(dp, num_splits=S, bitcast_decode=True)
        hw = G.run_attention(dp, num_splits=S)
        torch.cuda.synchronize()
        assert dp.err.item() == 0
        what = f"bitcast {lens} q{q_len} G{group} S={S}"
        G.assert_close(bc.float().cpu().numpy(), ref, what)
        G.assert_close(bc.float().cpu().numpy(), hw.float().cpu().numpy().astype(np.float64), what + " vs hardware")


def test_tc_bitcast_decoder_topk_nan_slots_and_partials():
    dp = _problem([700, 300, 90], 4, 8, True, sentinel=0x7F, topk=160, topk_fraction=0.67)
    ref = _oracle_out(dp)
    for S in (1, 2):
        out = G.run_attention(dp, num_splits=S, bitcast_decode=True)
        torch.cuda.synchronize()
        assert dp.err.item() == 0
        G.assert_close(out.float().cpu().numpy(), ref, f"bitcast tcgen05 top-k S={S}")
    # the split partials: m, l and o in the oracle's units (the decoder's 2^-8 folded back)
    dp = _problem([1000, 236, 33, 127], 4, 8, True)
    S = 3
    ws, p = G.run_attention(dp, num_splits=S, partial=True, bitcast_decode=True)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    o, m, l = [x.cpu().numpy() for x in kvq.workspace_views(ws, p)]
    pr = dp.host
    kc, vc, ks, vs = P.oracle_pools(pr, True, (dp.k_scale, dp.v_scale))
    ro, rm, rl, _ = oracle.attention_partials(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, S, ks, vs)
    nonempty = rl > 0
    assert np.array_equal(l > 0, nonempty)
    G.assert_close(m[nonempty], rm[nonempty], "tmp_max", atol=1e-4, rtol=1e-5)
    G.assert_close(l[nonempty], rl[nonempty], "tmp_sum", atol=1e-4, rtol=2e-3)
    G.assert_close(o[nonempty], ro[nonempty], "tmp_out")
