"""The fused decode / verify step (paged_decode_step_e4m3 / _fp16): this step's
append done by the attention launch's producer warps, then the attention over
the updated cache.

Every case runs the fused call on one copy of the pools and the two separate
calls (kv_append_*, then paged_decode_attn_*) on another, over several steps
whose new keys dominate the scores and whose new values change every step, so
that a page copied before its new rows were written would show.  The whole
pools (including every slot still holding the sentinel) and the outputs must
be bit-identical between the two, the pools must equal the oracle's append
byte for byte, and the outputs must match the oracle's attention within the
path's tolerance.  Quantise-on-append is the cache write of PR "[Model][SM70]
[FP8] Integrate calibrated E4M3 QSA KV capacity path", section Changes."""
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


def _history_pools(pr, e4m3):
    """Pools filled with the sentinel, then the history tokens appended by the
    library (this step's tokens are not); the layer's calibrated scales."""
    w = pr.w
    shape = (pr.P, w.num_kv_heads, 4, w.head_dim)
    if e4m3:
        kc = torch.full(shape, P.SENTINEL, dtype=torch.uint8, device="cuda")
        ks = kvq.calibrate_scale(G.to_dev(pr.k_calib))
        vs = kvq.calibrate_scale(G.to_dev(pr.v_calib))
    else:
        kc = torch.empty(shape, dtype=torch.float16, device="cuda")
        kc.view(torch.int16).fill_(int(np.uint16(P.SENTINEL * 0x101).view(np.int16)))
        ks = vs = 1.0
    vc = kc.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if pr.hist_slots.size:
        k, v, sm = G.to_dev(pr.k_tok[pr.hist_rows]), G.to_dev(pr.v_tok[pr.hist_rows]), G.to_dev(pr.hist_slots)
        if e4m3:
            kvq.kv_append_e4m3(k, v, sm, kc, vc, ks, vs, err)
        else:
            kvq.kv_append_fp16(k, v, sm, kc, vc, err)
    assert err.item() == 0
    return kc, vc, ks, vs


def _bytes(t):
    return t.view(torch.uint8).cpu().numpy() if t.dtype == torch.uint8 else t.view(torch.int16).cpu().numpy()


def _run(lens, q_len, e4m3, Hq=8, Hkv=2, D=64, S=0, split_pages=0, bitcast=False, mma_sync=False,
         longest_first=False, iters=3, bad_page_seq=None, bad_len_seq=None, strict=False):
    B = len(lens)
    w = inputs.Workload("step", 31, 1, B, q_len, Hq, Hkv, D, S, "list:" + ",".join(map(str, lens)),
                        outlier_channels=2, calib_tokens=64, split_pages=split_pages)
    pr = P.host_problem(w)
    kA, vA, ks, vs = _history_pools(pr, e4m3)
    kB, vB = kA.clone(), vA.clone()
    bt_np = pr.layout.block_tables.copy()
    lens_np = pr.layout.lens.copy()
    expect_err = 0
    if bad_page_seq is not None:
        # the page of the sequence's last position names no page of the pool
        bt_np[bad_page_seq, (lens_np[bad_page_seq] - 1) // 4] = pr.P + 7
        expect_err |= kvq.DEV_BAD_PAGE
    if bad_len_seq is not None:
        lens_np[bad_len_seq] = bt_np.shape[1] * 4 + 1     # past the block-table row
        expect_err |= kvq.DEV_BAD_LEN
    bt, cl = G.to_dev(bt_np), G.to_dev(lens_np)
    q = G.to_dev(pr.q)
    # slots of the separate append, from the same (possibly damaged) tables; a
    # sequence with an invalid length appends nothing
    seq = np.repeat(np.arange(B), q_len)
    pos = lens_np[seq] - q_len + np.tile(np.arange(q_len), B)
    ok = (lens_np[seq] >= q_len) & (lens_np[seq] <= bt_np.shape[1] * 4)
    pos_ok = np.where(ok, pos, 0)
    slots_np = np.where(ok, bt_np[seq, pos_ok // 4].astype(np.int64) * 4 + pos_ok % 4, -1).astype(np.int32)
    slots = G.to_dev(slots_np)
    p = kvq.AttnParams(B, q_len, Hq, Hkv, D, S, bt.shape[1], 0, 0.0, split_pages,
                       kvq._flags(bitcast, mma_sync, False, strict, longest_first))
    wsA, wsB = kvq.alloc_workspace(p, q.device), kvq.alloc_workspace(p, q.device)
    outA, outB = torch.empty_like(q), torch.empty_like(q)
    errA = torch.zeros(1, dtype=torch.int32, device="cuda")
    errB = torch.zeros(1, dtype=torch.int32, device="cuda")
    rng = np.random.default_rng(11)
    rows = pr.step_rows
    Gq = Hq // Hkv
    kw = dict(num_splits=S, split_pages=split_pages, mma_sync=mma_sync, longest_first=longest_first,
              strict_order=strict)
    for it in range(iters):
        if it == 0:
            knew, vnew = pr.k_tok[rows], pr.v_tok[rows]
        else:
            # new keys along the query of the group's first head (they dominate the scores)
            knew = np.empty((len(rows), Hkv, D), np.float16)
            for n, (b, i) in enumerate((b, i) for b in range(B) for i in range(q_len)):
                for g in range(Hkv):
                    knew[n, g] = (pr.q[b, i, g * Gq].astype(np.float32) * (1.5 + 0.2 * it)).astype(np.float16)
            vnew = (rng.standard_normal((len(rows), Hkv, D)) * 3).astype(np.float16)
        pr.k_tok[rows], pr.v_tok[rows] = knew, vnew
        kd, vd = G.to_dev(knew), G.to_dev(vnew)
        k4, v4 = kd.view(B, q_len, Hkv, D), vd.view(B, q_len, Hkv, D)
        if e4m3:
            kvq.paged_decode_step_e4m3(q, k4, v4, kA, vA, bt, cl, ks, vs, wsA, outA, err_flag=errA,
                                       bitcast_decode=bitcast, **kw)
            kvq.kv_append_e4m3(kd, vd, slots, kB, vB, ks, vs, errB)
            kvq.paged_decode_attn_e4m3(q, kB, vB, bt, cl, ks, vs, wsB, outB, err_flag=errB,
                                       bitcast_decode=bitcast, **kw)
        else:
            kvq.paged_decode_step_fp16(q, k4, v4, kA, vA, bt, cl, wsA, outA, err_flag=errA, **kw)
            kvq.kv_append_fp16(kd, vd, slots, kB, vB, errB)
            kvq.paged_decode_attn_fp16(q, kB, vB, bt, cl, wsB, outB, err_flag=errB, **kw)
        torch.cuda.synchronize()
        what = f"step {it} lens {lens} q_len {q_len} e4m3={e4m3} D={D} S={S} sp={split_pages} bitcast={bitcast}"
        assert errA.item() == expect_err, what
        assert torch.equal(kA.view(torch.uint8), kB.view(torch.uint8)), what
        assert torch.equal(vA.view(torch.uint8), vB.view(torch.uint8)), what
        assert torch.equal(outA.view(torch.int16), outB.view(torch.int16)), what
    # against the oracle: pools byte for byte, outputs within the path's tolerance
    kc_o, vc_o = P.empty_pools(pr, e4m3)
    okrows = slots_np >= 0
    for sl, rw in ((pr.hist_slots, pr.hist_rows), (slots_np[okrows], rows[okrows])):
        if sl.size == 0:
            continue
        kk, vv = pr.k_tok[rw], pr.v_tok[rw]
        # slots past the pool are the append's to skip; the oracle is given only real ones
        real = sl < pr.P * 4
        if e4m3:
            oracle.append_e4m3(kk[real], vv[real], sl[real], kc_o, vc_o, ks, vs)
        else:
            oracle.append_fp16(kk[real], vv[real], sl[real], kc_o, vc_o)
    view = np.uint8 if e4m3 else np.int16
    assert np.array_equal(_bytes(kA), kc_o.view(view)), "K pool differs from the oracle's append"
    assert np.array_equal(_bytes(vA), vc_o.view(view)), "V pool differs from the oracle's append"
    if bad_page_seq is None and bad_len_seq is None:
        ref, _ = oracle.attention(pr.q, kc_o, vc_o, bt_np, lens_np, ks, vs, None, None)
        G.assert_close(outA.float().cpu().numpy(), ref, what)


# contexts ending at each offset inside a page, long enough for several stages per split
LENS = [517, 518, 519, 520, 133]


@pytest.mark.parametrize("e4m3", [True, False])
@pytest.mark.parametrize("S", [1, 3])
@pytest.mark.parametrize("q_len", [1, 4])
def test_fused_step_equals_append_then_attention_d64(q_len, S, e4m3):
    _run(LENS, q_len, e4m3, S=S)


@pytest.mark.parametrize("e4m3", [True, False])
@pytest.mark.parametrize("q_len", [1, 3])
def test_fused_step_decode_shape_d128(q_len, e4m3):
    # 32 / 4 heads, head_dim 128: the split kernel (q_len 1) and the tcgen05 kernel (24 rows)
    _run([517, 4100, 259, 1026], q_len, e4m3, Hq=32, Hkv=4, D=128, S=4)


@pytest.mark.parametrize("mma_sync", [False, True])
def test_fused_step_verify_window_d128(mma_sync):
    # MTP3 verify: 32 rows per kv head on the tcgen05 kernel, or the mma.sync kernel
    _run([517, 518, 2051, 130], 4, True, Hq=32, Hkv=4, D=128, S=2, mma_sync=mma_sync)


def test_fused_step_refuses_the_other_decoder_and_fp8_scores():
    w = inputs.Workload("step", 31, 1, 2, 4, 32, 4, 128, 2, "list:300,517", calib_tokens=64)
    pr = P.host_problem(w)
    kA, vA, ks, vs = _history_pools(pr, True)
    before_k, before_v = kA.clone(), vA.clone()
    q, bt, cl = G.to_dev(pr.q), G.to_dev(pr.layout.block_tables), G.to_dev(pr.layout.lens)
    kn = G.to_dev(pr.k_tok[pr.step_rows]).view(2, 4, 4, 128)
    vn = G.to_dev(pr.v_tok[pr.step_rows]).view(2, 4, 4, 128)
    p = kvq.AttnParams(2, 4, 32, 4, 128, 2, bt.shape[1], 0, 0.0, 0, 0)
    ws = kvq.alloc_workspace(p, q.device)
    for kw in (dict(bitcast_decode=True), dict(fp8_qk=True)):
        with pytest.raises(kvq.KvqError) as e:
            kvq.paged_decode_step_e4m3(q, kn, vn, kA, vA, bt, cl, ks, vs, ws, num_splits=2, **kw)
        assert e.value.status == -4
    torch.cuda.synchronize()
    assert torch.equal(kA, before_k) and torch.equal(vA, before_v)    # refused before any launch


def test_fused_step_new_rows_straddle_splits():
    # 4 pages in 4 equal splits: positions L-4 .. L-1 fall in the last two splits
    _run([13, 14, 15, 16, 4, 6], 4, True, S=4)
    # fixed-size splits of 3 pages: the window crosses from one split into the next
    _run([519, 517, 35], 4, True, S=0, split_pages=3)


@pytest.mark.parametrize("q_len", [1, 4])
def test_fused_step_with_strict_ordering(q_len):
    # KVQ_ATTN_STRICT_ORDER: nothing is read before the dependency wait
    _run([517, 518, 1029, 36], q_len, True, Hq=32, Hkv=4, D=128, S=2, strict=True)


def test_fused_step_longest_first_and_more_splits_than_pages():
    _run([9, 700, 41, 1500], 1, True, Hq=32, Hkv=4, D=128, S=8, longest_first=True)


@pytest.mark.parametrize("e4m3", [True, False])
def test_fused_step_skips_a_bad_page_and_reports_it(e4m3):
    _run([517, 518, 133], 4, e4m3, S=2, bad_page_seq=1, iters=2)


def test_fused_step_appends_nothing_for_an_invalid_length():
    _run([517, 518, 133], 1, True, S=2, bad_len_seq=2, iters=2)


@pytest.mark.parametrize("e4m3", [True, False])
def test_fused_steps_back_to_back_with_growing_contexts(e4m3):
    """Consecutive decode steps through the fused call with nothing else in the
    stream between them (at this shape each call is one cluster-merging
    kernel): step t + 1 attends the row step t appended.  The new keys lie
    along the query of their group's first head, so every step's newest rows
    carry most of the attention weight, and a row read before the previous
    step had written it would show in that step's output."""
    T = 6
    L0 = np.array([517, 518, 300, 1029, 64, 2050])
    B, Hq, Hkv, D = len(L0), 32, 4, 128
    w = inputs.Workload("chain", 33, 1, B, 1, Hq, Hkv, D, 4, "list:" + ",".join(map(str, L0 + T)),
                        calib_tokens=64)
    pr = P.host_problem(w)
    Gq = Hq // Hkv
    for b in range(B):
        for t in range(T):
            for g in range(Hkv):
                pr.k_tok[pr.offsets[b] + L0[b] + t, g] = (
                    pr.q[b, 0, g * Gq].astype(np.float32) * (1.0 + 0.3 * t)).astype(np.float16)
    # history: positions below L0 of each sequence
    seq = np.repeat(np.arange(B), L0)
    pos = np.concatenate([np.arange(l) for l in L0])
    shape = (pr.P, Hkv, 4, D)
    if e4m3:
        kc = torch.full(shape, P.SENTINEL, dtype=torch.uint8, device="cuda")
        ks = kvq.calibrate_scale(G.to_dev(pr.k_calib))
        vs = kvq.calibrate_scale(G.to_dev(pr.v_calib))
    else:
        kc = torch.zeros(shape, dtype=torch.float16, device="cuda")
        ks = vs = 1.0
    vc = kc.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hk, hv = G.to_dev(pr.k_tok[pr.offsets[seq] + pos]), G.to_dev(pr.v_tok[pr.offsets[seq] + pos])
    hs = G.to_dev(inputs.slot_mapping(pr.layout.block_tables, seq, pos))
    if e4m3:
        kvq.kv_append_e4m3(hk, hv, hs, kc, vc, ks, vs, err)
    else:
        kvq.kv_append_fp16(hk, hv, hs, kc, vc, err)
    q, bt = G.to_dev(pr.q), G.to_dev(pr.layout.block_tables)
    lens = [(L0 + t + 1).astype(np.int32) for t in range(T)]
    cls = [G.to_dev(l) for l in lens]
    kn = [G.to_dev(pr.k_tok[pr.offsets + L0 + t]).view(B, 1, Hkv, D) for t in range(T)]
    vn = [G.to_dev(pr.v_tok[pr.offsets + L0 + t]).view(B, 1, Hkv, D) for t in range(T)]
    p = kvq.AttnParams(B, 1, Hq, Hkv, D, 4, bt.shape[1], 0, 0.0, 0, 0)
    assert kvq.attn_launches(p, e4m3, True) == 1     # 96 CTAs: one cluster-merging kernel
    ws = kvq.alloc_workspace(p, q.device)
    outs = [torch.empty_like(q) for _ in range(T)]
    torch.cuda.synchronize()
    for t in range(T):                       # back to back: no copy, no sync
        if e4m3:
            kvq.paged_decode_step_e4m3(q, kn[t], vn[t], kc, vc, bt, cls[t], ks, vs, ws, outs[t], num_splits=4,
                                       err_flag=err)
        else:
            kvq.paged_decode_step_fp16(q, kn[t], vn[t], kc, vc, bt, cls[t], ws, outs[t], num_splits=4, err_flag=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    seq_all = np.repeat(np.arange(B), L0 + T)
    pos_all = np.concatenate([np.arange(l) for l in L0 + T])
    kc_o, vc_o = P.empty_pools(pr, e4m3)
    if not e4m3:
        kc_o[:] = 0
        vc_o[:] = 0
    rows_all = pr.offsets[seq_all] + pos_all
    slots_all = inputs.slot_mapping(pr.layout.block_tables, seq_all, pos_all)
    if e4m3:
        oracle.append_e4m3(pr.k_tok[rows_all], pr.v_tok[rows_all], slots_all, kc_o, vc_o, ks, vs)
    else:
        oracle.append_fp16(pr.k_tok[rows_all], pr.v_tok[rows_all], slots_all, kc_o, vc_o)
    view = np.uint8 if e4m3 else np.int16
    assert np.array_equal(_bytes(kc), kc_o.view(view)) and np.array_equal(_bytes(vc), vc_o.view(view))
    for t in range(T):
        ref, _ = oracle.attention(pr.q, kc_o, vc_o, pr.layout.block_tables, lens[t], ks, vs, None, None)
        G.assert_close(outs[t].float().cpu().numpy(), ref, f"chained step {t} e4m3={e4m3}")
