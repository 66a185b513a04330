"""Pins for the oracle's paged append and attention (CPU only).

Each check compares the oracle with something other than itself: an
independent library reference (torch float8 decode + numpy gather +
torch.softmax in float64), closed forms, and invariants that a dropped term,
a wrong index or a transposed operand would break.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_e4m3_gb300 import inputs
from tests import _problems as P


@pytest.fixture(scope="module", params=["tiny", "tiny_verify"])
def tiny(request):
    pr = P.host_problem(request.param)
    kc, vc, ks, vs = P.oracle_pools(pr)
    return pr, kc, vc, ks, vs


# ---------------------------------------------------------------------------
# append

def test_append_bytes_match_library_conversion(tiny):
    pr, kc, vc, ks, vs = tiny
    bt, lens = pr.layout.block_tables, pr.layout.lens
    for b in range(pr.w.batch):
        for pos in range(int(lens[b])):
            page, slot = bt[b, pos // 4], pos % 4
            row = pr.offsets[b] + pos
            want_k = P.torch_dequant(kc[page, :, slot, :], 1.0)
            x = torch.from_numpy(pr.k_tok[row].astype(np.float32)) / torch.tensor(ks, dtype=torch.float32)
            ref = torch.clamp(x, -448, 448).to(torch.float8_e4m3fn).double().numpy()
            assert np.array_equal(want_k, ref)
    # V spot check on the last token of every sequence
    for b in range(pr.w.batch):
        pos = int(lens[b]) - 1
        x = torch.from_numpy(pr.v_tok[pr.offsets[b] + pos].astype(np.float32)) / torch.tensor(vs, dtype=torch.float32)
        ref = torch.clamp(x, -448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(vc[bt[b, pos // 4], :, pos % 4, :], ref)


def test_append_leaves_unowned_slots_untouched(tiny):
    pr, kc, vc, _, _ = tiny
    owned = np.zeros((pr.P, 4), bool)
    bt, lens = pr.layout.block_tables, pr.layout.lens
    for b in range(pr.w.batch):
        for pos in range(int(lens[b])):
            owned[bt[b, pos // 4], pos % 4] = True
    for pool in (kc, vc):
        by_slot = pool.transpose(0, 2, 1, 3)          # [P][4][Hkv][D]
        assert (by_slot[~owned] == P.SENTINEL).all()
        # owned slots were written: not every byte can still be the sentinel
        assert (by_slot[owned] != P.SENTINEL).any(axis=(-1, -2)).all()


def test_append_skips_negative_and_flags_out_of_range():
    pr = P.host_problem("tiny")
    kc, vc = P.empty_pools(pr)
    slots = pr.step_slots.copy()
    slots[0] = -1
    slots[1] = pr.P * 4 + 3       # beyond the pool
    flags = oracle.append_e4m3(pr.k_tok[pr.step_rows], pr.v_tok[pr.step_rows], slots, kc, vc, 0.1, 0.1)
    assert flags & oracle.BAD_SLOT
    assert (kc.reshape(pr.P, -1, 4, pr.w.head_dim)[:, :, :, :] == P.SENTINEL).sum() > 0


def test_fp16_append_is_a_copy():
    pr = P.host_problem("tiny")
    kc, vc, _, _ = P.oracle_pools(pr, e4m3=False)
    bt = pr.layout.block_tables
    for b in range(pr.w.batch):
        pos = int(pr.layout.lens[b]) - 1
        assert np.array_equal(kc[bt[b, pos // 4], :, pos % 4, :].view(np.uint16),
                              pr.k_tok[pr.offsets[b] + pos].view(np.uint16))


# ---------------------------------------------------------------------------
# attention against an independent library reference

def test_attention_matches_torch_softmax(tiny):
    pr, kc, vc, ks, vs = tiny
    out, flags = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, ks, vs)
    assert flags == 0
    ref = P.torch_reference(pr.q, P.torch_dequant(kc, ks), P.torch_dequant(vc, vs),
                            pr.layout.block_tables, pr.layout.lens, pr.w.q_len)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_fp16_arm_matches_unquantised_softmax(tiny):
    pr = tiny[0]
    kc, vc, _, _ = P.oracle_pools(pr, e4m3=False)
    out, flags = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens)
    assert flags == 0
    ref = P.torch_reference(pr.q, kc.astype(np.float64), vc.astype(np.float64),
                            pr.layout.block_tables, pr.layout.lens, pr.w.q_len)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_topk_matches_torch_softmax():
    w = inputs.get("tiny_verify", topk=24, topk_fraction=0.5)
    pr = P.host_problem(w)
    kc, vc, ks, vs = P.oracle_pools(pr)
    assert pr.topk_lens is not None and (pr.topk_lens > 0).sum() == 1
    out, flags = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, ks, vs,
                                  pr.topk_idx, pr.topk_lens)
    assert flags == 0
    ref = P.torch_reference(pr.q, P.torch_dequant(kc, ks), P.torch_dequant(vc, vs),
                            pr.layout.block_tables, pr.layout.lens, pr.w.q_len,
                            pr.topk_idx, pr.topk_lens)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# closed forms

def _single_seq(L, q, kvals, vvals, q_len=1, e4m3=True):
    """A one-sequence problem with an identity block table, from explicit values."""
    Hkv, D = kvals.shape[1], kvals.shape[2]
    pages = (L + 3) // 4
    bt = np.arange(pages, dtype=np.int32)[None, :]
    slots = np.arange(L, dtype=np.int32)
    if e4m3:
        kc = np.full((pages, Hkv, 4, D), P.SENTINEL, np.uint8)
        vc = kc.copy()
        oracle.append_e4m3(kvals, vvals, slots, kc, vc, 1.0, 1.0)
    else:
        kc = np.zeros((pages, Hkv, 4, D), np.float16)
        vc = kc.copy()
        oracle.append_fp16(kvals, vvals, slots, kc, vc)
    return oracle.attention(q, kc, vc, bt, np.array([L], np.int32))[0]


def test_single_key_returns_its_value():
    rng = np.random.default_rng(3)
    k = rng.standard_normal((1, 2, 16)).astype(np.float16)
    v = rng.standard_normal((1, 2, 16)).astype(np.float16)
    q = rng.standard_normal((1, 1, 4, 16)).astype(np.float16)
    out = _single_seq(1, q, k, v)
    vq = oracle.e4m3_decode_array(oracle.quantize(v, 1.0))
    for h in range(4):
        np.testing.assert_array_equal(out[0, 0, h], vq[0, h // 2])


def test_zero_query_gives_mean_of_values():
    rng = np.random.default_rng(4)
    L = 23
    k = rng.standard_normal((L, 1, 8)).astype(np.float16)
    v = rng.standard_normal((L, 1, 8)).astype(np.float16)
    q = np.zeros((1, 1, 2, 8), np.float16)
    out = _single_seq(L, q, k, v)
    vq = oracle.e4m3_decode_array(oracle.quantize(v, 1.0))
    np.testing.assert_allclose(out[0, 0, 0], vq[:, 0].mean(axis=0), rtol=1e-13, atol=1e-15)


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(5)
    L = 9
    k = np.repeat(rng.standard_normal((1, 1, 8)), L, axis=0).astype(np.float16)
    v = rng.standard_normal((L, 1, 8)).astype(np.float16)
    q = rng.standard_normal((1, 1, 1, 8)).astype(np.float16)
    out = _single_seq(L, q, k, v, e4m3=False)
    np.testing.assert_allclose(out[0, 0, 0], v[:, 0].astype(np.float64).mean(0), rtol=1e-13)


def test_dominant_key_selects_its_value():
    L, D = 12, 8
    k = np.zeros((L, 1, D), np.float16)
    k[7, 0, :] = 8.0                      # the only key aligned with q
    v = np.arange(L * D, dtype=np.float16).reshape(L, 1, D) / 16
    q = np.full((1, 1, 1, D), 8.0, np.float16)   # score 8*8*8/sqrt(8) ~ 181 above the rest
    out = _single_seq(L, q, k, v, e4m3=False)
    np.testing.assert_allclose(out[0, 0, 0], v[7, 0].astype(np.float64), rtol=1e-12)


def test_empty_key_set_gives_zero():
    """A top-k list whose entries all lie after the query position -> nothing to attend."""
    pr = P.host_problem("tiny")
    kc, vc, ks, vs = P.oracle_pools(pr)
    ti = np.full((2, 2, 4), 0, np.int32)
    ti[0] = 36    # == L-1 for sequence 0 (L = 37): visible to the decode row
    tl = np.array([4, 0], np.int32)
    out, flags = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, ks, vs, ti, tl)
    assert flags == 0 and np.isfinite(out).all()
    # a verify-style row that sits before every listed position sees an empty set
    lens = pr.layout.lens.copy()
    q4 = np.repeat(pr.q, 4, axis=1)
    ti2 = np.full((2, 2, 1), 36, np.int32)
    out2, _, lse = oracle.attention(q4, kc, vc, pr.layout.block_tables, lens, ks, vs, ti2,
                                    np.array([1, 0], np.int32), return_lse=True)
    assert (out2[0, 0] == 0).all() and np.isneginf(lse[0, 0]).all()      # pos 33 < 36
    assert np.isfinite(lse[0, 3]).all()                                    # pos 36 sees it


# ---------------------------------------------------------------------------
# invariants

def test_page_permutation_invariance(tiny):
    pr, kc, vc, ks, vs = tiny
    out, _ = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, ks, vs)
    perm = np.random.default_rng(11).permutation(pr.P)
    inv = np.argsort(perm)
    kp, vp = kc[perm], vc[perm]                   # new page i holds old page perm[i]
    bt = pr.layout.block_tables.copy()
    bt[bt >= 0] = inv[bt[bt >= 0]]
    out2, _ = oracle.attention(pr.q, kp, vp, bt, pr.layout.lens, ks, vs)
    np.testing.assert_array_equal(out, out2)


@pytest.mark.parametrize("S", [1, 2, 3, 4, 64])
def test_split_partials_combine_to_full(tiny, S):
    pr, kc, vc, ks, vs = tiny
    out, _ = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, ks, vs)
    o, m, l, flags = oracle.attention_partials(pr.q, kc, vc, pr.layout.block_tables,
                                               pr.layout.lens, S, ks, vs)
    assert flags == 0
    comb = oracle.combine(o, m, l)                                  # [B][Hq][q_len][D]
    np.testing.assert_allclose(comb.transpose(0, 2, 1, 3), out, rtol=1e-12, atol=1e-13)
    # the split ranges cover every key exactly once: total weight = full softmax denominator
    _, _, lse = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, ks, vs,
                                 return_lse=True)
    M = np.max(np.where(l > 0, m, -np.inf), axis=-1)
    tot = np.log(np.sum(np.where(l > 0, l * np.exp(m - M[..., None]), 0), axis=-1)) + M
    np.testing.assert_allclose(tot.transpose(0, 2, 1), lse, rtol=1e-12)


def _brute_split_max(pr, K, s_lo, s_hi, b, h, i, topk=None):
    """Max score over the keys of row (b, h, i) whose position lies in
    [s_lo, s_hi) -- or, with a list, whose list entry index does -- by a
    direct dot product over the dequantised pool values (numpy)."""
    L = int(pr.layout.lens[b])
    g = h // pr.w.group
    pos = L - pr.w.q_len + i
    if topk is None:
        keys = [j for j in range(s_lo, min(s_hi, pos + 1))]
    else:
        lst, n = topk
        keys = [int(t) for t in lst[b, g, s_lo:min(s_hi, n[b])] if 0 <= t <= pos]
    if not keys:
        return None
    bt = pr.layout.block_tables[b]
    q = pr.q[b, i, h].astype(np.float64)
    sc = [float(K[bt[j // 4], g, j % 4] @ q) / np.sqrt(pr.w.head_dim) for j in keys]
    return max(sc)


@pytest.mark.parametrize("split_pages,extra", [(1, 0), (3, 0), (8, 2), (25, 0), (40, 1)])
def test_fixed_size_split_partials(tiny, split_pages, extra):
    """Fixed-size splits: split s holds pages [s*sp, (s+1)*sp) of every
    sequence; splits past a sequence's end are empty; the partials still
    combine to the full attention."""
    pr, kc, vc, ks, vs = tiny
    max_pages = pr.layout.block_tables.shape[1]
    S = -(-max_pages // split_pages) + extra
    out, _ = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, ks, vs)
    o, m, l, flags = oracle.attention_partials(pr.q, kc, vc, pr.layout.block_tables,
                                               pr.layout.lens, S, ks, vs, split_pages=split_pages)
    assert flags == 0
    np.testing.assert_allclose(oracle.combine(o, m, l).transpose(0, 2, 1, 3), out, rtol=1e-12,
                               atol=1e-13)
    K = P.torch_dequant(kc, ks)
    for b in range(pr.w.batch):
        for s in range(S):
            for h in (0, pr.w.num_q_heads - 1):
                for i in range(pr.w.q_len):
                    want = _brute_split_max(pr, K, 4 * s * split_pages, 4 * (s + 1) * split_pages,
                                            b, h, i)
                    if want is None:
                        assert l[b, h, i, s] == 0 and np.isneginf(m[b, h, i, s])
                    else:
                        assert l[b, h, i, s] >= 1.0
                        np.testing.assert_allclose(m[b, h, i, s], want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("split_pages", [1, 2, 5])
def test_fixed_size_split_partials_topk(split_pages):
    w = inputs.get("tiny_verify", topk=24, topk_fraction=0.5)
    pr = P.host_problem(w)
    kc, vc, ks, vs = P.oracle_pools(pr)
    max_topk = pr.topk_idx.shape[2]
    S = max(-(-pr.layout.block_tables.shape[1] // split_pages), -(-max_topk // (4 * split_pages)))
    out, _ = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, ks, vs,
                              pr.topk_idx, pr.topk_lens)
    o, m, l, flags = oracle.attention_partials(pr.q, kc, vc, pr.layout.block_tables,
                                               pr.layout.lens, S, ks, vs, pr.topk_idx,
                                               pr.topk_lens, split_pages=split_pages)
    assert flags == 0
    np.testing.assert_allclose(oracle.combine(o, m, l).transpose(0, 2, 1, 3), out, rtol=1e-12,
                               atol=1e-13)
    K = P.torch_dequant(kc, ks)
    b = int(np.nonzero(pr.topk_lens > 0)[0][0])
    c = 4 * split_pages                                  # list entries per split
    for s in range(S):
        for i in range(pr.w.q_len):
            want = _brute_split_max(pr, K, s * c, (s + 1) * c, b, 0, i,
                                    topk=(pr.topk_idx, pr.topk_lens))
            if want is None:
                assert l[b, 0, i, s] == 0
            else:
                np.testing.assert_allclose(m[b, 0, i, s], want, rtol=1e-12, atol=1e-12)


def test_topk_all_positions_equals_dense(tiny):
    pr, kc, vc, ks, vs = tiny
    out, _ = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, ks, vs)
    Lmax = int(pr.layout.lens.max())
    ti = np.zeros((pr.w.batch, pr.w.num_kv_heads, Lmax), np.int32)
    for b in range(pr.w.batch):
        ti[b, :, : pr.layout.lens[b]] = np.arange(pr.layout.lens[b])
    out2, _ = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, ks, vs,
                               ti, pr.layout.lens.copy())
    np.testing.assert_allclose(out2, out, rtol=1e-13, atol=1e-15)


def test_verify_row_equals_shorter_decode():
    pr = P.host_problem("tiny_verify")
    kc, vc, ks, vs = P.oracle_pools(pr)
    out, _ = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, ks, vs)
    for i in range(4):
        lens_i = pr.layout.lens - 4 + i + 1
        dec, _ = oracle.attention(pr.q[:, i:i + 1], kc, vc, pr.layout.block_tables, lens_i, ks, vs)
        np.testing.assert_allclose(out[:, i], dec[:, 0], rtol=1e-13, atol=1e-15)


def test_gqa_equals_mha_with_repeated_kv_heads(tiny):
    pr, kc, vc, ks, vs = tiny
    out, _ = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, ks, vs)
    G = pr.w.group
    kr, vr = np.repeat(kc, G, axis=1), np.repeat(vc, G, axis=1)   # kv head g -> heads g*G..g*G+G-1
    out2, _ = oracle.attention(pr.q, kr, vr, pr.layout.block_tables, pr.layout.lens, ks, vs)
    np.testing.assert_allclose(out2, out, rtol=1e-13, atol=1e-15)


def test_scales_are_hoistable():
    """Scaling K by c multiplies every score by c (sm_scale / c gives the same output),
    and scaling V by c multiplies the output by c."""
    pr = P.host_problem("tiny")
    kc, vc, ks, vs = P.oracle_pools(pr)
    bt, lens = pr.layout.block_tables, pr.layout.lens
    base, _ = oracle.attention(pr.q, kc, vc, bt, lens, ks, vs)
    a, _ = oracle.attention(pr.q, kc, vc, bt, lens, ks * 4, vs, sm_scale=0.125 / 4)
    np.testing.assert_allclose(a, base, rtol=1e-12, atol=1e-14)
    b, _ = oracle.attention(pr.q, kc, vc, bt, lens, ks, vs * 8)
    np.testing.assert_allclose(b, base * 8, rtol=1e-13, atol=1e-14)


def test_bad_page_and_topk_entries_are_flagged_and_skipped():
    pr = P.host_problem("tiny")
    kc, vc, ks, vs = P.oracle_pools(pr)
    bt = pr.layout.block_tables.copy()
    bt[0, 2] = pr.P + 5
    _, flags = oracle.attention(pr.q, kc, vc, bt, pr.layout.lens, ks, vs)
    assert flags & oracle.BAD_PAGE
    ti = np.zeros((2, 2, 3), np.int32)
    ti[1, :, :] = [4, 9, 10_000]
    _, flags = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, ks, vs,
                                ti, np.array([0, 3], np.int32))
    assert flags & oracle.BAD_TOPK


def test_prefill_chunk_rows_equal_decodes_and_brute_force():
    """A prefill chunk (q_len 24, longer than any verify window, over 40
    earlier tokens and a context that ends mid-page) is causal token by
    token: row i equals a decode at context L - 24 + i + 1, and row 0 of the
    last head matches a softmax written out by hand over the decoded pools."""
    w = inputs.Workload("chunk", 31, 1, 1, 24, 4, 2, 64, 0, "list:63", calib_tokens=64)
    pr = P.host_problem(w)
    kc, vc, ks, vs = P.oracle_pools(pr)
    bt, lens = pr.layout.block_tables, pr.layout.lens
    out, _ = oracle.attention(pr.q, kc, vc, bt, lens, ks, vs)
    for i in (0, 1, 11, 23):
        dec, _ = oracle.attention(pr.q[:, i:i + 1], kc, vc, bt, lens - 24 + i + 1, ks, vs)
        np.testing.assert_allclose(out[:, i], dec[:, 0], rtol=1e-13, atol=1e-15)
    # brute force for (token 0, head 3 -> kv head 1): keys 0 .. 63 - 24
    dec_k = oracle.e4m3_decode_array(kc).astype(np.float64) * ks
    dec_v = oracle.e4m3_decode_array(vc).astype(np.float64) * vs
    n_keys = int(lens[0]) - 24 + 1
    K = np.stack([dec_k[bt[0, j // 4], 1, j % 4] for j in range(n_keys)])
    V = np.stack([dec_v[bt[0, j // 4], 1, j % 4] for j in range(n_keys)])
    s = K @ pr.q[0, 0, 3].astype(np.float64) / np.sqrt(64.0)
    p = np.exp(s - s.max())
    np.testing.assert_allclose(out[0, 0, 3], (p @ V) / p.sum(), rtol=1e-12, atol=1e-14)
