"""Pins of the oracle's FP8 score variant: the per-(sequence, kv head) query
quantisation and the attention over the quantised query.

The variant is not on the pages (they keep q in fp16); its reading is the one
stated in the oracle: one binary32 scale amax / 448 per group of G * q_len
rows sharing a kv head (1 for an all-zero group), every element quantised
like a cache element (binary32 division, RNE, satfinite).  The pins below
check it against a library route (the torch E4M3 cast), closed forms
(queries already on the scaled E4M3 grid, an all-zero group) and invariants
(group scope, power-of-two scaling, the group maximum at +-448).
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_e4m3_gb300 import inputs
from tests import _problems as P
from tests.test_oracle_e4m3 import _torch_decode, _torch_quantize


def _groups(q, Hkv):
    """(b, g) -> the group's rows as a view [q_len, G, D] of q [B, q_len, Hq, D]."""
    B, ql, Hq, D = q.shape
    G = Hq // Hkv
    return {(b, g): q[b, :, g * G:(g + 1) * G, :] for b in range(B) for g in range(Hkv)}


def _library_route(q, Hkv):
    """amax by numpy, the scale by one binary32 division, codes by the torch cast."""
    codes = np.zeros(q.shape, np.uint8)
    scales = np.zeros((q.shape[0], Hkv), np.float32)
    B, ql, Hq, D = q.shape
    G = Hq // Hkv
    for (b, g), rows in _groups(q, Hkv).items():
        amax = np.float32(np.abs(rows.astype(np.float32)).max())
        s = np.float32(amax / np.float32(448.0)) if amax > 0 else np.float32(1.0)
        scales[b, g] = s
        codes[b, :, g * G:(g + 1) * G, :] = _torch_quantize(rows, float(s))
    return codes, scales


@pytest.mark.parametrize("name", ["tiny", "tiny_verify", "verify"])
def test_q_groups_match_library_cast(name):
    w = inputs.get(name)
    q = inputs.queries(w, 0).numpy()   # the full-size verify query: [64, 4, 32, 128]
    Hkv = w.num_kv_heads
    codes, scales = oracle.quantize_q_groups(q, Hkv)
    ref_codes, ref_scales = _library_route(q, Hkv)
    assert np.array_equal(scales, ref_scales)
    assert np.array_equal(codes, ref_codes)


def test_group_maximum_maps_to_448_and_bounds_hold():
    pr = P.host_problem("tiny_verify")
    Hkv = pr.w.num_kv_heads
    codes, scales = oracle.quantize_q_groups(pr.q, Hkv)
    G = pr.w.num_q_heads // Hkv
    for (b, g), rows in _groups(pr.q, Hkv).items():
        c = codes[b, :, g * G:(g + 1) * G, :]
        vals = _torch_decode(c)
        a = np.abs(rows.astype(np.float64))
        k = np.unravel_index(np.argmax(a), a.shape)
        assert abs(vals[k]) == 448.0
        assert np.abs(vals).max() == 448.0
        # error bound: half an E4M3 ulp of the value's binade, 2^-10 below 2^-6
        v = a / float(scales[b, g])
        binade = np.floor(np.log2(np.maximum(v, 2.0 ** -6)))
        bound = np.where(v < 2.0 ** -6, 2.0 ** -10, 2.0 ** (binade - 4))
        # (plus the binary32 rounding of the quotient the method takes first)
        assert (np.abs(np.abs(vals) - v) <= bound + 2.0 ** -23 * v).all()


def test_group_scope_and_power_of_two_scaling():
    pr = P.host_problem("tiny_verify")
    Hkv = pr.w.num_kv_heads
    G = pr.w.num_q_heads // Hkv
    codes, scales = oracle.quantize_q_groups(pr.q, Hkv)
    # a group's values scaled by 2^3: its codes stay, its scale is 8x; the rest is unchanged
    q2 = pr.q.copy()
    q2[1, :, G:2 * G, :] = (q2[1, :, G:2 * G, :].astype(np.float32) * 8).astype(np.float16)
    codes2, scales2 = oracle.quantize_q_groups(q2, Hkv)
    assert np.array_equal(codes2, codes)
    assert scales2[1, 1] == np.float32(8) * scales[1, 1]
    mask = np.ones_like(scales, bool)
    mask[1, 1] = False
    assert np.array_equal(scales2[mask], scales[mask])
    # a larger value in one row of the window changes the whole group's scale (all rows, all heads)
    q3 = pr.q.copy()
    q3[0, 3, 0, 5] = np.float16(1000.0)
    codes3, scales3 = oracle.quantize_q_groups(q3, Hkv)
    assert scales3[0, 0] == np.float32(np.float32(1000.0) / np.float32(448.0))
    assert not np.array_equal(codes3[0, 0, :G], codes[0, 0, :G])
    assert np.array_equal(codes3[0, :, G:], codes[0, :, G:])


def _grid_query(pr, rng):
    """A query whose every group is already on a scaled E4M3 grid: codes c with
    one +-448 per group and the scale 2^-(g + 2b)."""
    B, ql, Hq, D = pr.q.shape
    Hkv = pr.w.num_kv_heads
    G = Hq // Hkv
    codes = rng.integers(0, 256, size=pr.q.shape).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3A            # no NaN codes
    codes[(codes & 0x7F) == 0x7E] = 0x30            # the group maximum is placed below
    q = np.zeros(pr.q.shape, np.float16)
    scales = np.zeros((B, Hkv), np.float32)
    for b in range(B):
        for g in range(Hkv):
            codes[b, 0, g * G, 0] = 0xFE if (b + g) % 2 else 0x7E
            s = 2.0 ** -(g + 2 * b)
            scales[b, g] = s
            blk = codes[b, :, g * G:(g + 1) * G, :]
            q[b, :, g * G:(g + 1) * G, :] = (_torch_decode(blk) * s).astype(np.float16)
    # every value is exact in fp16 (E4M3 values times 2^-k stay in the fp16 range here)
    assert np.array_equal(q.astype(np.float64), np.concatenate(
        [(_torch_decode(codes[:, :, g * G:(g + 1) * G]) * scales[:, g][:, None, None, None])
         for g in range(Hkv)], axis=2))
    return q, codes, scales


@pytest.mark.parametrize("name", ["tiny", "tiny_verify"])
def test_grid_query_is_reproduced_exactly(name):
    pr = P.host_problem(name)
    q, codes, scales = _grid_query(pr, np.random.default_rng(11))
    c2, s2 = oracle.quantize_q_groups(q, pr.w.num_kv_heads)
    assert np.array_equal(c2, codes)
    assert np.array_equal(s2, scales)
    # the quantised query is the query: the two attentions are the same binary64 numbers
    kc, vc, ks, vs = P.oracle_pools(pr)
    bt, lens = pr.layout.block_tables, pr.layout.lens
    a, _ = oracle.attention(q, kc, vc, bt, lens, ks, vs)
    b, _ = oracle.attention(q, kc, vc, bt, lens, ks, vs, fp8_q=True)
    assert np.array_equal(a, b)
    o1, m1, l1, _ = oracle.attention_partials(q, kc, vc, bt, lens, 3, ks, vs)
    o2, m2, l2, _ = oracle.attention_partials(q, kc, vc, bt, lens, 3, ks, vs, fp8_q=True)
    assert np.array_equal(o1, o2) and np.array_equal(m1, m2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("name", ["tiny", "tiny_verify"])
def test_fp8_q_attention_vs_library_softmax(name):
    pr = P.host_problem(name)
    Hkv = pr.w.num_kv_heads
    G = pr.w.num_q_heads // Hkv
    kc, vc, ks, vs = P.oracle_pools(pr)
    bt, lens = pr.layout.block_tables, pr.layout.lens
    codes, scales = _library_route(pr.q, Hkv)
    qhat = _torch_decode(codes) * np.repeat(scales, G, axis=1)[:, None, :, None].astype(np.float64)
    ref = P.torch_reference(qhat, P.torch_dequant(kc, ks), P.torch_dequant(vc, vs), bt, lens, pr.w.q_len)
    got, flags = oracle.attention(pr.q, kc, vc, bt, lens, ks, vs, fp8_q=True)
    assert flags == 0
    assert np.allclose(got, ref, rtol=1e-10, atol=1e-12)
    # the quantised query is a different computation: with the outlier channels
    # of this workload (x20 in q and k) the scores reach about 100, and a few
    # per cent of relative error in q moves them by whole units
    base, _ = oracle.attention(pr.q, kc, vc, bt, lens, ks, vs)
    assert not np.array_equal(got, base)


def test_all_zero_group_gives_the_mean_of_v():
    pr = P.host_problem("tiny")
    Hkv = pr.w.num_kv_heads
    G = pr.w.num_q_heads // Hkv
    q = pr.q.copy()
    q[0, :, 0:G, :] = 0
    codes, scales = oracle.quantize_q_groups(q, Hkv)
    assert scales[0, 0] == 1.0 and not codes[0, :, 0:G].any()
    kc, vc, ks, vs = P.oracle_pools(pr)
    bt, lens = pr.layout.block_tables, pr.layout.lens
    got, _ = oracle.attention(q, kc, vc, bt, lens, ks, vs, fp8_q=True)
    L = int(lens[0])
    pos = np.arange(L)
    vals = P.torch_dequant(vc, vs)[bt[0, pos // 4], 0, pos % 4, :]
    assert np.allclose(got[0, 0, :G], vals.mean(axis=0), rtol=1e-12, atol=1e-14)
