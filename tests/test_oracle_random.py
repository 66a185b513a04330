"""Seeded random problems for the oracle's attention, beyond the fixed small
cases: batch, window length (1..4), GQA ratio, head_dim, context lengths that
end anywhere inside a page, shuffled and partly unused pools, E4M3 codes over
the whole finite range with random per-layer scales, fp16 pools, top-k lists
on some sequences (also listing positions inside the verify window), and
sm_scale overrides.  Each is checked against the library route of the test
suite (numpy gather of the dequantised pools, explicit causal / list mask,
torch.softmax in binary64), and the split partials against the full result
through the oracle's combine."""
import numpy as np
import pytest

import oracle
from tests import _problems as P

_FINITE = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def _random_problem(rng):
    B = int(rng.integers(1, 4))
    q_len = int(rng.integers(1, 5))
    Hkv = int(rng.integers(1, 3))
    G = int(rng.integers(1, 5))
    D = int(rng.choice([8, 16, 64]))
    lens = rng.integers(q_len, 61, size=B).astype(np.int32)
    pages = (lens + 3) // 4
    max_pages = int(pages.max()) + int(rng.integers(0, 3))
    P_ = int(pages.sum()) + int(rng.integers(0, 5))
    perm = rng.permutation(P_).astype(np.int32)
    bt = np.full((B, max_pages), -1, np.int32)
    o = 0
    for b in range(B):
        bt[b, :pages[b]] = perm[o:o + pages[b]]
        o += pages[b]
    q = (rng.standard_normal((B, q_len, G * Hkv, D)) * rng.uniform(0.2, 2.0)).astype(np.float16)
    topk_idx = topk_lens = None
    if rng.random() < 0.5:
        K = int(rng.integers(1, 20))
        topk_idx = np.zeros((B, Hkv, K), np.int32)
        topk_lens = np.zeros(B, np.int32)
        for b in range(B):
            if rng.random() < 0.6:
                n = int(min(K, lens[b], rng.integers(1, K + 1)))
                topk_lens[b] = n
                for g in range(Hkv):
                    topk_idx[b, g, :n] = np.sort(rng.choice(int(lens[b]), size=n, replace=False))
    sm = None if rng.random() < 0.5 else float(rng.uniform(0.05, 0.5))
    return q, bt, lens, P_, Hkv, D, topk_idx, topk_lens, sm


@pytest.mark.parametrize("seed", range(24))
@pytest.mark.parametrize("e4m3", [True, False])
def test_random_problems_match_the_library_route(seed, e4m3):
    rng = np.random.default_rng([20, seed, int(e4m3)])
    q, bt, lens, P_, Hkv, D, ti, tl, sm = _random_problem(rng)
    q_len = q.shape[1]
    if e4m3:
        kc = rng.choice(_FINITE, size=(P_, Hkv, 4, D))
        vc = rng.choice(_FINITE, size=(P_, Hkv, 4, D))
        ks, vs = float(np.float32(rng.uniform(1e-3, 0.05))), float(np.float32(rng.uniform(1e-3, 0.05)))
        kv_k, kv_v = P.torch_dequant(kc, ks), P.torch_dequant(vc, vs)
    else:
        kc = (rng.standard_normal((P_, Hkv, 4, D)) * 2).astype(np.float16)
        vc = (rng.standard_normal((P_, Hkv, 4, D)) * 2).astype(np.float16)
        ks = vs = 1.0
        kv_k, kv_v = kc.astype(np.float64), vc.astype(np.float64)
    got, flags = oracle.attention(q, kc, vc, bt, lens, ks, vs, ti, tl, sm_scale=sm)
    assert flags == 0
    ref = P.torch_reference(q, kv_k, kv_v, bt, lens, q_len, ti, tl, sm_scale=sm)
    # rows whose key set is empty (a top-k list with nothing inside the window) are 0 in
    # the oracle (empty key set) and NaN in the library softmax
    empty = np.isnan(ref)
    assert (got[empty] == 0).all()
    assert np.allclose(got[~empty], ref[~empty], rtol=1e-9, atol=1e-12)
    S = int(rng.integers(1, 7))
    o, m, l, f2 = oracle.attention_partials(q, kc, vc, bt, lens, S, ks, vs, ti, tl, sm_scale=sm)
    assert f2 == 0
    merged = oracle.combine(o, m, l).transpose(0, 2, 1, 3)
    assert np.allclose(merged, got, rtol=1e-9, atol=1e-12)
