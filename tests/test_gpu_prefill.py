"""GPU parity of chunked-prefill attention (E4M3 and fp16 twins) against the
oracle, element by element on small chunks (several query and key tiles,
ragged tails, a causal diagonal off the tile grid), and on sampled rows of
the full 8192-token chunk."""
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


def _problem(lens, n, Hq=16, Hkv=2, wid=21):
    w = inputs.Workload("prefill_case", wid, 1, len(lens), n, Hq, Hkv, 128, 0,
                        "list:" + ",".join(map(str, lens)), calib_tokens=64)
    return P.host_problem(w)


def _oracle(dp):
    pr = dp.host
    kc, vc, ks, vs = P.oracle_pools(pr, dp.e4m3, (dp.k_scale, dp.v_scale) if dp.e4m3 else None)
    out, flags = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens, ks, vs)
    return out


def _prefill(dp, chunks=None, max_q_len=None, lens=None):
    """Prefill over the last chunks[b] query rows of each sequence (default:
    all q_len rows).  Returns the packed output and q_start."""
    B, n, Hq, D = dp.q.shape
    chunks = [n] * B if chunks is None else chunks
    q = torch.cat([dp.q[b, n - c:] for b, c in enumerate(chunks)]).contiguous()
    q_start = torch.tensor(np.concatenate([[0], np.cumsum(chunks)]), dtype=torch.int32, device=q.device)
    cl = dp.context_lens if lens is None else lens
    p = kvq.PrefillParams(B, Hq, dp.k_cache.shape[1], D, dp.block_tables.shape[1],
                          max_q_len or max(max(chunks), 1), q.shape[0], 0.0, 0)
    ws = kvq.alloc_prefill_workspace(p, q.device)
    out = torch.full_like(q, float("nan")) if q.numel() else torch.empty_like(q)
    if dp.e4m3:
        kvq.paged_prefill_attn_e4m3(q, dp.k_cache, dp.v_cache, dp.block_tables, cl, q_start, dp.k_scale,
                                    dp.v_scale, ws, out=out, max_q_len=p.max_q_len, err_flag=dp.err)
    else:
        kvq.paged_prefill_attn_fp16(q, dp.k_cache, dp.v_cache, dp.block_tables, cl, q_start, ws, out=out,
                                    max_q_len=p.max_q_len, err_flag=dp.err)
    torch.cuda.synchronize()
    return out, chunks


@pytest.mark.parametrize("lens,n", [
    ([300, 200], 200),          # 2 query tiles (ragged), up to 3 key tiles, diagonal 100 keys off the grid
    ([37, 129], 1),             # one-token chunks: the decode definition
    ([129, 520, 256], 129),     # a chunk one past a tile; key tiles 2..5
    ([700], 384),               # 3 full query tiles over 316 earlier keys
])
@pytest.mark.parametrize("e4m3", [True, False])
def test_prefill_matches_oracle(lens, n, e4m3):
    dp = G.device_problem(_problem(lens, n), e4m3)
    out, _ = _prefill(dp)
    assert dp.err.item() == 0
    B, _, Hq, D = dp.q.shape
    G.assert_close(out.float().cpu().numpy().reshape(B, n, Hq, D), _oracle(dp), f"prefill {lens} n={n}")


@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (32, 2), (12, 4)])
def test_prefill_group_sizes(Hq, Hkv):
    """MHA (one query head per kv head), 16 query heads per kv head, and an
    odd group of 3, over chunks that end mid-tile."""
    dp = G.device_problem(_problem([333, 190], 190, Hq=Hq, Hkv=Hkv, wid=26), True)
    out, _ = _prefill(dp)
    assert dp.err.item() == 0
    B, n, _, D = dp.q.shape
    G.assert_close(out.float().cpu().numpy().reshape(B, n, Hq, D), _oracle(dp), f"Hq={Hq} Hkv={Hkv}")


def test_prefill_is_deterministic_and_split_invariant():
    """Two calls give the same bits; and a chunk attended in one call equals
    the same rows attended as two consecutive chunks of 100 and 156 tokens
    (the second with the first already in its context)."""
    pr = _problem([512], 256, wid=27)
    dp = G.device_problem(pr, True)
    a, _ = _prefill(dp)
    b, _ = _prefill(dp)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    # the first 100 rows as a chunk of a 356-token context
    lens = dp.context_lens.clone()
    lens[0] = 512 - 156
    dp2 = G.device_problem(pr, True)
    dp2.q = dp.q[:, :100].contiguous()
    c, _ = _prefill(dp2, lens=lens)
    G.assert_close(c.float().cpu().numpy(), a.float().cpu().numpy()[:100], "chunk split")


@pytest.mark.parametrize("e4m3", [True, False])
def test_prefill_chunks_of_different_lengths(e4m3):
    """Chunks of 200, 0, 1 and 77 tokens packed back to back: each is the
    tail of the q_len window, so its rows equal the oracle's rows for the
    same absolute positions; the empty chunk writes nothing."""
    dp = G.device_problem(_problem([250, 300, 260, 400], 200, wid=22), e4m3)
    chunks = [200, 0, 1, 77]
    out, _ = _prefill(dp, chunks)
    assert dp.err.item() == 0
    ref = _oracle(dp)
    got = out.float().cpu().numpy()
    o = 0
    for b, c in enumerate(chunks):
        if c:
            G.assert_close(got[o:o + c], ref[b, 200 - c:], f"chunk {b} of {c}")
        o += c


@pytest.mark.parametrize("e4m3", [True, False])
def test_prefill_nan_bits_in_unowned_slots_do_not_leak(e4m3):
    dp = G.device_problem(_problem([301, 150], 150, wid=23), e4m3, sentinel=0x7F)
    out, _ = _prefill(dp)
    got = out.float().cpu().numpy()
    assert np.isfinite(got).all()
    B, n, Hq, D = dp.q.shape
    G.assert_close(got.reshape(B, n, Hq, D), _oracle(dp), "NaN sentinel pools")


def test_prefill_bad_lengths_are_flagged_and_not_written():
    dp = G.device_problem(_problem([300, 200], 200, wid=24))
    lens = dp.context_lens.clone()
    lens[1] = 150                                  # chunk of 200 in a context of 150
    out, _ = _prefill(dp, lens=lens)
    assert dp.err.item() & kvq.DEV_BAD_LEN
    got = out.float().cpu().numpy()
    assert np.isnan(got[200:]).all()              # sequence 1: rows untouched
    G.assert_close(got[:200], _oracle(dp)[0], "the valid sequence")


def test_prefill_bad_page_is_flagged_and_skipped():
    """Keys whose block-table entry lies outside the pool are left out of
    the softmax, as the oracle leaves them out."""
    pr = _problem([300], 100, wid=25)
    dp = G.device_problem(pr)
    dp.block_tables[0, 10] = pr.P + 7              # keys 40..43 point outside the pool
    out, _ = _prefill(dp)
    assert dp.err.item() & kvq.DEV_BAD_PAGE
    kc, vc, ks, vs = P.oracle_pools(pr, True, (dp.k_scale, dp.v_scale))
    bt = pr.layout.block_tables.copy()
    bt[0, 10] = pr.P + 7
    ref, _ = oracle.attention(pr.q, kc, vc, bt, pr.layout.lens, ks, vs)
    G.assert_close(out.float().cpu().numpy().reshape(ref.shape), ref, "bad page skipped")


@pytest.mark.parametrize("e4m3", [True, False])
def test_full_chunk_sampled_rows_match_oracle(e4m3):
    """The 8192-token chunk of the mixed batch (32 q / 4 kv heads), in the
    launch configuration the benchmark times; rows sampled at tile edges.
    Row i of a chunk that fills its context attends keys 0..i, which is the
    decode definition with context i + 1 (checked one row at a time)."""
    w = inputs.get("prefill")
    pr = P.host_problem(w)
    dp = G.device_problem(pr, e4m3)
    out, _ = _prefill(dp)
    assert dp.err.item() == 0
    kc, vc, ks, vs = P.oracle_pools(pr, e4m3, (dp.k_scale, dp.v_scale) if e4m3 else None)
    got = out.float().cpu().numpy()
    for i in (0, 1, 127, 128, 4095, 5000, 8191):
        ref, _ = oracle.attention(pr.q[:, i:i + 1], kc, vc, pr.layout.block_tables,
                                  np.array([i + 1], np.int32), ks, vs)
        G.assert_close(got[i], ref[0, 0], f"row {i}")
