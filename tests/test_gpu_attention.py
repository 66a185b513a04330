"""GPU parity of split-K paged attention (E4M3 and fp16 twins) against the
oracle, element by element, on the small workloads and edge cases."""
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


def _oracle_out(dp, topk=True, lens=None, bt=None, q=None):
    pr = dp.host
    kc, vc, ks, vs = P.oracle_pools(pr, dp.e4m3, (dp.k_scale, dp.v_scale) if dp.e4m3 else None)
    out, flags = oracle.attention(pr.q if q is None else q, kc, vc,
                                  pr.layout.block_tables if bt is None else bt,
                                  pr.layout.lens if lens is None else lens, ks, vs,
                                  pr.topk_idx if topk else None, pr.topk_lens if topk else None)
    return out


@pytest.mark.parametrize("name", ["tiny", "tiny_verify"])
@pytest.mark.parametrize("e4m3", [True, False])
@pytest.mark.parametrize("S", [1, 2, 4, 0])
def test_tiny_matches_oracle(name, e4m3, S):
    dp = G.device_problem(P.host_problem(name), e4m3)
    out = G.run_attention(dp, num_splits=S)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    G.assert_close(out.float().cpu().numpy(), _oracle_out(dp), f"{name} e4m3={e4m3} S={S}")


@pytest.mark.parametrize("name", ["tiny", "tiny_verify"])
@pytest.mark.parametrize("S", [1, 2, 4, 0])
def test_bitcast_decoder_matches_oracle_and_hardware_conversion(name, S):
    """The pages' bitcast decoder (value * 2^-8, the 2^8 folded into the
    hoisted scales) against the oracle, and bit for bit against the hardware
    conversion: the two decode every byte to the same value up to a power of
    two, so every product and sum scales exactly."""
    dp = G.device_problem(P.host_problem(name), True)
    hw = G.run_attention(dp, num_splits=S)
    bc = G.run_attention(dp, num_splits=S, bitcast_decode=True)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    G.assert_close(bc.float().cpu().numpy(), _oracle_out(dp), f"bitcast {name} S={S}")
    assert torch.equal(bc.view(torch.int16), hw.view(torch.int16))


def test_bitcast_decoder_topk_and_nan_slots():
    w = inputs.get("tiny_verify", topk=24, topk_fraction=0.5)
    dp = G.device_problem(P.host_problem(w), True, sentinel=0x7F)   # NaN codes in unowned slots
    for S in (1, 3):
        hw = G.run_attention(dp, num_splits=S)
        bc = G.run_attention(dp, num_splits=S, bitcast_decode=True)
        torch.cuda.synchronize()
        assert dp.err.item() == 0
        G.assert_close(bc.float().cpu().numpy(), _oracle_out(dp), f"bitcast top-k S={S}")
        assert torch.equal(bc.view(torch.int16), hw.view(torch.int16))


@pytest.mark.parametrize("name", ["tiny", "tiny_verify"])
@pytest.mark.parametrize("e4m3", [True, False])
@pytest.mark.parametrize("split_pages,extra", [(2, 1), (8, 0), (16, 3)])
def test_fixed_size_split_partials_match_oracle(name, e4m3, split_pages, extra):
    dp = G.device_problem(P.host_problem(name), e4m3)
    S = -(-dp.block_tables.shape[1] // split_pages) + extra
    ws, p = G.run_attention(dp, num_splits=S, partial=True, split_pages=split_pages)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    o, m, l = [x.cpu().numpy() for x in kvq.workspace_views(ws, p)]
    pr = dp.host
    kc, vc, ks, vs = P.oracle_pools(pr, e4m3, (dp.k_scale, dp.v_scale) if e4m3 else None)
    ro, rm, rl, _ = oracle.attention_partials(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens,
                                              S, ks, vs, split_pages=split_pages)
    nonempty = rl > 0
    assert np.array_equal(l > 0, nonempty)
    assert np.isneginf(m[~nonempty]).all()
    G.assert_close(m[nonempty], rm[nonempty], "tmp_max", atol=1e-4, rtol=1e-5)
    G.assert_close(l[nonempty], rl[nonempty], "tmp_sum", atol=1e-4, rtol=2e-3)
    G.assert_close(o[nonempty], ro[nonempty], "tmp_out")
    out = G.run_attention(dp, num_splits=0, split_pages=split_pages)
    torch.cuda.synchronize()
    G.assert_close(out.float().cpu().numpy(), _oracle_out(dp), f"{name} split_pages={split_pages}")


@pytest.mark.parametrize("split_pages", [1, 3])
def test_fixed_size_splits_topk_match_oracle(split_pages):
    w = inputs.get("tiny_verify", topk=24, topk_fraction=0.5)
    for e4m3 in (True, False):
        dp = G.device_problem(P.host_problem(w), e4m3)
        out = G.run_attention(dp, num_splits=0, split_pages=split_pages)
        torch.cuda.synchronize()
        assert dp.err.item() == 0
        G.assert_close(out.float().cpu().numpy(), _oracle_out(dp), f"top-k split_pages={split_pages}")


@pytest.mark.parametrize("S", [16, 40])
def test_combine_with_many_splits(S):
    """Split lists of 16 or more go to the four-warps-per-row combine."""
    dp = G.device_problem(P.host_problem("tiny_verify"), True)
    out = G.run_attention(dp, num_splits=S)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    G.assert_close(out.float().cpu().numpy(), _oracle_out(dp), f"S={S}")


@pytest.mark.parametrize("name", ["tiny", "tiny_verify"])
@pytest.mark.parametrize("e4m3", [True, False])
def test_workspace_partials_match_oracle(name, e4m3):
    dp = G.device_problem(P.host_problem(name), e4m3)
    S = 3
    ws, p = G.run_attention(dp, num_splits=S, partial=True)
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


def test_topk_matches_oracle():
    w = inputs.get("tiny_verify", topk=24, topk_fraction=0.5)
    for e4m3 in (True, False):
        dp = G.device_problem(P.host_problem(w), e4m3)
        for S in (1, 2):
            out = G.run_attention(dp, num_splits=S)
            torch.cuda.synchronize()
            assert dp.err.item() == 0
            G.assert_close(out.float().cpu().numpy(), _oracle_out(dp), f"topk e4m3={e4m3} S={S}")


def test_topk_long_lists_and_duplicates_of_dense():
    """top-k = every position (list longer than one 32-token stage) equals dense."""
    pr = P.host_problem("tiny_verify")
    dp = G.device_problem(pr)
    dense = G.run_attention(dp, num_splits=2, topk=False)
    Lmax = int(pr.layout.lens.max())
    ti = np.zeros((2, 2, Lmax), np.int32)
    for b in range(2):
        ti[b, :, : pr.layout.lens[b]] = np.arange(pr.layout.lens[b])
    dp.topk_idx, dp.topk_lens = G.to_dev(ti), G.to_dev(pr.layout.lens)
    full = G.run_attention(dp, num_splits=2)
    torch.cuda.synchronize()
    G.assert_close(full.float().cpu().numpy(), dense.float().cpu().numpy().astype(np.float64),
                   "topk-all vs dense", atol=1e-3, rtol=1e-3)


def test_page_permutation_is_bit_identical():
    pr = P.host_problem("tiny_verify")
    dp = G.device_problem(pr)
    out = G.run_attention(dp, num_splits=2)
    perm = torch.from_numpy(np.random.default_rng(5).permutation(pr.P)).cuda()
    inv = torch.argsort(perm)
    kc, vc = dp.k_cache[perm].contiguous(), dp.v_cache[perm].contiguous()
    bt = dp.block_tables.clone()
    m = bt >= 0
    bt[m] = inv[bt[m].long()].int()
    out2 = G.run_attention(dp, num_splits=2, block_tables=bt, k_cache=kc, v_cache=vc)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


def test_split_count_invariance():
    dp = G.device_problem(P.host_problem("tiny"))
    outs = [G.run_attention(dp, num_splits=S).float().cpu().numpy() for S in (1, 2, 4, 7, 64)]
    for o in outs[1:]:
        G.assert_close(o, outs[0].astype(np.float64), "split invariance", atol=1e-3, rtol=1e-3)


def test_gpu_verify_row_equals_shorter_decode():
    pr = P.host_problem("tiny_verify")
    dp = G.device_problem(pr)
    full = G.run_attention(dp, num_splits=2).float().cpu().numpy()
    for i in range(4):
        lens = G.to_dev(pr.layout.lens - 4 + i + 1)
        qi = dp.q[:, i:i + 1].contiguous()
        dec = G.run_attention(dp, num_splits=2, context_lens=lens, q=qi).float().cpu().numpy()
        G.assert_close(full[:, i], dec[:, 0].astype(np.float64), f"row {i}", atol=1e-3, rtol=1e-3)


# ---------------------------------------------------------------------------
# shapes and edge cases

@pytest.mark.parametrize("lens,q_len,G_,D", [
    ([1, 2, 3, 4], 1, 8, 128),           # one token, page tails
    ([236, 1000, 33], 1, 8, 128),        # partial last stage landing in a reused ring slot
    ([236, 1000, 33], 4, 8, 128),
    ([4, 5, 9, 33], 4, 8, 128),          # verify window covering the whole context
    ([257, 31, 64, 100], 1, 16, 64),     # 16 query heads per kv head
    ([70, 130], 4, 16, 64),              # 64 query rows per kv head (largest)
    ([45, 200], 3, 5, 128),              # odd group, odd q_len
    ([600, 2], 2, 1, 64),                # MHA-like group of 1
])
@pytest.mark.parametrize("e4m3", [True, False])
def test_shapes_match_oracle(lens, q_len, G_, D, e4m3):
    w = inputs.Workload("edge", 11, 1, len(lens), q_len, 2 * G_, 2, D, 0,
                        "list:" + ",".join(map(str, lens)), calib_tokens=64)
    dp = G.device_problem(P.host_problem(w), e4m3)
    for S in (1, 3):
        out = G.run_attention(dp, num_splits=S)
        torch.cuda.synchronize()
        assert dp.err.item() == 0
        G.assert_close(out.float().cpu().numpy(), _oracle_out(dp), f"{lens} q{q_len} G{G_} D{D} S{S}")


@pytest.mark.parametrize("q_len", [1, 4])
@pytest.mark.parametrize("e4m3", [True, False])
def test_many_sequences_in_longest_first_order(q_len, e4m3):
    """Seventy sequences whose lengths fall in many work classes, with ties,
    a shortest possible one and a top-k share: the kernels attend them in
    longest-first order (a scan over three 32-sequence groups), which must
    not change which sequence's rows a CTA writes.  q_len 4 with 8 query
    heads per kv head runs the tensor-core kernel, q_len 1 the split kernel."""
    rng = np.random.default_rng(7)
    lens = rng.integers(30, 420, size=70)
    lens[10:15] = 300                          # ties inside one class
    lens[40] = 30
    lens[69] = 419
    w = inputs.Workload("many", 12, 1, 70, q_len, 16, 2, 128, 0, "list:" + ",".join(map(str, lens)),
                        calib_tokens=64, topk=24, topk_fraction=0.3)
    dp = G.device_problem(P.host_problem(w), e4m3)
    for S in (1, 3):
        out = G.run_attention(dp, num_splits=S)
        torch.cuda.synchronize()
        assert dp.err.item() == 0
        G.assert_close(out.float().cpu().numpy(), _oracle_out(dp), f"70 sequences q{q_len} S{S}")


@pytest.mark.parametrize("e4m3", [True, False])
@pytest.mark.parametrize("q_len", [1, 3])
def test_split_kernel_longest_first_is_bit_identical(e4m3, q_len):
    """KVQ_ATTN_LONGEST_FIRST on the split kernel: seventy sequences of varied
    lengths (ties, a top-k share) over a grid of several waves; which CTA takes
    which (sequence, split) must not change a bit of the outputs or partials."""
    rng = np.random.default_rng(9)
    lens = rng.integers(5, 900, size=70)
    lens[20:26] = 640
    w = inputs.Workload("many", 13, 1, 70, q_len, 8, 2, 128, 0, "list:" + ",".join(map(str, lens)),
                        calib_tokens=64, topk=40, topk_fraction=0.3)
    dp = G.device_problem(P.host_problem(w), e4m3)
    ref = _oracle_out(dp)
    for S in (2, 5):
        base = G.run_attention(dp, num_splits=S, mma_sync=True)
        lpt = G.run_attention(dp, num_splits=S, mma_sync=True, longest_first=True)
        ws0, p0 = G.run_attention(dp, num_splits=S, mma_sync=True, partial=True)
        ws1, p1 = G.run_attention(dp, num_splits=S, mma_sync=True, partial=True, longest_first=True)
        torch.cuda.synchronize()
        assert dp.err.item() == 0
        assert torch.equal(base.view(torch.int16), lpt.view(torch.int16))
        for a, b in zip(kvq.workspace_views(ws0, p0), kvq.workspace_views(ws1, p1)):
            ok = torch.isnan(a) == torch.isnan(b)     # tmp_out of empty splits stays unwritten (NaN fill)
            assert ok.all() and torch.equal(torch.nan_to_num(a), torch.nan_to_num(b))
        G.assert_close(lpt.float().cpu().numpy(), ref, f"longest first q{q_len} S{S} e4m3={e4m3}")


@pytest.mark.parametrize("q_len", [1, 3])
def test_bitcast_decoder_longest_first_is_bit_identical(q_len):
    """The bitcast decoder's longest-first instances over the same seventy
    sequences: outputs and partials bit-identical to the hardware conversion
    in index order (the decoders agree on every finite code, and the order is
    a scheduling choice only)."""
    rng = np.random.default_rng(9)
    lens = rng.integers(5, 900, size=70)
    lens[20:26] = 640
    w = inputs.Workload("many", 13, 1, 70, q_len, 8, 2, 128, 0, "list:" + ",".join(map(str, lens)),
                        calib_tokens=64, topk=40, topk_fraction=0.3)
    dp = G.device_problem(P.host_problem(w), True)
    ref = _oracle_out(dp)
    for S in (2, 5):
        base = G.run_attention(dp, num_splits=S, mma_sync=True)
        bc = G.run_attention(dp, num_splits=S, mma_sync=True, bitcast_decode=True, longest_first=True)
        ws0, p0 = G.run_attention(dp, num_splits=S, mma_sync=True, partial=True)
        ws1, p1 = G.run_attention(dp, num_splits=S, mma_sync=True, partial=True, bitcast_decode=True,
                                  longest_first=True)
        torch.cuda.synchronize()
        assert dp.err.item() == 0
        assert torch.equal(base.view(torch.int16), bc.view(torch.int16))
        for a, b in zip(kvq.workspace_views(ws0, p0), kvq.workspace_views(ws1, p1)):
            ok = torch.isnan(a) == torch.isnan(b)     # tmp_out of empty splits stays unwritten (NaN fill)
            assert ok.all() and torch.equal(torch.nan_to_num(a), torch.nan_to_num(b))
        G.assert_close(bc.float().cpu().numpy(), ref, f"bitcast longest first q{q_len} S{S}")


@pytest.mark.parametrize("e4m3", [True, False])
@pytest.mark.parametrize("name", ["tiny", "tiny_verify"])
def test_nan_bits_in_unowned_slots_do_not_leak(name, e4m3):
    """Unowned slots (the tail of each sequence's last page, pages nobody
    owns) filled with NaN patterns: 0x7F (E4M3 NaN) or 0x7F7F (fp16 NaN)."""
    dp = G.device_problem(P.host_problem(name), e4m3, sentinel=0x7F)
    for S in (1, 2, 3):
        out = G.run_attention(dp, num_splits=S)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert np.isfinite(got).all()
        G.assert_close(got, _oracle_out(dp), f"{name} e4m3={e4m3} S={S} NaN sentinel")


def test_more_splits_than_pages_gives_empty_splits():
    dp = G.device_problem(P.host_problem("tiny"))
    out = G.run_attention(dp, num_splits=40)     # sequence 0 has 10 pages: 30 empty splits
    torch.cuda.synchronize()
    G.assert_close(out.float().cpu().numpy(), _oracle_out(dp), "S=40")


def test_bad_entries_are_flagged_and_skipped():
    pr = P.host_problem("tiny")
    dp = G.device_problem(pr)
    bt = dp.block_tables.clone()
    bt[1, 3] = pr.P + 100                      # out of the pool
    dp.err.zero_()
    out = G.run_attention(dp, num_splits=2, block_tables=bt)
    torch.cuda.synchronize()
    assert dp.err.item() & kvq.DEV_BAD_PAGE
    ref_bt = pr.layout.block_tables.copy()
    ref_bt[1, 3] = pr.P + 100
    G.assert_close(out.float().cpu().numpy(), _oracle_out(dp, bt=ref_bt), "bad page skipped")
    # a context longer than the block table allows: the row is zero and flagged
    dp.err.zero_()
    lens = dp.context_lens.clone()
    lens[0] = 10_000
    out = G.run_attention(dp, num_splits=2, context_lens=lens)
    torch.cuda.synchronize()
    assert dp.err.item() & kvq.DEV_BAD_LEN
    assert (out[0] == 0).all()
    # top-k entries outside [0, L)
    dp.err.zero_()
    ti = torch.tensor([[[1, 2, 500]] * 2, [[0, 5, -3]] * 2], dtype=torch.int32, device="cuda")
    dp.topk_idx, dp.topk_lens = ti, torch.tensor([3, 3], dtype=torch.int32, device="cuda")
    G.run_attention(dp, num_splits=1)
    torch.cuda.synchronize()
    assert dp.err.item() & kvq.DEV_BAD_TOPK


def test_fp16_workspace_is_refused():
    dp = G.device_problem(P.host_problem("tiny"))
    p = kvq.attn_params(dp.q, 2, dp.block_tables.shape[1], 2)
    ws16 = torch.empty(kvq.workspace_bytes(p) // 2, dtype=torch.float16, device="cuda")
    with pytest.raises(TypeError):
        kvq.paged_decode_attn_e4m3(dp.q, dp.k_cache, dp.v_cache, dp.block_tables,
                                   dp.context_lens, dp.k_scale, dp.v_scale, ws16, num_splits=2)


def test_short_workspace_is_refused_before_launch():
    dp = G.device_problem(P.host_problem("tiny"))
    p = kvq.attn_params(dp.q, 2, dp.block_tables.shape[1], 2)
    ws = torch.empty(kvq.workspace_bytes(p) // 4 - 64, dtype=torch.float32, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.paged_decode_attn_e4m3(dp.q, dp.k_cache, dp.v_cache, dp.block_tables,
                                   dp.context_lens, dp.k_scale, dp.v_scale, ws, num_splits=2)
    assert e.value.status == -3


def test_empty_batch_is_a_no_op():
    q = torch.empty((0, 1, 8, 64), dtype=torch.float16, device="cuda")
    kc = torch.zeros((4, 2, 4, 64), dtype=torch.uint8, device="cuda")
    bt = torch.zeros((0, 1), dtype=torch.int32, device="cuda")
    cl = torch.zeros((0,), dtype=torch.int32, device="cuda")
    p = kvq.attn_params(q, 2, 1, 1)
    ws = torch.empty(64, dtype=torch.float32, device="cuda")
    out = kvq.paged_decode_attn_e4m3(q, kc, kc, bt, cl, 0.1, 0.1, ws, num_splits=1)
    assert out.shape == q.shape


def test_e4m3_error_vs_unquantised_is_reported():
    """Not gated: E4M3 output against fp64 attention over the unquantised fp16 K/V."""
    pr = P.host_problem("tiny_verify")
    dp = G.device_problem(pr)
    out = G.run_attention(dp, num_splits=2).float().cpu().numpy()
    kc, vc, _, _ = P.oracle_pools(pr, e4m3=False)
    ref, _ = oracle.attention(pr.q, kc, vc, pr.layout.block_tables, pr.layout.lens)
    err = np.abs(out - ref)
    cos = (out * ref).sum(-1) / (np.linalg.norm(out, axis=-1) * np.linalg.norm(ref, axis=-1))
    print(f"E4M3 vs unquantised: max abs {err.max():.4g}, mean cos {cos.mean():.6f}")
    assert np.isfinite(out).all() and cos.mean() > 0.9
