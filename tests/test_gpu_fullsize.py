"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times.

Pools: every byte of the K and V pools -- the quantised (or, for the fp16
arm, copied) tokens and the sentinel of every slot and page that no token
owns -- must equal pools the oracle fills from the same fp16 inputs, for the
decode workload (both arms), decode at 32K context, the long-context
workload, two layers each of the 24-layer verify and mixed workloads and one
layer each of the verify, mixed and long workloads' fp16 arms
(PR "[Model][SM70][FP8] Integrate calibrated E4M3 QSA KV capacity path",
section Changes: the main K/V cache is stored in calibrated E4M3).

The fused step call, which the benchmark times for its dense workloads,
must give whole pools and outputs bit-identical to the append call and the
attention call at full size (decode both arms, decode at 32K, the long
context, a verify layer of both arms).

Attention: sampled (layer, sequence, query head) units that the oracle
recomputes one by one from the same seeded fp16 inputs must match within
atol 2e-3 / rtol 1e-2; the E4M3 K and V bytes of each sampled sequence's kv
head are compared again there.  The oracle computes its own calibrated
scale, which must equal the GPU's.

The oracle runs in a process pool started with "spawn" (workers never
inherit a CUDA context).
"""
import concurrent.futures as cf
import multiprocessing as mp
import os
import shutil
import tempfile

import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_e4m3_gb300 import build, inputs, kvq
from tests import _problems as P

pytestmark = pytest.mark.gpu

DEV = "cuda"


WORKERS = max(2, min(16, os.cpu_count() or 2))


@pytest.fixture(scope="module")
def pool():
    build.build()
    kvq.load()
    oracle.build()
    ex = cf.ProcessPoolExecutor(max_workers=WORKERS, mp_context=mp.get_context("spawn"))
    yield ex
    ex.shutdown(cancel_futures=True)


class Layer:
    """One layer of a workload pushed through the GPU path, in the launch
    configuration bench.py times (longest-first order for batches of varied
    lengths)."""

    def __init__(self, w, layer, lay, e4m3=True, with_prefill=True, bitcast=False, fp8_qk=False, fused=False):
        longest_first = not w.lens.startswith("fixed")
        self.w, self.layer, self.lay, self.e4m3 = w, layer, lay, e4m3
        lens = lay.lens.astype(np.int64)
        total = int(lens.sum())
        self.offs = np.concatenate([[0], np.cumsum(lens)[:-1]])
        self.k = inputs.kv_tokens(w, layer, total, "k", device=DEV)
        self.v = inputs.kv_tokens(w, layer, total, "v", device=DEV)
        self.q = inputs.queries(w, layer, device=DEV)
        shape = (lay.num_pages, w.num_kv_heads, 4, w.head_dim)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        self.err = err
        if e4m3:
            self.kcal = inputs.calibration_draw(w, layer, "k", device=DEV)
            self.vcal = inputs.calibration_draw(w, layer, "v", device=DEV)
            self.ks = kvq.calibrate_scale(self.kcal)
            self.vs = kvq.calibrate_scale(self.vcal)
            self.kc = torch.full(shape, P.SENTINEL, dtype=torch.uint8, device=DEV)
            self.vc = torch.full(shape, P.SENTINEL, dtype=torch.uint8, device=DEV)
            app = lambda k, v, s: kvq.kv_append_e4m3(k, v, s, self.kc, self.vc, self.ks, self.vs, err)
        else:
            self.ks = self.vs = 1.0
            self.kc = torch.empty(shape, dtype=torch.float16, device=DEV)
            self.kc.view(torch.int16).fill_(int(np.int16(np.uint16(P.SENTINEL * 0x101).view(np.int16))))
            self.vc = self.kc.clone()
            app = lambda k, v, s: kvq.kv_append_fp16(k, v, s, self.kc, self.vc, err)
        # the cached history, then this step's tokens (one append call each, as a step does); with
        # `fused`, this step's tokens are appended by the fused step call instead
        step_seq, step_pos = inputs.step_tokens(w, lay)
        for seq, pos in ((inputs.history_tokens(w, lay),) if fused else
                         (inputs.history_tokens(w, lay), (step_seq, step_pos))):
            if seq.size == 0:
                continue
            rows = torch.from_numpy(self.offs[seq] + pos).to(DEV)
            slots = torch.from_numpy(inputs.slot_mapping(lay.block_tables, seq, pos)).to(DEV)
            app(self.k[rows].contiguous(), self.v[rows].contiguous(), slots)
        self.prefill = None
        if w.prefill_chunk and with_prefill:
            pk = inputs.prefill_tokens(w, layer, "k", device=DEV)
            pv = inputs.prefill_tokens(w, layer, "v", device=DEV)
            app(pk, pv, torch.from_numpy(inputs.prefill_slots(lay)[: w.prefill_chunk]).to(DEV))
            self.prefill = (pk, pv)
        self.bt = torch.from_numpy(lay.block_tables).to(DEV)
        self.cl = torch.from_numpy(lay.lens).to(DEV)
        ti, tl = inputs.topk_lists(w, lay.lens)
        self.topk_np = (ti, tl)
        ti_d = tl_d = None
        if ti is not None:
            ti_d, tl_d = torch.from_numpy(ti).to(DEV), torch.from_numpy(tl).to(DEV)
        p = kvq.attn_params(self.q, w.num_kv_heads, lay.block_tables.shape[1], w.num_splits,
                            0 if ti is None else ti.shape[2], split_pages=w.split_pages,
                            longest_first=longest_first)
        self.S = kvq.num_splits(p)
        ws = kvq.alloc_workspace(p, DEV)
        if fused:
            shape4 = (w.batch, w.q_len, w.num_kv_heads, w.head_dim)
            rows = torch.from_numpy(self.offs[step_seq] + step_pos).to(DEV)   # (b, i) order
            kn, vn = self.k[rows].contiguous().view(shape4), self.v[rows].contiguous().view(shape4)
            if e4m3:
                self.out = kvq.paged_decode_step_e4m3(self.q, kn, vn, self.kc, self.vc, self.bt, self.cl, self.ks,
                                                      self.vs, ws, None, w.num_splits, err_flag=err,
                                                      split_pages=w.split_pages, longest_first=longest_first)
            else:
                self.out = kvq.paged_decode_step_fp16(self.q, kn, vn, self.kc, self.vc, self.bt, self.cl, ws, None,
                                                      w.num_splits, err_flag=err, split_pages=w.split_pages,
                                                      longest_first=longest_first)
        elif e4m3:
            self.out = kvq.paged_decode_attn_e4m3(self.q, self.kc, self.vc, self.bt, self.cl, self.ks,
                                                  self.vs, ws, None, ti_d, tl_d, w.num_splits,
                                                  err_flag=err, split_pages=w.split_pages,
                                                  bitcast_decode=bitcast, longest_first=longest_first,
                                                  fp8_qk=fp8_qk)
        else:
            self.out = kvq.paged_decode_attn_fp16(self.q, self.kc, self.vc, self.bt, self.cl, ws, None,
                                                  ti_d, tl_d, w.num_splits, err_flag=err,
                                                  split_pages=w.split_pages, longest_first=longest_first)
        torch.cuda.synchronize()
        assert err.item() == 0, f"device error bits {err.item()}"

    def oracle_scales(self):
        if not self.e4m3:
            return 1.0, 1.0
        ks = oracle.calibrate_scale(self.kcal.cpu().numpy())
        vs = oracle.calibrate_scale(self.vcal.cpu().numpy())
        assert (ks, vs) == (self.ks, self.vs), "GPU calibration differs from the oracle"
        return ks, vs

    def submit(self, ex, b, h, scales):
        w = self.w
        g = h // w.group
        L = int(self.lay.lens[b])
        ks, vs = scales
        k_seq = self.k[self.offs[b]:self.offs[b] + L, g].cpu().numpy()
        v_seq = self.v[self.offs[b]:self.offs[b] + L, g].cpu().numpy()
        q_rows = self.q[b, :, h, :].cpu().numpy()
        ti, tl = self.topk_np
        lst = None if ti is None or tl[b] == 0 else ti[b, g, : tl[b]]
        return ex.submit(P.oracle_unit, q_rows, k_seq, v_seq, L, ks, vs, self.e4m3, lst)

    def gpu_pool_rows(self, b, g):
        """E4M3 K and V bytes the GPU stored for sequence b, kv head g, positions 0..L-1."""
        L = int(self.lay.lens[b])
        pos = torch.arange(L, device=DEV)
        pages = self.bt[b, pos // 4].long()
        return self.kc[pages, g, pos % 4].cpu().numpy(), self.vc[pages, g, pos % 4].cpu().numpy()


def _check(layer_obj, ex, units, tag):
    scales = layer_obj.oracle_scales()
    futs = [(b, h, layer_obj.submit(ex, b, h, scales)) for b, h in units]
    got_all = layer_obj.out.float().cpu().numpy()
    bad = []
    for b, h, f in futs:
        ref, flags, pool_k, pool_v = f.result()
        assert flags == 0
        got = got_all[b, :, h, :]
        ok = P.tolerance_ok(got, ref)
        if not ok.all():
            bad.append((b, h, float(np.abs(got - ref).max())))
        if layer_obj.e4m3 and h % layer_obj.w.group == 0:
            gk, gv = layer_obj.gpu_pool_rows(b, h // layer_obj.w.group)
            assert np.array_equal(gk, pool_k), \
                f"{tag}: K pool bytes differ for sequence {b}, kv head {h // layer_obj.w.group}"
            assert np.array_equal(gv, pool_v), \
                f"{tag}: V pool bytes differ for sequence {b}, kv head {h // layer_obj.w.group}"
    assert not bad, f"{tag}: {len(bad)} units outside tolerance, e.g. {bad[:4]}"


def _scratch_dir(need_bytes):
    """A folder for the memory-mapped hand-over to the oracle workers: shared
    memory when it has room, else the temporary directory."""
    for base in ("/dev/shm", tempfile.gettempdir()):
        try:
            if os.path.isdir(base) and shutil.disk_usage(base).free > 1.25 * need_bytes:
                return tempfile.mkdtemp(prefix="kvq_pools_", dir=base)
        except OSError:
            continue
    return tempfile.mkdtemp(prefix="kvq_pools_")


def _check_pools(layer_obj, ex, tag, shards_per_worker=4):
    """Every byte of the layer's K and V pools against the oracle's fill of
    sentinel pools with every token the layer appended (the cached history,
    this step's tokens and, for the mixed batch, the prefill chunk), sharded
    over the process pool by page range."""
    L = layer_obj
    w, lay = L.w, L.lay
    lens = lay.lens.astype(np.int64)
    seq = np.repeat(np.arange(w.batch), lens)
    pos = np.arange(int(lens.sum())) - np.repeat(L.offs, lens)
    slots = inputs.slot_mapping(lay.block_tables, seq, pos)          # token row r of L.k -> its slot
    parts = [(L.k, L.v, slots)]
    if L.prefill is not None:
        parts.append((L.prefill[0], L.prefill[1], inputs.prefill_slots(lay)[: w.prefill_chunk]))
    T = sum(int(p[2].size) for p in parts)
    row_bytes = w.num_kv_heads * w.head_dim * 2
    pool_bytes = L.kc.numel() * L.kc.element_size()
    folder = _scratch_dir(2 * T * row_bytes + 2 * pool_bytes + 12 * T)
    try:
        fk = np.lib.format.open_memmap(os.path.join(folder, "k.npy"), "w+", np.float16,
                                       (T, w.num_kv_heads, w.head_dim))
        fv = np.lib.format.open_memmap(os.path.join(folder, "v.npy"), "w+", np.float16,
                                       (T, w.num_kv_heads, w.head_dim))
        all_slots = np.concatenate([p[2] for p in parts]).astype(np.int32)
        t0 = 0
        for k, v, sl in parts:
            n = int(sl.size)
            fk[t0:t0 + n] = k[:n].cpu().numpy()
            fv[t0:t0 + n] = v[:n].cpu().numpy()
            t0 += n
        fk.flush()
        fv.flush()
        del fk, fv
        np.save(os.path.join(folder, "slots.npy"), all_slots)
        pages = all_slots.astype(np.int64) // 4
        order = np.argsort(pages, kind="stable")
        np.save(os.path.join(folder, "order.npy"), order)
        np.save(os.path.join(folder, "pool_k.npy"), L.kc.cpu().numpy())
        np.save(os.path.join(folder, "pool_v.npy"), L.vc.cpu().numpy())
        Ptot = lay.num_pages
        n = max(1, min(Ptot, shards_per_worker * WORKERS))
        p_edges = np.linspace(0, Ptot, n + 1).astype(np.int64)
        i_edges = np.searchsorted(pages[order], p_edges)
        ks, vs = L.oracle_scales()
        futs = [ex.submit(P.oracle_pool_shard, folder, int(p_edges[j]), int(p_edges[j + 1]),
                          int(i_edges[j]), int(i_edges[j + 1]), ks, vs, L.e4m3) for j in range(n)]
        bad = [r for r in (f.result() for f in futs) if r[1] or r[2]]
    finally:
        shutil.rmtree(folder, ignore_errors=True)
    assert not bad, (f"{tag}: pools differ from the oracle's in {len(bad)} of {n} page shards, e.g. "
                     f"(first page, K bytes, V bytes) {[(r[3], r[1], r[2]) for r in bad[:4]]}")


def _sample(rng, w, n):
    b = rng.integers(0, w.batch, n)
    h = rng.integers(0, w.num_q_heads, n)
    h[: n // 2] -= h[: n // 2] % w.group      # half of them are the group's first head (pool check)
    return list(zip(b.tolist(), h.tolist()))


def test_decode_all_units(pool):
    """batch 32 x 4096, split-K 4: every (sequence, query head) checked."""
    w = inputs.get("decode")
    lay = inputs.page_layout(w)
    L = Layer(w, 0, lay)
    assert L.S == 4
    units = [(b, h) for b in range(w.batch) for h in range(w.num_q_heads)]
    _check(L, pool, units, "decode e4m3")
    _check_pools(L, pool, "decode e4m3")
    # the bitcast decoder in the same launch configuration: bit-identical output
    Lb = Layer(w, 0, lay, bitcast=True)
    assert torch.equal(Lb.out.view(torch.int16), L.out.view(torch.int16))
    del Lb
    _same_as_fused(L, w, lay)


def _same_as_fused(L, w, lay, e4m3=True):
    """The fused step call (the benchmark's step) at full size: whole pools and
    outputs bit-identical to those of the append call and the attention call,
    which the oracle has checked."""
    Lf = Layer(w, L.layer, lay, e4m3=e4m3, fused=True)
    assert torch.equal(Lf.kc.view(torch.uint8), L.kc.view(torch.uint8)), "fused step: K pool differs"
    assert torch.equal(Lf.vc.view(torch.uint8), L.vc.view(torch.uint8)), "fused step: V pool differs"
    assert torch.equal(Lf.out.view(torch.int16), L.out.view(torch.int16)), "fused step: output differs"
    del Lf
    torch.cuda.empty_cache()


def test_decode_fp16_arm(pool):
    w = inputs.get("decode")
    lay = inputs.page_layout(w)
    L = Layer(w, 0, lay, e4m3=False)
    _check(L, pool, _sample(np.random.default_rng(1), w, 96), "decode fp16")
    _check_pools(L, pool, "decode fp16")
    _same_as_fused(L, w, lay, e4m3=False)


def test_decode_32k(pool):
    w = inputs.get("decode32k")
    lay = inputs.page_layout(w)
    L = Layer(w, 0, lay)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert L.S == min(2 * 4 * sms // (w.batch * w.num_kv_heads), 8192 // 256)   # the library's choice
    _check(L, pool, _sample(np.random.default_rng(2), w, 48), "decode32k")
    _check_pools(L, pool, "decode32k")
    _same_as_fused(L, w, lay)


def test_long_context(pool):
    """batch 4 x 262,144 tokens, split-K 64 with the FP32 workspace and combine."""
    w = inputs.get("long")
    lay = inputs.page_layout(w)
    L = Layer(w, 0, lay)
    assert L.S == 64
    _check(L, pool, _sample(np.random.default_rng(3), w, 12), "long")
    _check_pools(L, pool, "long")
    _same_as_fused(L, w, lay)


def test_verify_24_layers(pool):
    """MTP3 verify: 24 layers, each with its own calibrated scales; >= 256 sampled units."""
    w = inputs.get("verify")
    lay = inputs.page_layout(w)
    rng = np.random.default_rng(4)
    seen = set()
    for layer in range(w.layers):
        L = Layer(w, layer, lay)
        seen.add((L.ks, L.vs))
        _check(L, pool, _sample(rng, w, 11), f"verify layer {layer}")
        if layer in (0, w.layers - 1):
            _check_pools(L, pool, f"verify layer {layer}")
        if layer == 0:
            _same_as_fused(L, w, lay)   # the tcgen05 shapes: the append by block table, then the attention
        del L
        torch.cuda.empty_cache()
    assert len(seen) == w.layers          # per-layer scales really differ


def test_verify_fp16_arm(pool):
    """The fp16-KV arm of MTP3 verify at full size (the comparison arm of the
    bench's E4M3-vs-fp16 report): one layer on the tcgen05 kernel's fp16
    instance, sampled units against the oracle, whole pools, and the fused
    step call bit-identical."""
    w = inputs.get("verify")
    lay = inputs.page_layout(w)
    L = Layer(w, 0, lay, e4m3=False)
    _check(L, pool, _sample(np.random.default_rng(6), w, 24), "verify fp16")
    _check_pools(L, pool, "verify fp16")
    _same_as_fused(L, w, lay, e4m3=False)


def test_mixed_24_layers(pool):
    """Mixed batch: 8192-token prefill chunk appended per layer + 48 decodes,
    half over a top-2048 list; >= 256 sampled units, prefill bytes checked."""
    w = inputs.get("mixed")
    lay = inputs.page_layout(w)
    ti, tl = inputs.topk_lists(w, lay.lens)
    assert (tl > 0).sum() == 24
    rng = np.random.default_rng(5)
    pre_slots = inputs.prefill_slots(lay)[: w.prefill_chunk]
    for layer in range(w.layers):
        L = Layer(w, layer, lay)
        units = _sample(rng, w, 11)
        _check(L, pool, units, f"mixed layer {layer}")
        if layer in (0, w.layers - 1):
            _check_pools(L, pool, f"mixed layer {layer}")   # includes the prefill chunk
        # the prefill chunk's quantised bytes, one kv head per layer
        g = layer % w.num_kv_heads
        ks, _ = L.oracle_scales()
        pk = L.prefill[0][:, g].cpu().numpy()
        want = oracle.quantize(pk, ks)
        sl = torch.from_numpy(pre_slots.astype(np.int64)).to(DEV)
        got = L.kc[sl // 4, g, sl % 4].cpu().numpy()
        assert np.array_equal(got, want), f"prefill bytes differ, layer {layer}"
        del L
        torch.cuda.empty_cache()


def test_mixed_and_long_fp16_arms(pool):
    """The fp16-KV arms of the mixed batch (top-k lists, the prefill chunk in
    the same append) and of the long context at full size: one layer each,
    sampled units against the oracle and whole pools."""
    rng = np.random.default_rng(7)
    for name, n in (("mixed", 16), ("long", 8)):
        w = inputs.get(name)
        L = Layer(w, 0, inputs.page_layout(w), e4m3=False)
        _check(L, pool, _sample(rng, w, n), f"{name} fp16")
        _check_pools(L, pool, f"{name} fp16")
        del L
        torch.cuda.empty_cache()


def test_verify_fp8_scores(pool):
    """The FP8 score variant at the verify workload's full size: sampled
    (sequence, kv head) groups against the oracle's reading, each group's
    G x q_len query rows quantised together as the kernel's CTA does."""
    w = inputs.get("verify")
    L = Layer(w, 0, inputs.page_layout(w), fp8_qk=True)
    ks, vs = L.oracle_scales()
    rng = np.random.default_rng(6)
    G = w.group
    groups = list(zip(rng.integers(0, w.batch, 12).tolist(), rng.integers(0, w.num_kv_heads, 12).tolist()))
    futs = []
    for b, g in groups:
        n = int(L.lay.lens[b])
        q_group = L.q[b, :, g * G:(g + 1) * G, :].cpu().numpy()
        k_seq = L.k[L.offs[b]:L.offs[b] + n, g].cpu().numpy()
        v_seq = L.v[L.offs[b]:L.offs[b] + n, g].cpu().numpy()
        futs.append((b, g, pool.submit(P.oracle_group_fp8, q_group, k_seq, v_seq, n, ks, vs)))
    got_all = L.out.float().cpu().numpy()
    bad = []
    for b, g, f in futs:
        ref, flags = f.result()
        assert flags == 0
        got = got_all[b, :, g * G:(g + 1) * G, :]
        ok = P.tolerance_ok(got, ref)
        if not ok.all():
            bad.append((b, g, float(np.abs(got - ref).max())))
    assert not bad, f"verify fp8 scores: {len(bad)} groups outside tolerance, e.g. {bad[:4]}"
