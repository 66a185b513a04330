"""Test helpers: host-side problems built from the seeded generators.

`host_problem` draws one layer of a workload on the CPU and lays it out as
numpy arrays.  `oracle_pools` fills page pools with the oracle's quantiser;
GPU tests fill their own pools with the CUDA library from the same fp16
inputs, so no expected value ever comes from the CUDA path.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

import oracle
from fp8_paged_kv_e4m3_gb300 import inputs

SENTINEL = 0xCC


@dataclasses.dataclass
class HostProblem:
    w: inputs.Workload
    layout: inputs.PageLayout
    k_tok: np.ndarray          # fp16 [total_tokens, Hkv, D], sequences back to back
    v_tok: np.ndarray
    offsets: np.ndarray        # int64 [B] start of each sequence in k_tok / v_tok
    q: np.ndarray              # fp16 [B, q_len, Hq, D]
    k_calib: np.ndarray        # fp16 calibration draws
    v_calib: np.ndarray
    hist_slots: np.ndarray     # int32 slots of the cached history tokens
    hist_rows: np.ndarray      # int64 rows of k_tok / v_tok for those tokens
    step_slots: np.ndarray     # int32 slots of this step's q_len tokens per sequence
    step_rows: np.ndarray
    topk_idx: Optional[np.ndarray]
    topk_lens: Optional[np.ndarray]

    @property
    def P(self):
        return self.layout.num_pages


def host_problem(name_or_w, layer: int = 0, **overrides) -> HostProblem:
    w = inputs.get(name_or_w, **overrides) if isinstance(name_or_w, str) else name_or_w
    layout = inputs.page_layout(w)
    lens = layout.lens.astype(np.int64)
    total = int(lens.sum())
    offsets = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int64)
    k_tok = inputs.kv_tokens(w, layer, total, "k").numpy()
    v_tok = inputs.kv_tokens(w, layer, total, "v").numpy()
    q = inputs.queries(w, layer).numpy()
    k_cal = inputs.calibration_draw(w, layer, "k").numpy()
    v_cal = inputs.calibration_draw(w, layer, "v").numpy()
    hs, hp = inputs.history_tokens(w, layout)
    ss, sp = inputs.step_tokens(w, layout)
    ti, tl = inputs.topk_lists(w, layout.lens)
    return HostProblem(
        w, layout, k_tok, v_tok, offsets, q, k_cal, v_cal,
        inputs.slot_mapping(layout.block_tables, hs, hp), offsets[hs] + hp,
        inputs.slot_mapping(layout.block_tables, ss, sp), offsets[ss] + sp,
        ti, tl)


def empty_pools(pr: HostProblem, e4m3: bool = True):
    w = pr.w
    shape = (pr.P, w.num_kv_heads, inputs.PAGE, w.head_dim)
    if e4m3:
        return (np.full(shape, SENTINEL, np.uint8), np.full(shape, SENTINEL, np.uint8))
    fill = np.uint16(SENTINEL * 0x101)
    return (np.full(shape, fill, np.uint16).view(np.float16),
            np.full(shape, fill, np.uint16).view(np.float16))


def oracle_scales(pr: HostProblem):
    return oracle.calibrate_scale(pr.k_calib), oracle.calibrate_scale(pr.v_calib)


def oracle_pools(pr: HostProblem, e4m3: bool = True, scales=None):
    """Pools filled by the oracle: history tokens, then this step's tokens."""
    kc, vc = empty_pools(pr, e4m3)
    if e4m3:
        ks, vs = scales if scales is not None else oracle_scales(pr)
        for slots, rows in ((pr.hist_slots, pr.hist_rows), (pr.step_slots, pr.step_rows)):
            if slots.size:
                oracle.append_e4m3(pr.k_tok[rows], pr.v_tok[rows], slots, kc, vc, ks, vs)
        return kc, vc, ks, vs
    for slots, rows in ((pr.hist_slots, pr.hist_rows), (pr.step_slots, pr.step_rows)):
        if slots.size:
            oracle.append_fp16(pr.k_tok[rows], pr.v_tok[rows], slots, kc, vc)
    return kc, vc, 1.0, 1.0


def tolerance_ok(got, ref, atol=2e-3, rtol=1e-2):
    """Element-wise |got - ref| <= atol + rtol * |ref| (the parity gate)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return np.abs(got - ref) <= atol + rtol * np.abs(ref)


def torch_reference(q, k_pool_vals, v_pool_vals, block_tables, lens, q_len, topk_idx=None,
                    topk_lens=None, sm_scale=None):
    """Independent binary64 reference built from library pieces: gather the
    dequantised pool values by numpy fancy indexing, mask explicitly, and
    call torch.softmax.  k_pool_vals / v_pool_vals are float64 [P][Hkv][4][D]."""
    B, ql, Hq, D = q.shape
    Hkv = k_pool_vals.shape[1]
    G = Hq // Hkv
    scale = 1.0 / np.sqrt(D) if sm_scale is None else sm_scale
    out = np.zeros((B, ql, Hq, D))
    for b in range(B):
        L = int(lens[b])
        pos = np.arange(L)
        pages = block_tables[b, pos // 4]
        Kb = k_pool_vals[pages, :, pos % 4, :]      # [L, Hkv, D]
        Vb = v_pool_vals[pages, :, pos % 4, :]
        for h in range(Hq):
            g = h // G
            qh = torch.from_numpy(q[b, :, h, :].astype(np.float64))            # [ql, D]
            s = qh @ torch.from_numpy(Kb[:, g, :]).T * scale                   # [ql, L]
            allowed = torch.zeros((ql, L), dtype=torch.bool)
            for i in range(ql):
                lim = L - ql + i
                if topk_idx is not None and topk_lens[b] > 0:
                    sel = topk_idx[b, g, :topk_lens[b]]
                    sel = sel[sel <= lim]
                    allowed[i, torch.from_numpy(sel.astype(np.int64))] = True
                else:
                    allowed[i, : lim + 1] = True
            s = s.masked_fill(~allowed, float("-inf"))
            p = torch.softmax(s, dim=-1)
            out[b, :, h, :] = (p @ torch.from_numpy(Vb[:, g, :])).numpy()
    return out


def torch_dequant(pool_u8, scale):
    return torch.from_numpy(pool_u8).view(torch.float8_e4m3fn).double().numpy() * float(scale)


def oracle_unit(q_rows, k_seq, v_seq, L, ks, vs, e4m3=True, topk_list=None):
    """Oracle attention of one (sequence, query head) unit from its own data.

    q_rows fp16 [q_len, D]; k_seq / v_seq fp16 [L, D] (the sequence's tokens of
    the head's kv group, positions 0..L-1); topk_list int32 [n] or None.
    Builds a one-sequence, one-head problem with an identity block table and
    returns (out [q_len, D] float64, flags, pool_k bytes [L, D], pool_v bytes
    [L, D]) -- the pool bytes for the E4M3 arm, None for fp16."""
    q_len, D = q_rows.shape
    pages = (L + 3) // 4
    bt = np.arange(pages, dtype=np.int32)[None, :]
    slots = np.arange(L, dtype=np.int32)
    if e4m3:
        kc = np.full((pages, 1, 4, D), SENTINEL, np.uint8)
        vc = kc.copy()
        oracle.append_e4m3(k_seq[:, None, :], v_seq[:, None, :], slots, kc, vc, ks, vs)
    else:
        kc = np.zeros((pages, 1, 4, D), np.float16)
        vc = kc.copy()
        oracle.append_fp16(k_seq[:, None, :], v_seq[:, None, :], slots, kc, vc)
        ks = vs = 1.0
    ti = tl = None
    if topk_list is not None:
        ti = np.ascontiguousarray(topk_list, np.int32)[None, None, :]
        tl = np.array([len(topk_list)], np.int32)
    out, flags = oracle.attention(np.ascontiguousarray(q_rows)[None, :, None, :], kc, vc, bt,
                                  np.array([L], np.int32), ks, vs, ti, tl)
    pool_k = kc.reshape(pages * 4, D)[:L] if e4m3 else None
    pool_v = vc.reshape(pages * 4, D)[:L] if e4m3 else None
    return out[0, :, 0, :], flags, pool_k, pool_v


def oracle_pool_shard(folder, p0, p1, i0, i1, ks, vs, e4m3):
    """The oracle's fill of pool pages [p0, p1), compared with the GPU's.

    `folder` holds (as .npy files) every token the layer appended -- k, v
    fp16 [T][Hkv][D] and their slots int32 [T] -- plus `order`, the token
    indices sorted by page, whose entries [i0, i1) are the tokens of pages
    [p0, p1), and the GPU's pools pool_k, pool_v [P][Hkv][4][D].  Starting
    from sentinel pools, the oracle appends those tokens (their slots
    re-based to page p0); every byte of the shard, including the slots no
    token owns, must equal the GPU's.  Returns (p0, differing K bytes,
    differing V bytes, first differing page or -1)."""
    import os
    ld = lambda name: np.load(os.path.join(folder, name + ".npy"), mmap_mode="r")
    idx = np.sort(np.asarray(ld("order")[i0:i1]))
    k = np.ascontiguousarray(ld("k")[idx])
    v = np.ascontiguousarray(ld("v")[idx])
    slots = (np.asarray(ld("slots")[idx]).astype(np.int64) - 4 * p0).astype(np.int32)
    gk = np.asarray(ld("pool_k")[p0:p1])
    gv = np.asarray(ld("pool_v")[p0:p1])
    shape = gk.shape
    if e4m3:
        kc = np.full(shape, SENTINEL, np.uint8)
        vc = np.full(shape, SENTINEL, np.uint8)
        if idx.size:
            oracle.append_e4m3(k, v, slots, kc, vc, ks, vs)
        dk, dv = kc != gk, vc != gv
    else:
        fill = np.uint16(SENTINEL * 0x101)
        kc = np.full(shape, fill, np.uint16).view(np.float16)
        vc = np.full(shape, fill, np.uint16).view(np.float16)
        if idx.size:
            oracle.append_fp16(k, v, slots, kc, vc)
        dk, dv = kc.view(np.uint16) != gk.view(np.uint16), vc.view(np.uint16) != gv.view(np.uint16)
    bad_pages = np.flatnonzero(dk.reshape(shape[0], -1).any(1) | dv.reshape(shape[0], -1).any(1))
    return p0, int(dk.sum()), int(dv.sum()), int(p0 + bad_pages[0]) if bad_pages.size else -1


def oracle_group_fp8(q_group, k_seq, v_seq, L, ks, vs):
    """Oracle attention of one (sequence, kv head) group under the FP8 score
    reading: q_group fp16 [q_len, G, D] (all the query rows that share the kv
    head, so that the group's query scale is the one the kernel takes),
    k_seq / v_seq fp16 [L, D].  Returns out [q_len, G, D] float64 and flags."""
    q_len, G, D = q_group.shape
    pages = (L + 3) // 4
    bt = np.arange(pages, dtype=np.int32)[None, :]
    slots = np.arange(L, dtype=np.int32)
    kc = np.full((pages, 1, 4, D), SENTINEL, np.uint8)
    vc = kc.copy()
    oracle.append_e4m3(k_seq[:, None, :], v_seq[:, None, :], slots, kc, vc, ks, vs)
    out, flags = oracle.attention(np.ascontiguousarray(q_group)[None], kc, vc, bt, np.array([L], np.int32), ks, vs,
                                  fp8_q=True)
    return out[0], flags
