"""Seeded synthetic inputs for the paged-KV decode / verify workloads.

This module only draws numbers and lays out indices (lengths, block tables,
slot mappings, top-k lists, fp16 Q/K/V and calibration draws).  It holds none
of the method's arithmetic -- no quantisation, no scale computation, no
attention -- so that the CUDA path and the CPU oracle can both consume the
same input bytes without sharing any of the computation under test.

Workloads (the pages measure on a private serving deployment; these synthetic
tensors stand in for the K/V that such traffic would produce):

  tiny      1 layer, batch 2, contexts 37 and 100, 8 q heads / 2 kv heads,
            head_dim 64, N(0,1) with 2 outlier channels x20, q_len 1 or 4
  decode    batch 32 x 4096 context, 32 q / 4 kv heads, head_dim 128, q_len 1,
            4 splits
  decode32k as decode at 32768 context, the library's split count
  verify    24 layers, batch 64, q_len 4 (1 + 3 drafts), contexts
            log-uniform in [1024, 32768], N(0,1) with 4 Student-t(3) channels
            per kv head
  long      batch 4 x 262144 context, 64 splits
  mixed     24 layers; an 8192-token prefill chunk appended plus 48 decode
            sequences with contexts uniform in [8192, 32768]; half of them
            attend over a sorted top-2048 token list per (sequence, kv head)
  prefill   the mixed batch's 8192-token chunk attended: one new sequence,
            q_len 8192 over its own 8192 tokens (causal), 32 q / 4 kv heads

Seeding: every draw uses its own torch.Generator seeded from
(workload id, purpose, layer), so any layer can be regenerated alone.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

PAGE = 4  # tokens per page

# seed purposes
_DATA, _CALIB, _TABLE, _LENS, _TOPK, _CHANNELS, _QUERY = range(7)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    wid: int
    layers: int
    batch: int            # decode sequences attended this step
    q_len: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    num_splits: int       # 0 = let the library choose
    lens: str             # "fixed:<L>", "list:<a,b,..>", "loguniform:<lo>:<hi>", "uniform:<lo>:<hi>"
    outlier_channels: int = 0     # channels scaled x20 (same for Q, K, V, all heads)
    heavy_channels: int = 0       # channels per kv head drawn from Student-t(3)
    calib_tokens: int = 4096
    topk: int = 0                 # list length for the top-k sequences
    topk_fraction: float = 0.0    # share of sequences that use a top-k list
    prefill_chunk: int = 0        # extra tokens appended for one new sequence
    spare_pages: float = 0.125    # pool slack beyond the pages in use
    seed: int = 0
    split_pages: int = 0          # 0 = equal split division; > 0 = pages per split

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 2, 1, 8, 2, 64, 2, "list:37,100",
                     outlier_channels=2, calib_tokens=128),
    "tiny_verify": Workload("tiny_verify", 1, 1, 2, 4, 8, 2, 64, 2, "list:37,100",
                            outlier_channels=2, calib_tokens=128),
    "decode": Workload("decode", 2, 1, 32, 1, 32, 4, 128, 4, "fixed:4096"),
    "decode32k": Workload("decode32k", 6, 1, 32, 1, 32, 4, 128, 0, "fixed:32768"),
    "verify": Workload("verify", 3, 24, 64, 4, 32, 4, 128, 0, "loguniform:1024:32768",
                       heavy_channels=4),
    "long": Workload("long", 4, 1, 4, 1, 32, 4, 128, 64, "fixed:262144"),
    "mixed": Workload("mixed", 5, 24, 48, 1, 32, 4, 128, 0, "uniform:8192:32768",
                      topk=2048, topk_fraction=0.5, prefill_chunk=8192),
    "prefill": Workload("prefill", 7, 24, 1, 8192, 32, 4, 128, 0, "fixed:8192"),
}


def get(name: str, **overrides) -> Workload:
    w = WORKLOADS[name]
    return dataclasses.replace(w, **overrides) if overrides else w


def _gen(w: Workload, purpose: int, layer: int = 0, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(((w.seed * 97 + w.wid) * 1_000_003 + purpose * 10_007 + layer) & 0x7FFF_FFFF)
    return g


def _np_rng(w: Workload, purpose: int, layer: int = 0) -> np.random.Generator:
    return np.random.default_rng([w.seed, w.wid, purpose, layer])


# ---------------------------------------------------------------------------
# structure: lengths, block tables, slot mappings, top-k lists

def context_lens(w: Workload) -> np.ndarray:
    """int32 [B]: cached tokens per sequence, including this step's q_len."""
    kind, *rest = w.lens.split(":")
    if kind == "fixed":
        return np.full(w.batch, int(rest[0]), dtype=np.int32)
    if kind == "list":
        v = np.array([int(x) for x in rest[0].split(",")], dtype=np.int32)
        assert v.size == w.batch
        return v
    rng = _np_rng(w, _LENS)
    lo, hi = int(rest[0]), int(rest[1])
    if kind == "loguniform":
        u = rng.uniform(math.log(lo), math.log(hi), size=w.batch)
        return np.clip(np.floor(np.exp(u)), lo, hi).astype(np.int32)
    if kind == "uniform":
        return rng.integers(lo, hi + 1, size=w.batch).astype(np.int32)
    raise ValueError(w.lens)


@dataclasses.dataclass
class PageLayout:
    lens: np.ndarray           # int32 [B]
    block_tables: np.ndarray   # int32 [B][max_pages], -1 where unused
    num_pages: int             # pool size P
    prefill_pages: np.ndarray  # int32 [ceil(prefill/4)] pages of the new prefill sequence


def page_layout(w: Workload, lens: Optional[np.ndarray] = None) -> PageLayout:
    """Each sequence takes the next slice of one seeded permutation of the pool."""
    if lens is None:
        lens = context_lens(w)
    need = (lens.astype(np.int64) + PAGE - 1) // PAGE
    pre = (w.prefill_chunk + PAGE - 1) // PAGE
    used = int(need.sum()) + pre
    P = used + int(math.ceil(used * w.spare_pages))
    perm = torch.randperm(P, generator=_gen(w, _TABLE)).numpy().astype(np.int32)
    max_pages = int(need.max()) if need.size else 0
    bt = np.full((w.batch, max(max_pages, 1)), -1, dtype=np.int32)
    off = 0
    for b in range(w.batch):
        n = int(need[b])
        bt[b, :n] = perm[off:off + n]
        off += n
    return PageLayout(lens.astype(np.int32), bt, P, perm[off:off + pre].copy())


def slot_mapping(block_tables: np.ndarray, seq_ids: np.ndarray, positions: np.ndarray) -> np.ndarray:
    """int32 slot = block_table[b][pos // 4] * 4 + pos % 4 for each (b, pos)."""
    pages = block_tables[seq_ids, positions // PAGE].astype(np.int64)
    return (pages * PAGE + positions % PAGE).astype(np.int32)


def step_tokens(w: Workload, layout: PageLayout):
    """(seq_ids, positions) of the q_len tokens each decode sequence appends this step."""
    L = layout.lens.astype(np.int64)
    seq = np.repeat(np.arange(w.batch), w.q_len)
    pos = (L[seq] - w.q_len + np.tile(np.arange(w.q_len), w.batch))
    return seq.astype(np.int64), pos.astype(np.int64)


def history_tokens(w: Workload, layout: PageLayout):
    """(seq_ids, positions) of the tokens already cached before this step."""
    L = layout.lens.astype(np.int64) - w.q_len
    seq = np.repeat(np.arange(w.batch), L)
    starts = np.cumsum(np.concatenate([[0], L[:-1]]))
    pos = np.arange(int(L.sum())) - np.repeat(starts, L)
    return seq.astype(np.int64), pos.astype(np.int64)


def prefill_slots(layout: PageLayout) -> np.ndarray:
    """Slots of the new sequence's prefill chunk (positions 0 .. chunk-1)."""
    n = layout.prefill_pages.size * PAGE
    pos = np.arange(n, dtype=np.int64)
    return (layout.prefill_pages[pos // PAGE].astype(np.int64) * PAGE + pos % PAGE).astype(np.int32)


def topk_lists(w: Workload, lens: np.ndarray):
    """(topk_idx int32 [B][Hkv][K], topk_lens int32 [B]) or (None, None).

    A seeded share of the sequences gets, per kv head, K distinct positions
    drawn uniformly from [0, L_b) and sorted ascending; the others get length 0
    (dense attention)."""
    if w.topk <= 0:
        return None, None
    rng = _np_rng(w, _TOPK)
    B, H, K = w.batch, w.num_kv_heads, w.topk
    chosen = rng.permutation(B)[: int(round(B * w.topk_fraction))]
    idx = np.zeros((B, H, K), dtype=np.int32)
    tl = np.zeros(B, dtype=np.int32)
    for b in sorted(chosen.tolist()):
        L = int(lens[b])
        k = min(K, L)
        for g in range(H):
            idx[b, g, :k] = np.sort(rng.choice(L, size=k, replace=False))
        tl[b] = k
    return idx, tl


# ---------------------------------------------------------------------------
# values

def _channels(w: Workload, layer: int, count: int, per_head: bool):
    rng = _np_rng(w, _CHANNELS, layer)
    if per_head:
        return [np.sort(rng.choice(w.head_dim, size=count, replace=False)) for _ in range(w.num_kv_heads)]
    return np.sort(rng.choice(w.head_dim, size=count, replace=False))


def _draw_kv(w: Workload, n_tokens: int, layer: int, purpose: int, device) -> torch.Tensor:
    """fp16 [n_tokens, Hkv, D] with the workload's value distribution."""
    g = _gen(w, purpose, layer, device)
    x = torch.randn((n_tokens, w.num_kv_heads, w.head_dim), generator=g, device=device,
                    dtype=torch.float32)
    if w.outlier_channels:
        ch = torch.as_tensor(_channels(w, 0, w.outlier_channels, False), device=device)
        x[:, :, ch] *= 20.0
    if w.heavy_channels:
        for h, ch in enumerate(_channels(w, layer, w.heavy_channels, True)):
            ch = torch.as_tensor(ch, device=device)
            z = torch.randn((n_tokens, ch.numel()), generator=g, device=device)
            c = torch.randn((n_tokens, ch.numel(), 3), generator=g, device=device).pow(2).sum(-1)
            x[:, h, ch] = z / torch.sqrt(c / 3.0)
    return x.to(torch.float16)


def kv_tokens(w: Workload, layer: int, n_tokens: int, which: str, device="cpu") -> torch.Tensor:
    """K or V for n_tokens cached tokens of one layer, fp16 [n_tokens, Hkv, D]."""
    purpose = _DATA * 2 + (0 if which == "k" else 1) + 100
    return _draw_kv(w, n_tokens, layer, purpose, device)


def prefill_tokens(w: Workload, layer: int, which: str, device="cpu") -> torch.Tensor:
    """K or V of the new sequence's prefill chunk, fp16 [prefill_chunk, Hkv, D]."""
    purpose = _DATA * 2 + (0 if which == "k" else 1) + 300
    return _draw_kv(w, w.prefill_chunk, layer, purpose, device)


def calibration_draw(w: Workload, layer: int, which: str, device="cpu") -> torch.Tensor:
    """A separate draw of the same distribution, used only to calibrate the scale."""
    purpose = _CALIB * 2 + (0 if which == "k" else 1) + 200
    return _draw_kv(w, w.calib_tokens, layer, purpose, device)


def queries(w: Workload, layer: int, device="cpu") -> torch.Tensor:
    """fp16 [B, q_len, Hq, D]."""
    g = _gen(w, _QUERY, layer, device)
    x = torch.randn((w.batch, w.q_len, w.num_q_heads, w.head_dim), generator=g, device=device,
                    dtype=torch.float32)
    if w.outlier_channels:
        ch = torch.as_tensor(_channels(w, 0, w.outlier_channels, False), device=device)
        x[..., ch] *= 20.0
    return x.to(torch.float16)
