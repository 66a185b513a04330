"""Decode context parallelism (DCP) over the paged E4M3 cache.

PR "[Model][SM70] Calibrated E4M3 KV cache for Qwen4Exp QSA with MTP",
sections Status and history and Validation: with DCP2 the KV tokens of
every sequence are spread over two ranks, which raises the KV capacity of
the deployment.  The attention of such a sequence is split-K over ranks:

  1. every rank holds a contiguous range of each sequence's logical pages
     (`shard_pages`) and computes the split-K partials (o, m, l) of its own
     range with the library's partial call;
  2. the partials are all-gathered over the process group
     (`gather_partials`): one exchange step, on the host-visible tensors, no
     cross-GPU copy engine or multicast;
  3. the log-sum-exp combine merges the world x S partials of every row.

The combine is exact up to rounding whatever the partition, so the result is
the single-GPU attention.

MTP verify windows (q_len > 1, causal inside the window, PR "[Model][SM70]
Calibrated E4M3 KV cache for Qwen4Exp QSA with MTP", section Purpose): a
rank below the window sees all of its keys from every window row, the rank
that holds the window a causal prefix of them.  `shard_window_rows` states
this with the calls as they are: the window's q_len rows become q_len
one-row sequences per sequence (the query viewed as [B * q_len][1][Hq][D],
row i of sequence b at b * q_len + i), each with its own local context
length, the count of this rank's positions up to the row's causal limit.
The partials, the exchange and the combine are then those of decode, and
the output comes out in the [B][q_len][Hq][D] order.  Each page is read once
per window row on this route (the single-GPU verify call reads it once).
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np
import torch

from . import kvq

PAGE = kvq.PAGE_SIZE


def shard_pages(block_tables: np.ndarray, context_lens: np.ndarray, world: int, rank: int):
    """Rank `rank`'s share of every sequence: logical pages [r c, min((r + 1) c, n))
    with n = ceil(L / 4) and c = ceil(n / world).

    Returns (local block table int32 [B][c_max] with -1 past a shard's pages,
    local context lengths int32 [B]).  Every sequence must span at least
    `world` pages, so that no rank's share is empty (the attention of an
    empty key set is not a partial the combine can weigh)."""
    bt = np.asarray(block_tables, dtype=np.int32)
    lens = np.asarray(context_lens, dtype=np.int64)
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad world / rank")
    n = (lens + PAGE - 1) // PAGE
    if (n < world).any():
        raise ValueError("every sequence needs at least `world` pages for DCP")
    c = (n + world - 1) // world
    first = rank * c
    last = np.minimum((rank + 1) * c, n)
    if (last <= first).any():
        raise ValueError("a rank would hold no page of some sequence; use fewer ranks")
    width = int(c.max())
    local = np.full((bt.shape[0], width), -1, dtype=np.int32)
    for b in range(bt.shape[0]):
        k = int(last[b] - first[b])
        local[b, :k] = bt[b, first[b]:last[b]]
    local_lens = np.minimum(lens, PAGE * last) - PAGE * first
    return local, local_lens.astype(np.int32)


def shard_window_rows(block_tables: np.ndarray, context_lens: np.ndarray, q_len: int, world: int, rank: int):
    """Rank `rank`'s share of a verify window of q_len rows, as q_len one-row
    sequences per sequence (row i of sequence b at b * q_len + i): each gets
    this rank's local block table of sequence b (`shard_pages`) and, as its
    context length, the number of this rank's positions at or below the row's
    causal limit L - q_len + i.

    Returns (local block table int32 [B * q_len][c_max], local context lengths
    int32 [B * q_len]).  Every rank must hold a key that every row sees, that
    is a first position at or below L - q_len; otherwise a row's share would be
    empty (use fewer ranks)."""
    if q_len < 1:
        raise ValueError("q_len must be at least 1")
    local, local_lens = shard_pages(block_tables, context_lens, world, rank)
    lens = np.asarray(context_lens, dtype=np.int64)
    if (lens < q_len).any():
        raise ValueError("every context must hold its window")
    n = (lens + PAGE - 1) // PAGE
    first_pos = PAGE * rank * ((n + world - 1) // world)      # this rank's first position per sequence
    if (first_pos > lens - q_len).any():
        raise ValueError("a rank would hold no key of some window row; use fewer ranks")
    B = lens.shape[0]
    i = np.tile(np.arange(q_len, dtype=np.int64), B)
    seen = np.repeat(lens - q_len - first_pos, q_len) + i + 1   # this rank's positions up to each row's limit
    rows_lens = np.minimum(np.repeat(local_lens.astype(np.int64), q_len), seen)
    return np.repeat(local, q_len, axis=0), rows_lens.astype(np.int32)


def _global_params(p_local: kvq.AttnParams, world: int) -> kvq.AttnParams:
    S = kvq.num_splits(p_local)
    return kvq.AttnParams(p_local.batch, p_local.q_len, p_local.num_q_heads, p_local.num_kv_heads,
                          p_local.head_dim, world * S, p_local.max_pages_per_seq, 0, p_local.sm_scale,
                          0, 0)


def gather_partials(ws_local, p_local: kvq.AttnParams, world: int, group=None,
                    parts: Optional[Sequence[torch.Tensor]] = None):
    """The exchange: every rank's workspace (o, m, l) gathered into one
    workspace whose split axis lists rank 0's splits, then rank 1's, ...
    (layout of kvq_attn_workspace_bytes with num_splits = world x S).

    With a process group, `ws_local` is this rank's workspace and the
    gather is torch.distributed.all_gather (NCCL on GPUs, gloo on CPUs).
    Without one, `parts` holds the world workspaces already at hand (one
    process computing every rank's share, as the tests do).
    Returns (global workspace, its parameters)."""
    if p_local.q_len != 1:
        raise ValueError("DCP partials have one query row per sequence (verify windows: shard_window_rows)")
    o, m, l = kvq.workspace_views(ws_local if parts is None else parts[0], p_local)
    if parts is None:
        import torch.distributed as dist
        gathered = []
        for t in (o, m, l):
            bufs = [torch.empty_like(t) for _ in range(world)]
            dist.all_gather(bufs, t.contiguous(), group=group)
            gathered.append(bufs)
    else:
        if len(parts) != world:
            raise ValueError("need one workspace per rank")
        views = [kvq.workspace_views(w, p_local) for w in parts]
        gathered = [[v[i] for v in views] for i in range(3)]
    p_g = _global_params(p_local, world)
    n_floats = (kvq.workspace_bytes(p_g) + 3) // 4
    ws_g = torch.empty(n_floats, dtype=torch.float32, device=o.device)
    go, gm, gl = kvq.workspace_views(ws_g, p_g)
    # split axis: rank-major
    go.copy_(torch.cat(gathered[0], dim=3))
    gm.copy_(torch.cat(gathered[1], dim=3))
    gl.copy_(torch.cat(gathered[2], dim=3))
    return ws_g, p_g


def dcp_decode_attn_e4m3(q, k_cache, v_cache, local_block_tables, local_context_lens, k_scale: float,
                         v_scale: float, world: int, group=None, out=None, num_splits: int = 0,
                         err_flag=None):
    """This rank's part of a DCP decode or verify step: the partials of its own
    pages, the all-gather, then the combine.  q is the full fp16
    [B][q_len][Hq][D] query (every rank attends the same rows); the pools hold
    this rank's pages; the local tables and lengths are `shard_pages`' for
    q_len 1, `shard_window_rows`' for a verify window.  Returns the fp16
    output [B][q_len][Hq][D] (the same on every rank)."""
    B, q_len, Hq, D = q.shape
    if q_len > 1 and local_block_tables.shape[0] != B * q_len:
        raise ValueError("a verify window takes the rows of shard_window_rows")
    rows = q.reshape(B * q_len, 1, Hq, D)       # a view: row i of sequence b at b * q_len + i
    p = kvq.attn_params(rows, k_cache.shape[1], local_block_tables.shape[1], num_splits)
    ws = kvq.alloc_workspace(p, q.device)
    kvq.paged_decode_attn_e4m3_partial(rows, k_cache, v_cache, local_block_tables, local_context_lens,
                                       k_scale, v_scale, ws, num_splits=num_splits, err_flag=err_flag)
    ws_g, p_g = gather_partials(ws, p, world, group=group)
    if out is None:
        out = torch.empty_like(q)
    kvq.lse_combine(ws_g, out.view(B * q_len, 1, Hq, D), p_g)
    return out
