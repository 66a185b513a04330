"""GPU-side problem setup for the parity tests: every GPU value is produced by
the CUDA library (calibration, append, attention) from the same seeded fp16
inputs the oracle consumes."""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from fp8_paged_kv_e4m3_gb300 import inputs, kvq
from tests import _problems as P


@dataclasses.dataclass
class DeviceProblem:
    host: P.HostProblem
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_tables: torch.Tensor
    context_lens: torch.Tensor
    topk_idx: torch.Tensor | None
    topk_lens: torch.Tensor | None
    k_scale: float
    v_scale: float
    e4m3: bool
    err: torch.Tensor


def to_dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t if dtype is None else t.to(dtype)


def device_problem(pr: P.HostProblem, e4m3: bool = True, sentinel: int = P.SENTINEL) -> DeviceProblem:
    """Pools pre-filled with `sentinel` (a byte; for fp16 pools the 16-bit
    pattern sentinel * 0x101), then filled by the library's append."""
    dev = torch.device("cuda")
    w = pr.w
    shape = (pr.P, w.num_kv_heads, 4, w.head_dim)
    if e4m3:
        kc = torch.full(shape, sentinel, dtype=torch.uint8, device=dev)
        vc = torch.full(shape, sentinel, dtype=torch.uint8, device=dev)
        ks = kvq.calibrate_scale(to_dev(pr.k_calib))
        vs = kvq.calibrate_scale(to_dev(pr.v_calib))
    else:
        fill = torch.tensor(sentinel * 0x101, dtype=torch.int32).to(torch.int16)
        kc = torch.empty(shape, dtype=torch.float16, device=dev)
        kc.view(torch.int16).fill_(int(fill))
        vc = kc.clone()
        ks = vs = 1.0
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    for slots, rows in ((pr.hist_slots, pr.hist_rows), (pr.step_slots, pr.step_rows)):
        if slots.size == 0:
            continue
        k = to_dev(pr.k_tok[rows])
        v = to_dev(pr.v_tok[rows])
        sm = to_dev(slots)
        if e4m3:
            kvq.kv_append_e4m3(k, v, sm, kc, vc, ks, vs, err)
        else:
            kvq.kv_append_fp16(k, v, sm, kc, vc, err)
    ti = tl = None
    if pr.topk_idx is not None:
        ti, tl = to_dev(pr.topk_idx), to_dev(pr.topk_lens)
    return DeviceProblem(pr, to_dev(pr.q), kc, vc, to_dev(pr.layout.block_tables),
                         to_dev(pr.layout.lens), ti, tl, ks, vs, e4m3, err)


def run_attention(dp: DeviceProblem, num_splits=0, topk=True, partial=False, block_tables=None,
                  k_cache=None, v_cache=None, context_lens=None, q=None, split_pages=0,
                  bitcast_decode=False, mma_sync=False, fp8_qk=False, longest_first=False):
    q = dp.q if q is None else q
    bt = dp.block_tables if block_tables is None else block_tables
    kc = dp.k_cache if k_cache is None else k_cache
    vc = dp.v_cache if v_cache is None else v_cache
    cl = dp.context_lens if context_lens is None else context_lens
    ti, tl = (dp.topk_idx, dp.topk_lens) if topk else (None, None)
    p = kvq.AttnParams(q.shape[0], q.shape[1], q.shape[2], kc.shape[1], q.shape[3], num_splits,
                       bt.shape[1], 0 if ti is None else ti.shape[2], 0.0, split_pages,
                       kvq._flags(bitcast_decode, mma_sync, fp8_qk, False, longest_first))
    ws = kvq.alloc_workspace(p, q.device)
    ws.fill_(float("nan"))
    if partial:
        if dp.e4m3:
            kvq.paged_decode_attn_e4m3_partial(q, kc, vc, bt, cl, dp.k_scale, dp.v_scale, ws, ti, tl,
                                               num_splits, err_flag=dp.err, split_pages=split_pages,
                                               bitcast_decode=bitcast_decode, mma_sync=mma_sync,
                                               fp8_qk=fp8_qk, longest_first=longest_first)
        else:
            kvq.paged_decode_attn_fp16_partial(q, kc, vc, bt, cl, ws, ti, tl, num_splits,
                                               err_flag=dp.err, split_pages=split_pages,
                                               mma_sync=mma_sync, longest_first=longest_first)
        return ws, p
    if dp.e4m3:
        out = kvq.paged_decode_attn_e4m3(q, kc, vc, bt, cl, dp.k_scale, dp.v_scale, ws, None, ti, tl,
                                         num_splits, err_flag=dp.err, split_pages=split_pages,
                                         bitcast_decode=bitcast_decode, mma_sync=mma_sync,
                                         fp8_qk=fp8_qk, longest_first=longest_first)
    else:
        out = kvq.paged_decode_attn_fp16(q, kc, vc, bt, cl, ws, None, ti, tl, num_splits,
                                         err_flag=dp.err, split_pages=split_pages, mma_sync=mma_sync,
                                         longest_first=longest_first)
    return out


def assert_close(got, ref, what="", atol=2e-3, rtol=1e-2):
    got = np.asarray(got, np.float64)
    ok = P.tolerance_ok(got, ref, atol, rtol)
    if not ok.all():
        bad = np.argwhere(~ok)[:5]
        detail = [(tuple(i), float(got[tuple(i)]), float(ref[tuple(i)])) for i in bad]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outside atol {atol} rtol {rtol}: {detail}")
