"""ctypes binding of libkvq.so (include/kvq.h).

Argument marshalling only: tensors become device pointers, the current torch
stream becomes the cudaStream_t, and dtypes / shapes / devices are checked so
that a wrong buffer is refused before the C call.  Every step of the path
runs in the library's CUDA kernels.  There is no fallback: if the library is
missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libkvq.so")

PAGE_SIZE = 4
KVQ_OK = 0
STATUS = {0: "ok", -1: "invalid argument", -2: "bad scale", -3: "workspace", -4: "unsupported",
          -5: "CUDA error", -6: "alignment"}
DEV_BAD_PAGE, DEV_BAD_SLOT, DEV_BAD_TOPK, DEV_BAD_LEN, DEV_TIMEOUT = 1, 2, 4, 8, 16
ATTN_BITCAST_DECODE = 1
ATTN_MMA_SYNC = 2
ATTN_FP8_QK = 4
ATTN_STRICT_ORDER = 8
ATTN_LONGEST_FIRST = 32

_lock = threading.Lock()
_lib = None


class KvqError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)} ({status})")


class AttnParams(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("q_len", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("num_splits", ctypes.c_int32),
                ("max_pages_per_seq", ctypes.c_int32), ("max_topk", ctypes.c_int32),
                ("sm_scale", ctypes.c_float), ("split_pages", ctypes.c_int32),
                ("flags", ctypes.c_int32)]


class PrefillParams(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("max_pages_per_seq", ctypes.c_int32), ("max_q_len", ctypes.c_int32),
                ("total_q", ctypes.c_int32), ("sm_scale", ctypes.c_float), ("flags", ctypes.c_int32)]


EXPORTS = ("kvq_version", "kvq_status_string", "kvq_validate_scales", "kvq_amax_f16",
           "kvq_scale_from_amax", "kv_append_e4m3", "kv_append_fp16", "kvq_attn_num_splits",
           "kvq_attn_workspace_bytes", "paged_decode_attn_e4m3", "paged_decode_attn_fp16",
           "paged_decode_attn_e4m3_partial", "paged_decode_attn_fp16_partial", "kvq_lse_combine",
           "paged_decode_step_e4m3", "paged_decode_step_fp16", "kvq_attn_launches",
           "paged_decode_attn_e4m3_noalloc", "kvq_prefill_workspace_bytes", "paged_prefill_attn_e4m3",
           "paged_prefill_attn_fp16")


def load(path: Optional[str] = None):
    """Load libkvq.so (built by fp8_paged_kv_e4m3_gb300.build); raise if absent."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"CUDA library not built: {p} is missing "
                               "(run `python -m fp8_paged_kv_e4m3_gb300.build`)")
        lib = ctypes.CDLL(p)
        V, P, i32, i64, f32 = (ctypes.c_void_p, ctypes.POINTER(AttnParams), ctypes.c_int32,
                               ctypes.c_int64, ctypes.c_float)
        sz = ctypes.c_size_t
        lib.kvq_version.restype = ctypes.c_int
        lib.kvq_status_string.argtypes = [ctypes.c_int]
        lib.kvq_status_string.restype = ctypes.c_char_p
        lib.kvq_validate_scales.argtypes = [V, V, i32]
        lib.kvq_amax_f16.argtypes = [V, i64, V, V]
        lib.kvq_scale_from_amax.argtypes = [f32]
        lib.kvq_scale_from_amax.restype = f32
        lib.kv_append_e4m3.argtypes = [V, V, V, i32, i32, i32, V, V, i64, f32, f32, V, V]
        lib.kv_append_fp16.argtypes = [V, V, V, i32, i32, i32, V, V, i64, V, V]
        lib.kvq_attn_num_splits.argtypes = [P]
        lib.kvq_attn_num_splits.restype = i32
        lib.kvq_attn_launches.argtypes = [P, i32, i32]
        lib.kvq_attn_launches.restype = i32
        lib.kvq_attn_workspace_bytes.argtypes = [P]
        lib.kvq_attn_workspace_bytes.restype = sz
        lib.paged_decode_attn_e4m3.argtypes = [V, V, V, i64, V, V, f32, f32, V, V, V, sz, V, P, V, V]
        lib.paged_decode_attn_fp16.argtypes = [V, V, V, i64, V, V, V, V, V, sz, V, P, V, V]
        lib.paged_decode_attn_e4m3_partial.argtypes = [V, V, V, i64, V, V, f32, f32, V, V, V, sz, P, V, V]
        lib.paged_decode_attn_fp16_partial.argtypes = [V, V, V, i64, V, V, V, V, V, sz, P, V, V]
        lib.kvq_lse_combine.argtypes = [V, sz, V, P, V]
        lib.paged_decode_step_e4m3.argtypes = [V, V, V, V, V, i64, V, V, f32, f32, V, sz, V, P, V, V]
        lib.paged_decode_step_fp16.argtypes = [V, V, V, V, V, i64, V, V, V, sz, V, P, V, V]
        PP = ctypes.POINTER(PrefillParams)
        lib.kvq_prefill_workspace_bytes.argtypes = [PP]
        lib.kvq_prefill_workspace_bytes.restype = sz
        lib.paged_prefill_attn_e4m3.argtypes = [V, V, V, i64, V, V, V, f32, f32, V, sz, V, PP, V, V]
        lib.paged_prefill_attn_fp16.argtypes = [V, V, V, i64, V, V, V, V, sz, V, PP, V, V]
        for name in ("kvq_validate_scales", "kvq_amax_f16", "kv_append_e4m3", "kv_append_fp16",
                     "paged_decode_attn_e4m3", "paged_decode_attn_fp16",
                     "paged_decode_attn_e4m3_partial", "paged_decode_attn_fp16_partial",
                     "kvq_lse_combine", "paged_decode_step_e4m3", "paged_decode_step_fp16",
                     "paged_prefill_attn_e4m3", "paged_prefill_attn_fp16"):
            getattr(lib, name).restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def _check(fn: str, status: int):
    if status != KVQ_OK:
        raise KvqError(fn, status)


# ---------------------------------------------------------------------------
# marshalling helpers

def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, ndim: Optional[int] = None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name}: expected {ndim} dims, got {tuple(t.shape)}")


# ---------------------------------------------------------------------------
# scales and calibration

def validate_scales(k_scales, v_scales) -> None:
    """Fail closed unless every per-layer K and V scale is finite and > 0."""
    k = (ctypes.c_float * len(k_scales))(*[float(x) for x in k_scales])
    v = (ctypes.c_float * len(v_scales))(*[float(x) for x in v_scales])
    if len(k_scales) != len(v_scales) or len(k_scales) == 0:
        raise KvqError("kvq_validate_scales", -1)
    _check("kvq_validate_scales", load().kvq_validate_scales(k, v, len(k_scales)))


def amax_f16(x: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """max |x| over an fp16 device tensor, as a device float32[1] (no host sync)."""
    _need(x, "x", torch.float16)
    if out is None:
        out = torch.empty(1, dtype=torch.float32, device=x.device)
    _need(out, "amax_out", torch.float32)
    _check("kvq_amax_f16", load().kvq_amax_f16(_ptr(x), x.numel(), _ptr(out), _stream(x)))
    return out


def scale_from_amax(amax: float) -> float:
    return float(load().kvq_scale_from_amax(ctypes.c_float(amax)))


def calibrate_scale(x: torch.Tensor) -> float:
    """scale = amax / 448 of a calibration draw (synchronises to read amax)."""
    return scale_from_amax(float(amax_f16(x).item()))


# ---------------------------------------------------------------------------
# append

def _append_common(k_new, v_new, slot_mapping, k_cache, v_cache, cache_dtype):
    _need(k_new, "k_new", torch.float16, 3)
    _need(v_new, "v_new", torch.float16, 3)
    if k_new.shape != v_new.shape:
        raise ValueError("k_new and v_new shapes differ")
    T, Hkv, D = k_new.shape
    _need(slot_mapping, "slot_mapping", torch.int32, 1)
    if slot_mapping.numel() != T:
        raise ValueError("slot_mapping length != number of tokens")
    for name, c in (("k_cache", k_cache), ("v_cache", v_cache)):
        _need(c, name, cache_dtype, 4)
        if c.shape[1:] != (Hkv, PAGE_SIZE, D):
            raise ValueError(f"{name}: expected [P, {Hkv}, {PAGE_SIZE}, {D}], got {tuple(c.shape)}")
    return T, Hkv, D


def kv_append_e4m3(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale: float, v_scale: float,
                   err_flag: Optional[torch.Tensor] = None) -> None:
    """Quantise fp16 K/V of new tokens into uint8 (E4M3) pools [P][Hkv][4][D]."""
    T, Hkv, D = _append_common(k_new, v_new, slot_mapping, k_cache, v_cache, torch.uint8)
    if err_flag is not None:
        _need(err_flag, "err_flag", torch.int32)
    _check("kv_append_e4m3", load().kv_append_e4m3(
        _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), T, Hkv, D, _ptr(k_cache), _ptr(v_cache),
        k_cache.shape[0], ctypes.c_float(k_scale), ctypes.c_float(v_scale), _ptr(err_flag),
        _stream(k_new)))


def kv_append_fp16(k_new, v_new, slot_mapping, k_cache, v_cache,
                   err_flag: Optional[torch.Tensor] = None) -> None:
    T, Hkv, D = _append_common(k_new, v_new, slot_mapping, k_cache, v_cache, torch.float16)
    if err_flag is not None:
        _need(err_flag, "err_flag", torch.int32)
    _check("kv_append_fp16", load().kv_append_fp16(
        _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), T, Hkv, D, _ptr(k_cache), _ptr(v_cache),
        k_cache.shape[0], _ptr(err_flag), _stream(k_new)))


# ---------------------------------------------------------------------------
# attention

def attn_params(q: torch.Tensor, num_kv_heads: int, max_pages_per_seq: int, num_splits: int = 0,
                max_topk: int = 0, sm_scale: float = 0.0, split_pages: int = 0,
                bitcast_decode: bool = False, mma_sync: bool = False, fp8_qk: bool = False,
                strict_order: bool = False, longest_first: bool = False) -> AttnParams:
    B, q_len, Hq, D = q.shape
    return AttnParams(B, q_len, Hq, num_kv_heads, D, num_splits, max_pages_per_seq, max_topk,
                      sm_scale, split_pages,
                      _flags(bitcast_decode, mma_sync, fp8_qk, strict_order, longest_first))


def _flags(bitcast_decode: bool, mma_sync: bool, fp8_qk: bool = False, strict_order: bool = False,
           longest_first: bool = False) -> int:
    return ((ATTN_BITCAST_DECODE if bitcast_decode else 0) | (ATTN_MMA_SYNC if mma_sync else 0) |
            (ATTN_FP8_QK if fp8_qk else 0) | (ATTN_STRICT_ORDER if strict_order else 0) |
            (ATTN_LONGEST_FIRST if longest_first else 0))


def num_splits(p: AttnParams) -> int:
    s = load().kvq_attn_num_splits(ctypes.byref(p))
    if s < 1:
        raise KvqError("kvq_attn_num_splits", s)
    return s


def attn_launches(p: AttnParams, e4m3: bool, fused_step: bool = False) -> int:
    """Kernels the full call (fused_step: the fused step call) launches with
    these parameters on the current device."""
    n = load().kvq_attn_launches(ctypes.byref(p), int(e4m3), int(fused_step))
    if n < 0:
        raise KvqError("kvq_attn_launches", n)
    return n


def workspace_bytes(p: AttnParams) -> int:
    n = load().kvq_attn_workspace_bytes(ctypes.byref(p))
    if n == 0:
        raise KvqError("kvq_attn_workspace_bytes", -1)
    return n


def alloc_workspace(p: AttnParams, device) -> torch.Tensor:
    """An FP32 workspace of the size the call needs (caller-owned)."""
    return torch.empty(math.ceil(workspace_bytes(p) / 4), dtype=torch.float32, device=device)


def workspace_views(ws: torch.Tensor, p: AttnParams):
    """(tmp_out [B][Hq][q_len][S][D], tmp_max [B][Hq][q_len][S], tmp_sum) views of a workspace."""
    S = num_splits(p)
    units = p.batch * p.num_q_heads * p.q_len * S
    r256 = lambda n: (n + 255) // 256 * 256
    o_n = units * p.head_dim
    m_off = r256(o_n * 4) // 4
    l_off = m_off + r256(units * 4) // 4
    shp = (p.batch, p.num_q_heads, p.q_len, S)
    return (ws[:o_n].view(*shp, p.head_dim), ws[m_off:m_off + units].view(shp),
            ws[l_off:l_off + units].view(shp))


def _attn_check(q, k_cache, v_cache, block_tables, context_lens, workspace, out, topk_idx,
                topk_lens, cache_dtype, num_splits_, sm_scale, split_pages, bitcast_decode=False,
                mma_sync=False, fp8_qk=False, strict_order=False, longest_first=False):
    _need(q, "q", torch.float16, 4)
    B, q_len, Hq, D = q.shape
    _need(k_cache, "k_cache", cache_dtype, 4)
    _need(v_cache, "v_cache", cache_dtype, 4)
    if k_cache.shape != v_cache.shape or k_cache.shape[2:] != (PAGE_SIZE, D):
        raise ValueError(f"caches must be [P, Hkv, {PAGE_SIZE}, {D}]")
    Hkv = k_cache.shape[1]
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    if block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("block_tables / context_lens batch mismatch")
    # the split workspace is FP32 by contract; an fp16 buffer is refused here
    _need(workspace, "workspace", torch.float32)
    if out is not None:
        _need(out, "out", torch.float16, 4)
        if out.shape != q.shape:
            raise ValueError("out must have the shape of q")
    max_topk = 0
    if (topk_idx is None) != (topk_lens is None):
        raise ValueError("topk_idx and topk_lens go together")
    if topk_idx is not None:
        _need(topk_idx, "topk_idx", torch.int32, 3)
        _need(topk_lens, "topk_lens", torch.int32, 1)
        if topk_idx.shape[:2] != (B, Hkv) or topk_lens.shape[0] != B:
            raise ValueError("topk_idx must be [B, Hkv, K], topk_lens [B]")
        max_topk = topk_idx.shape[2]
    p = AttnParams(B, q_len, Hq, Hkv, D, num_splits_, block_tables.shape[1], max_topk, sm_scale,
                   split_pages, _flags(bitcast_decode, mma_sync, fp8_qk, strict_order, longest_first))
    return p


def paged_decode_attn_e4m3(q, k_cache, v_cache, block_tables, context_lens, k_scale: float,
                           v_scale: float, workspace, out=None, topk_idx=None, topk_lens=None,
                           num_splits: int = 0, sm_scale: float = 0.0, err_flag=None,
                           split_pages: int = 0, bitcast_decode: bool = False, mma_sync: bool = False,
                           fp8_qk: bool = False, strict_order: bool = False, longest_first: bool = False):
    """Decode / verify attention over E4M3 pools; returns `out` (fp16, shape of q).
    fp8_qk: scores from the query quantised to E4M3 per (sequence, kv head)
    on E4M3 tensor-core instructions (verify shapes at head_dim 128 only).
    strict_order: read no input before the preceding kernel in the stream
    completes (by default, without a top-k list, block tables, lengths and
    the pages of positions below L - q_len may be read earlier).
    longest_first: the split kernel takes the sequences longest first (for
    batches of varied lengths over several waves; same results)."""
    p = _attn_check(q, k_cache, v_cache, block_tables, context_lens, workspace, out, topk_idx,
                    topk_lens, torch.uint8, num_splits, sm_scale, split_pages, bitcast_decode, mma_sync,
                    fp8_qk, strict_order, longest_first)
    if out is None:
        out = torch.empty_like(q)
    _check("paged_decode_attn_e4m3", load().paged_decode_attn_e4m3(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0], _ptr(block_tables),
        _ptr(context_lens), ctypes.c_float(k_scale), ctypes.c_float(v_scale), _ptr(topk_idx),
        _ptr(topk_lens), _ptr(workspace), workspace.numel() * 4, _ptr(out), ctypes.byref(p),
        _ptr(err_flag), _stream(q)))
    return out


def paged_decode_attn_fp16(q, k_cache, v_cache, block_tables, context_lens, workspace, out=None,
                           topk_idx=None, topk_lens=None, num_splits: int = 0,
                           sm_scale: float = 0.0, err_flag=None, split_pages: int = 0,
                           mma_sync: bool = False, strict_order: bool = False, longest_first: bool = False):
    """fp16-KV twin of paged_decode_attn_e4m3."""
    p = _attn_check(q, k_cache, v_cache, block_tables, context_lens, workspace, out, topk_idx,
                    topk_lens, torch.float16, num_splits, sm_scale, split_pages, False, mma_sync,
                    strict_order=strict_order, longest_first=longest_first)
    if out is None:
        out = torch.empty_like(q)
    _check("paged_decode_attn_fp16", load().paged_decode_attn_fp16(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0], _ptr(block_tables),
        _ptr(context_lens), _ptr(topk_idx), _ptr(topk_lens), _ptr(workspace),
        workspace.numel() * 4, _ptr(out), ctypes.byref(p), _ptr(err_flag), _stream(q)))
    return out


def _step_rows_check(q, k_new, v_new, Hkv):
    B, q_len, _, D = q.shape
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        _need(t, name, torch.float16, 4)
        if t.shape != (B, q_len, Hkv, D):
            raise ValueError(f"{name} must be [B, q_len, Hkv, D] = {(B, q_len, Hkv, D)}")


def paged_decode_step_e4m3(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, k_scale: float,
                           v_scale: float, workspace, out=None, num_splits: int = 0, sm_scale: float = 0.0,
                           err_flag=None, split_pages: int = 0, bitcast_decode: bool = False,
                           mma_sync: bool = False, fp8_qk: bool = False, strict_order: bool = False,
                           longest_first: bool = False):
    """This step's append (k_new, v_new: fp16 [B, q_len, Hkv, D], written at
    positions L - q_len .. L - 1 of each sequence) and the attention over the
    updated cache in one attention launch plus the combine; the same pools
    and outputs as kv_append_e4m3 then paged_decode_attn_e4m3.  Returns out."""
    p = _attn_check(q, k_cache, v_cache, block_tables, context_lens, workspace, out, None, None,
                    torch.uint8, num_splits, sm_scale, split_pages, bitcast_decode, mma_sync, fp8_qk,
                    strict_order, longest_first)
    _step_rows_check(q, k_new, v_new, k_cache.shape[1])
    if out is None:
        out = torch.empty_like(q)
    _check("paged_decode_step_e4m3", load().paged_decode_step_e4m3(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
        _ptr(block_tables), _ptr(context_lens), ctypes.c_float(k_scale), ctypes.c_float(v_scale),
        _ptr(workspace), workspace.numel() * 4, _ptr(out), ctypes.byref(p), _ptr(err_flag), _stream(q)))
    return out


def paged_decode_step_fp16(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, workspace,
                           out=None, num_splits: int = 0, sm_scale: float = 0.0, err_flag=None,
                           split_pages: int = 0, mma_sync: bool = False, strict_order: bool = False,
                           longest_first: bool = False):
    """fp16-KV twin of paged_decode_step_e4m3."""
    p = _attn_check(q, k_cache, v_cache, block_tables, context_lens, workspace, out, None, None,
                    torch.float16, num_splits, sm_scale, split_pages, False, mma_sync,
                    strict_order=strict_order, longest_first=longest_first)
    _step_rows_check(q, k_new, v_new, k_cache.shape[1])
    if out is None:
        out = torch.empty_like(q)
    _check("paged_decode_step_fp16", load().paged_decode_step_fp16(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
        _ptr(block_tables), _ptr(context_lens), _ptr(workspace), workspace.numel() * 4, _ptr(out),
        ctypes.byref(p), _ptr(err_flag), _stream(q)))
    return out


def paged_decode_attn_e4m3_partial(q, k_cache, v_cache, block_tables, context_lens,
                                   k_scale: float, v_scale: float, workspace, topk_idx=None,
                                   topk_lens=None, num_splits: int = 0, sm_scale: float = 0.0,
                                   err_flag=None, split_pages: int = 0,
                                   bitcast_decode: bool = False, mma_sync: bool = False,
                                   fp8_qk: bool = False, strict_order: bool = False,
                                   longest_first: bool = False) -> AttnParams:
    p = _attn_check(q, k_cache, v_cache, block_tables, context_lens, workspace, None, topk_idx,
                    topk_lens, torch.uint8, num_splits, sm_scale, split_pages, bitcast_decode, mma_sync,
                    fp8_qk, strict_order, longest_first)
    _check("paged_decode_attn_e4m3_partial", load().paged_decode_attn_e4m3_partial(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0], _ptr(block_tables),
        _ptr(context_lens), ctypes.c_float(k_scale), ctypes.c_float(v_scale), _ptr(topk_idx),
        _ptr(topk_lens), _ptr(workspace), workspace.numel() * 4, ctypes.byref(p),
        _ptr(err_flag), _stream(q)))
    return p


def paged_decode_attn_fp16_partial(q, k_cache, v_cache, block_tables, context_lens, workspace,
                                   topk_idx=None, topk_lens=None, num_splits: int = 0,
                                   sm_scale: float = 0.0, err_flag=None,
                                   split_pages: int = 0, mma_sync: bool = False,
                                   strict_order: bool = False, longest_first: bool = False) -> AttnParams:
    p = _attn_check(q, k_cache, v_cache, block_tables, context_lens, workspace, None, topk_idx,
                    topk_lens, torch.float16, num_splits, sm_scale, split_pages, False, mma_sync,
                    strict_order=strict_order, longest_first=longest_first)
    _check("paged_decode_attn_fp16_partial", load().paged_decode_attn_fp16_partial(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0], _ptr(block_tables),
        _ptr(context_lens), _ptr(topk_idx), _ptr(topk_lens), _ptr(workspace),
        workspace.numel() * 4, ctypes.byref(p), _ptr(err_flag), _stream(q)))
    return p


def lse_combine(workspace: torch.Tensor, out: torch.Tensor, p: AttnParams) -> torch.Tensor:
    _need(workspace, "workspace", torch.float32)
    _need(out, "out", torch.float16, 4)
    _check("kvq_lse_combine", load().kvq_lse_combine(
        _ptr(workspace), workspace.numel() * 4, _ptr(out), ctypes.byref(p), _stream(out)))
    return out


# ---------------------------------------------------------------------------
# chunked prefill

def prefill_params(q: torch.Tensor, num_kv_heads: int, batch: int, max_pages_per_seq: int,
                   max_q_len: int, sm_scale: float = 0.0) -> PrefillParams:
    """Parameters of a prefill call; q is the packed [total_q, Hq, D] chunk tensor."""
    return PrefillParams(batch, q.shape[1], num_kv_heads, q.shape[2], max_pages_per_seq, max_q_len,
                         q.shape[0], sm_scale, 0)


def prefill_workspace_bytes(p: PrefillParams) -> int:
    n = int(load().kvq_prefill_workspace_bytes(ctypes.byref(p)))
    if n == 0:
        raise KvqError("kvq_prefill_workspace_bytes", -1)
    return n


def alloc_prefill_workspace(p: PrefillParams, device) -> torch.Tensor:
    return torch.empty(prefill_workspace_bytes(p), dtype=torch.uint8, device=device)


def _prefill_check(q, k_cache, v_cache, block_tables, context_lens, q_start, workspace, out,
                   cache_dtype, max_q_len, sm_scale):
    _need(q, "q", torch.float16, 3)
    Tq, Hq, D = q.shape
    _need(k_cache, "k_cache", cache_dtype, 4)
    _need(v_cache, "v_cache", cache_dtype, 4)
    if k_cache.shape != v_cache.shape or k_cache.shape[2:] != (PAGE_SIZE, D):
        raise ValueError(f"caches must be [P, Hkv, {PAGE_SIZE}, {D}]")
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    _need(q_start, "q_start", torch.int32, 1)
    B = context_lens.shape[0]
    if block_tables.shape[0] != B or q_start.shape[0] != B + 1:
        raise ValueError("block_tables [B, max_pages], context_lens [B], q_start [B + 1] expected")
    _need(workspace, "workspace", torch.uint8, 1)
    if out is not None:
        _need(out, "out", torch.float16, 3)
        if out.shape != q.shape:
            raise ValueError("out must have the shape of q")
    if max_q_len is None:
        max_q_len = max(1, Tq)
    return PrefillParams(B, Hq, k_cache.shape[1], D, block_tables.shape[1], max_q_len, Tq, sm_scale, 0)


def paged_prefill_attn_e4m3(q, k_cache, v_cache, block_tables, context_lens, q_start, k_scale: float,
                            v_scale: float, workspace, out=None, max_q_len: Optional[int] = None,
                            sm_scale: float = 0.0, err_flag=None):
    """Chunked-prefill attention over E4M3 pools; q and the returned out are [total_q, Hq, D] fp16,
    q_start [B + 1] the chunk offsets.  max_q_len bounds every chunk (default: total_q)."""
    p = _prefill_check(q, k_cache, v_cache, block_tables, context_lens, q_start, workspace, out,
                       torch.uint8, max_q_len, sm_scale)
    if out is None:
        out = torch.empty_like(q)
    _check("paged_prefill_attn_e4m3", load().paged_prefill_attn_e4m3(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0], _ptr(block_tables), _ptr(context_lens),
        _ptr(q_start), ctypes.c_float(k_scale), ctypes.c_float(v_scale), _ptr(workspace), workspace.numel(),
        _ptr(out), ctypes.byref(p), _ptr(err_flag), _stream(q)))
    return out


def paged_prefill_attn_fp16(q, k_cache, v_cache, block_tables, context_lens, q_start, workspace, out=None,
                            max_q_len: Optional[int] = None, sm_scale: float = 0.0, err_flag=None):
    """fp16-KV twin of paged_prefill_attn_e4m3."""
    p = _prefill_check(q, k_cache, v_cache, block_tables, context_lens, q_start, workspace, out,
                       torch.float16, max_q_len, sm_scale)
    if out is None:
        out = torch.empty_like(q)
    _check("paged_prefill_attn_fp16", load().paged_prefill_attn_fp16(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0], _ptr(block_tables), _ptr(context_lens),
        _ptr(q_start), _ptr(workspace), workspace.numel(), _ptr(out), ctypes.byref(p), _ptr(err_flag),
        _stream(q)))
    return out
