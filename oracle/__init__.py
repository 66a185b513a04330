"""CPU oracle for the calibrated E4M3 paged KV cache -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  The product (the CUDA library and its
Python binding) never imports, links or calls it, and it never imports the
product: the two share no code.  The arithmetic lives in ``kvq_oracle.c``
(plain C, binary64 attention, integer-rounded E4M3 encoder); this module only
builds that file with gcc and marshals numpy arrays into it.

Every function is pinned in tests against something other than itself:
exhaustive library conversions (torch / ml_dtypes float8_e4m3fn), closed
forms, invariants and brute force on tiny inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libkvq_oracle.so")
_lock = threading.Lock()
_lib = None

BAD_PAGE, BAD_SLOT, BAD_TOPK, BAD_LEN = 1, 2, 4, 8


def build(force: bool = False) -> str:
    """Compile kvq_oracle.c with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c99", "-fno-fast-math", "-ffp-contract=off",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
        return _lib


def build_variant(src_text: str, out_path: str) -> str:
    """Compile an edited copy of the oracle source (used by the mutation tests,
    which plant a mistake in the oracle and check that a pin catches it)."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O2", "-std=c99", "-fno-fast-math", "-ffp-contract=off",
                    "-fPIC", "-shared", "-o", out_path, src, "-lm"], check=True)
    return out_path


class use_library:
    """Context manager: route every oracle call through another build."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        _load()
        self._saved = _lib
        _lib = _configure(ctypes.CDLL(self.path))
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _configure(lib):
    P = ctypes.c_void_p
    i32, i64, f32, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_double
    lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_to_f64.restype = f64
    lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_decode.restype = f64
    lib.oracle_e4m3_encode_f32.argtypes = [f32]
    lib.oracle_e4m3_encode_f32.restype = ctypes.c_uint8
    lib.oracle_quantize.argtypes = [ctypes.c_uint16, f32]
    lib.oracle_quantize.restype = ctypes.c_uint8
    lib.oracle_quantize_array.argtypes = [P, i64, f32, P]
    lib.oracle_quantize_array.restype = None
    lib.oracle_calibrate_scale.argtypes = [P, i64]
    lib.oracle_calibrate_scale.restype = f32
    lib.oracle_count_bad_scales.argtypes = [P, P, ctypes.c_int]
    lib.oracle_count_bad_scales.restype = ctypes.c_int
    lib.oracle_append_e4m3.argtypes = [P, P, P, i32, i32, i32, P, P, i64, f32, f32]
    lib.oracle_append_e4m3.restype = ctypes.c_int
    lib.oracle_append_fp16.argtypes = [P, P, P, i32, i32, i32, P, P, i64]
    lib.oracle_append_fp16.restype = ctypes.c_int
    attn_args = [P, P, P, ctypes.c_int, i64, P, P, f64, f64, P, P,
                 ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                 ctypes.c_int, ctypes.c_int, f64, P, P]
    lib.oracle_attn.argtypes = attn_args + [P, P]
    lib.oracle_attn.restype = ctypes.c_int
    lib.oracle_attn_partials.argtypes = attn_args + [ctypes.c_int, ctypes.c_int, P, P, P]
    lib.oracle_attn_partials.restype = ctypes.c_int
    lib.oracle_combine.argtypes = [P, P, P, i64, ctypes.c_int, ctypes.c_int, P]
    lib.oracle_combine.restype = None
    lib.oracle_quantize_q_groups.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, P, P]
    lib.oracle_quantize_q_groups.restype = ctypes.c_int
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _as(a, dtype):
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def _f16_bits(x):
    a = np.ascontiguousarray(np.asarray(x))
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype == np.uint16:
        return a
    raise TypeError(f"expected float16 or uint16 bits, got {a.dtype}")


# ---------------------------------------------------------------------------
# scalar and element-wise format functions

def f16_to_f64(bits: int) -> float:
    return _load().oracle_f16_to_f64(int(bits))


def e4m3_decode(code: int) -> float:
    """OCP E4M3 (E4M3FN) byte -> value (NaN for 0x7F / 0xFF)."""
    return _load().oracle_e4m3_decode(int(code))


def e4m3_decode_array(codes) -> np.ndarray:
    lib = _load()
    c = _as(codes, np.uint8)
    table = np.array([lib.oracle_e4m3_decode(i) for i in range(256)], dtype=np.float64)
    return table[c]


def e4m3_encode_f32(v: float) -> int:
    return int(_load().oracle_e4m3_encode_f32(ctypes.c_float(v)))


def quantize(x, scale: float) -> np.ndarray:
    """code = E4M3_RNE_sat(fp32(x) / scale) for an fp16 array x."""
    lib = _load()
    bits = _f16_bits(x)
    out = np.empty(bits.shape, dtype=np.uint8)
    lib.oracle_quantize_array(_ptr(bits), bits.size, ctypes.c_float(scale), _ptr(out))
    return out


def calibrate_scale(x) -> float:
    """scale = fp32(amax) / 448 over an fp16 calibration tensor (0.0 if invalid)."""
    bits = _f16_bits(x)
    return float(np.float32(_load().oracle_calibrate_scale(_ptr(bits), bits.size)))


def count_bad_scales(k_scales, v_scales) -> int:
    k = _as(k_scales, np.float32)
    v = _as(v_scales, np.float32)
    if k.shape != v.shape:
        return -1
    return _load().oracle_count_bad_scales(_ptr(k), _ptr(v), k.size)


# ---------------------------------------------------------------------------
# paged append

def append_e4m3(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale) -> int:
    """Quantise-on-append into pools [P][Hkv][4][D] (uint8), in place."""
    kb, vb = _f16_bits(k_new), _f16_bits(v_new)
    T, Hkv, D = kb.shape
    sm = _as(slot_mapping, np.int32)
    assert k_cache.dtype == np.uint8 and k_cache.flags.c_contiguous
    assert v_cache.dtype == np.uint8 and v_cache.flags.c_contiguous
    P = k_cache.shape[0]
    return _load().oracle_append_e4m3(_ptr(kb), _ptr(vb), _ptr(sm), T, Hkv, D,
                                      _ptr(k_cache), _ptr(v_cache), P,
                                      ctypes.c_float(k_scale), ctypes.c_float(v_scale))


def append_fp16(k_new, v_new, slot_mapping, k_cache, v_cache) -> int:
    kb, vb = _f16_bits(k_new), _f16_bits(v_new)
    T, Hkv, D = kb.shape
    sm = _as(slot_mapping, np.int32)
    kc, vc = k_cache.view(np.uint16), v_cache.view(np.uint16)
    assert kc.flags.c_contiguous and vc.flags.c_contiguous
    P = k_cache.shape[0]
    return _load().oracle_append_fp16(_ptr(kb), _ptr(vb), _ptr(sm), T, Hkv, D,
                                      _ptr(kc), _ptr(vc), P)


# ---------------------------------------------------------------------------
# attention

def quantize_q_groups(q, num_kv_heads: int):
    """The FP8 score variant's query quantisation: per (sequence, kv head) one
    binary32 scale amax / 448 over the G * q_len rows of the group (1 for an
    all-zero group), every element quantised like a cache element.
    q fp16 [B][q_len][Hq][D].  Returns (codes uint8 [B][q_len][Hq][D],
    scales float32 [B][Hkv])."""
    qb = _f16_bits(q)
    B, q_len, Hq, D = qb.shape
    codes = np.zeros(qb.shape, dtype=np.uint8)
    scales = np.zeros((B, num_kv_heads), dtype=np.float32)
    rc = _load().oracle_quantize_q_groups(_ptr(qb), B, q_len, Hq, int(num_kv_heads), D,
                                          _ptr(codes), _ptr(scales))
    if rc != 0:
        raise ValueError("oracle_quantize_q_groups: bad arguments")
    return codes, scales


def _attn_common(q, k_cache, v_cache, block_tables, context_lens, k_scale, v_scale,
                 topk_idx, topk_lens, sm_scale, fp8_q=False):
    qb = _f16_bits(q)
    B, q_len, Hq, D = qb.shape
    is_e4m3 = 1 if k_cache.dtype == np.uint8 else 0
    kc = np.ascontiguousarray(k_cache if is_e4m3 else k_cache.view(np.uint16))
    vc = np.ascontiguousarray(v_cache if is_e4m3 else v_cache.view(np.uint16))
    P, Hkv = kc.shape[0], kc.shape[1]
    assert kc.shape == (P, Hkv, 4, D) and vc.shape == kc.shape
    bt = _as(block_tables, np.int32)
    cl = _as(context_lens, np.int32)
    assert bt.shape[0] == B and cl.shape == (B,)
    ti = tl = None
    max_topk = 0
    if topk_idx is not None:
        ti = _as(topk_idx, np.int32)
        tl = _as(topk_lens, np.int32)
        assert ti.shape[:2] == (B, Hkv) and tl.shape == (B,)
        max_topk = ti.shape[2]
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    qc = qs = None
    if fp8_q:
        qc, qs = quantize_q_groups(qb, Hkv)
    keep = (qb, kc, vc, bt, cl, ti, tl, qc, qs)
    args = [_ptr(qb), _ptr(kc), _ptr(vc), is_e4m3, P, _ptr(bt), _ptr(cl),
            float(k_scale), float(v_scale), _ptr(ti), _ptr(tl),
            B, q_len, Hq, Hkv, D, bt.shape[1], max_topk, float(sm_scale), _ptr(qc), _ptr(qs)]
    return keep, args, (B, q_len, Hq, D)


def attention(q, k_cache, v_cache, block_tables, context_lens, k_scale=1.0, v_scale=1.0,
              topk_idx=None, topk_lens=None, sm_scale=None, return_lse=False, fp8_q=False):
    """Plain binary64 decode / verify attention over a paged cache.

    q fp16 [B][q_len][Hq][D]; caches uint8 (E4M3 arm) or fp16 [P][Hkv][4][D];
    block_tables int32 [B][max_pages]; context_lens int32 [B] (including the
    q_len tokens of this step).  fp8_q: the scores use the query quantised by
    quantize_q_groups (decoded code times its group's scale) instead of the
    fp16 query.  Returns (out [B][q_len][Hq][D] float64,
    flags[, lse [B][q_len][Hq]]).
    """
    keep, args, (B, q_len, Hq, D) = _attn_common(q, k_cache, v_cache, block_tables,
                                                 context_lens, k_scale, v_scale,
                                                 topk_idx, topk_lens, sm_scale, fp8_q)
    out = np.zeros((B, q_len, Hq, D), dtype=np.float64)
    lse = np.zeros((B, q_len, Hq), dtype=np.float64)
    flags = _load().oracle_attn(*args, _ptr(out), _ptr(lse))
    del keep
    if flags < 0:
        raise ValueError("oracle_attn: bad arguments")
    return (out, flags, lse) if return_lse else (out, flags)


def attention_partials(q, k_cache, v_cache, block_tables, context_lens, num_splits,
                       k_scale=1.0, v_scale=1.0, topk_idx=None, topk_lens=None, sm_scale=None,
                       split_pages=0, fp8_q=False):
    """Per-split partials: o [B][Hq][q_len][S][D], m and l [B][Hq][q_len][S].
    split_pages = 0 divides each sequence into S equal parts; > 0 gives every
    split that many pages (4 list entries per page in top-k mode)."""
    keep, args, (B, q_len, Hq, D) = _attn_common(q, k_cache, v_cache, block_tables,
                                                 context_lens, k_scale, v_scale,
                                                 topk_idx, topk_lens, sm_scale, fp8_q)
    S = int(num_splits)
    o = np.zeros((B, Hq, q_len, S, D), dtype=np.float64)
    m = np.zeros((B, Hq, q_len, S), dtype=np.float64)
    l = np.zeros((B, Hq, q_len, S), dtype=np.float64)
    flags = _load().oracle_attn_partials(*args, S, int(split_pages), _ptr(o), _ptr(m), _ptr(l))
    del keep
    if flags < 0:
        raise ValueError("oracle_attn_partials: bad arguments")
    return o, m, l, flags


def combine(o, m, l) -> np.ndarray:
    """Log-sum-exp combine of split partials along the split axis."""
    o = _as(o, np.float64)
    m = _as(m, np.float64)
    l = _as(l, np.float64)
    S, D = o.shape[-2], o.shape[-1]
    rows = int(np.prod(o.shape[:-2]))
    out = np.zeros(o.shape[:-2] + (D,), dtype=np.float64)
    _load().oracle_combine(_ptr(o), _ptr(m), _ptr(l), rows, S, D, _ptr(out))
    return out
