"""The C ABI library: it builds, loads, exports every symbol include/kvq.h
declares, and its host-side checks fail closed (CPU only: nothing here
launches a kernel or touches a device)."""
import ctypes
import math
import os
import re

import pytest

from fp8_paged_kv_e4m3_gb300 import build, kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return kvq.load()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "kvq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "sizeof")))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for must in ("kv_append_e4m3", "kv_append_fp16", "paged_decode_attn_e4m3",
                 "paged_decode_attn_fp16", "kvq_attn_workspace_bytes", "kvq_validate_scales"):
        assert must in names
    assert set(names) == set(kvq.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_library_has_no_torch_dependency():
    # plain C ABI: the shared object must not need libtorch / libc10
    with open(kvq.LIB_PATH, "rb") as f:
        blob = f.read()
    assert b"libtorch" not in blob and b"libc10" not in blob


def test_version_and_status_strings(lib):
    assert lib.kvq_version() == 1
    assert lib.kvq_status_string(0) == b"ok"
    assert b"scale" in lib.kvq_status_string(-2)


def test_scale_gate_fails_closed(lib):
    ok = [0.01] * 24
    kvq.validate_scales(ok, ok)
    for bad in (0.0, -1.0, math.nan, math.inf):
        k = list(ok)
        k[7] = bad
        with pytest.raises(kvq.KvqError) as e:
            kvq.validate_scales(k, ok)
        assert e.value.status == -2
    with pytest.raises(kvq.KvqError):
        kvq.validate_scales(ok[:23], ok)   # missing entry: no default is substituted


def test_scale_from_amax(lib):
    assert kvq.scale_from_amax(448.0) == 1.0
    assert kvq.scale_from_amax(56.0) == 0.125
    for bad in (0.0, -3.0, math.inf, math.nan):
        assert kvq.scale_from_amax(bad) == 0.0


def _params(**kw):
    p = dict(batch=2, q_len=1, num_q_heads=8, num_kv_heads=2, head_dim=64, num_splits=2,
             max_pages_per_seq=25, max_topk=0, sm_scale=0.0, split_pages=0, flags=0)
    p.update(kw)
    return kvq.AttnParams(**p)


def test_workspace_size_matches_layout(lib):
    p = _params()
    units = 2 * 8 * 1 * 2
    r = lambda n: (n + 255) // 256 * 256
    assert lib.kvq_attn_workspace_bytes(ctypes.byref(p)) == r(units * 64 * 4) + 2 * r(units * 4)
    assert lib.kvq_attn_num_splits(ctypes.byref(p)) == 2


@pytest.mark.parametrize("field,value,status", [
    ("head_dim", 96, -4), ("q_len", 5, -4), ("q_len", 0, -1), ("num_kv_heads", 3, -1),
    ("num_splits", -1, -1), ("max_pages_per_seq", 0, -1), ("num_q_heads", 136, -4),
    ("flags", 64, -1), ("flags", -1, -1),
])
def test_bad_params_are_refused(lib, field, value, status):
    p = _params(**{field: value})
    if field == "num_q_heads":
        p.num_kv_heads = 2    # 68 rows per kv head > 64
    assert lib.kvq_attn_workspace_bytes(ctypes.byref(p)) == 0
    assert lib.kvq_attn_num_splits(ctypes.byref(p)) == status


def test_fixed_size_splits_must_cover_every_page(lib):
    # 25 pages in splits of 8 pages need 4 splits
    assert lib.kvq_attn_num_splits(ctypes.byref(_params(num_splits=0, split_pages=8))) == 4
    assert lib.kvq_attn_num_splits(ctypes.byref(_params(num_splits=4, split_pages=8))) == 4
    assert lib.kvq_attn_num_splits(ctypes.byref(_params(num_splits=9, split_pages=8))) == 9
    assert lib.kvq_attn_num_splits(ctypes.byref(_params(num_splits=3, split_pages=8))) == -1
    assert lib.kvq_attn_workspace_bytes(ctypes.byref(_params(num_splits=3, split_pages=8))) == 0
    # a top-k list of 200 entries in splits of 8 pages (32 entries) needs 7
    p = _params(num_splits=0, split_pages=8, max_topk=200)
    assert lib.kvq_attn_num_splits(ctypes.byref(p)) == 7
    assert lib.kvq_attn_num_splits(ctypes.byref(_params(num_splits=6, split_pages=8, max_topk=200))) == -1
    assert lib.kvq_attn_num_splits(ctypes.byref(_params(split_pages=-1))) == -1
    # more than 65535 automatic splits is refused
    assert lib.kvq_attn_num_splits(ctypes.byref(_params(num_splits=0, split_pages=1,
                                                        max_pages_per_seq=70000))) == -4


FAKE = ctypes.c_void_p(0x10000)     # never dereferenced: every call below fails before a launch


def _attn(lib, p, k_scale=0.1, v_scale=0.1, ws_bytes=1 << 20, q=FAKE, ws=FAKE, topk=None):
    return lib.paged_decode_attn_e4m3(q, FAKE, FAKE, 40, FAKE, FAKE, ctypes.c_float(k_scale),
                                      ctypes.c_float(v_scale), topk, None, ws, ws_bytes, FAKE,
                                      ctypes.byref(p), None, None)


def test_attention_host_checks_fail_closed(lib):
    p = _params()
    assert _attn(lib, p, k_scale=0.0) == -2
    assert _attn(lib, p, v_scale=math.nan) == -2
    assert _attn(lib, p, ws_bytes=16) == -3
    assert _attn(lib, p, ws=None) == -3
    assert _attn(lib, p, q=ctypes.c_void_p(0x10008)) == -6
    assert _attn(lib, p, topk=FAKE) == -1          # top-k indices without lengths
    assert _attn(lib, _params(head_dim=80)) == -4


def _attn_fp16(lib, p):
    return lib.paged_decode_attn_fp16(FAKE, FAKE, FAKE, 40, FAKE, FAKE, None, None, FAKE, 1 << 20, FAKE,
                                      ctypes.byref(p), None, None)


def test_fp8_scores_outside_the_tcgen05_shapes_are_unsupported(lib):
    fp8 = kvq.ATTN_FP8_QK
    verify = dict(head_dim=128, q_len=4, num_q_heads=8, num_kv_heads=2)   # 16 rows per kv head
    assert _attn(lib, _params(flags=fp8)) == -4                            # head_dim 64
    assert _attn(lib, _params(flags=fp8, head_dim=128)) == -4              # 4 rows: the mma.sync kernel's
    assert _attn(lib, _params(flags=fp8 | kvq.ATTN_BITCAST_DECODE, **verify)) == -4
    assert _attn(lib, _params(flags=fp8 | kvq.ATTN_MMA_SYNC, **verify)) == -4
    assert _attn_fp16(lib, _params(flags=fp8, **verify)) == -4           # fp16 pools
    assert _attn(lib, _params(flags=fp8, **verify), k_scale=0.0) == -2    # the scale gate comes first


def test_scheduling_flags_change_no_sizes(lib):
    """Strict ordering and longest-first order are scheduling choices: the same
    split count and workspace as without them, for decode and verify shapes."""
    for shape in (dict(), dict(head_dim=128, q_len=4)):
        base = _params(**shape)
        for f in (kvq.ATTN_STRICT_ORDER, kvq.ATTN_LONGEST_FIRST, kvq.ATTN_STRICT_ORDER | kvq.ATTN_LONGEST_FIRST):
            p = _params(flags=f, **shape)
            assert lib.kvq_attn_num_splits(ctypes.byref(p)) == lib.kvq_attn_num_splits(ctypes.byref(base))
            assert lib.kvq_attn_workspace_bytes(ctypes.byref(p)) == lib.kvq_attn_workspace_bytes(ctypes.byref(base))
    assert kvq._flags(False, False, False, True, True) == kvq.ATTN_STRICT_ORDER | kvq.ATTN_LONGEST_FIRST


def test_append_host_checks_fail_closed(lib):
    f = lib.kv_append_e4m3
    assert f(FAKE, FAKE, FAKE, 4, 2, 64, FAKE, FAKE, 10, ctypes.c_float(0.0), ctypes.c_float(1.0), None, None) == -2
    assert f(FAKE, FAKE, FAKE, 4, 2, 60, FAKE, FAKE, 10, ctypes.c_float(1.0), ctypes.c_float(1.0), None, None) == -4
    assert f(FAKE, FAKE, FAKE, -1, 2, 64, FAKE, FAKE, 10, ctypes.c_float(1.0), ctypes.c_float(1.0), None, None) == -1
    assert f(ctypes.c_void_p(0x10004), FAKE, FAKE, 4, 2, 64, FAKE, FAKE, 10, ctypes.c_float(1.0),
             ctypes.c_float(1.0), None, None) == -6
    assert f(None, None, None, 0, 2, 64, None, None, 10, ctypes.c_float(1.0), ctypes.c_float(1.0), None, None) == 0


def _step(lib, p, k_new=FAKE, v_new=FAKE, k_scale=0.1, ws_bytes=1 << 20):
    return lib.paged_decode_step_e4m3(FAKE, k_new, v_new, FAKE, FAKE, 40, FAKE, FAKE, ctypes.c_float(k_scale),
                                      ctypes.c_float(0.1), FAKE, ws_bytes, FAKE, ctypes.byref(p), None, None)


def test_fused_step_host_checks_fail_closed(lib):
    p = _params()
    assert _step(lib, p, k_new=None) == -1
    assert _step(lib, p, v_new=None) == -1
    assert _step(lib, p, k_scale=0.0) == -2
    assert _step(lib, p, ws_bytes=16) == -3
    assert _step(lib, p, k_new=ctypes.c_void_p(0x10008)) == -6
    assert _step(lib, p, v_new=ctypes.c_void_p(0x10004)) == -6
    assert _step(lib, _params(head_dim=80)) == -4
    assert _step(lib, _params(q_len=5)) == -4
    assert _step(lib, _params(flags=kvq.ATTN_BITCAST_DECODE)) == -4     # the fused instances: hardware decoder
    assert _step(lib, _params(flags=kvq.ATTN_FP8_QK, head_dim=128, q_len=4)) == -4
    f16 = lib.paged_decode_step_fp16
    assert f16(FAKE, None, FAKE, FAKE, FAKE, 40, FAKE, FAKE, FAKE, 1 << 20, FAKE, ctypes.byref(p), None, None) == -1
    assert f16(FAKE, FAKE, FAKE, FAKE, FAKE, 40, FAKE, FAKE, FAKE, 16, FAKE, ctypes.byref(p), None, None) == -3


def test_launch_count_query(lib):
    """kvq_attn_launches: the kernels a call launches (host only).  Without a GPU
    the library assumes 148 SMs, so one wave holds 592 E4M3 or 296 fp16 CTAs of
    the split kernel."""
    f = lambda p, e4m3, fused=0: lib.kvq_attn_launches(ctypes.byref(p), e4m3, fused)
    dec = dict(batch=32, q_len=1, num_q_heads=32, num_kv_heads=4, head_dim=128, num_splits=4,
               max_pages_per_seq=1024)
    assert f(_params(**dec), 1) == 1 and f(_params(**dec), 1, 1) == 1      # 512 CTAs: the cluster merge
    assert f(_params(**dec), 0) == 2                                        # fp16: 512 > 296, the combine
    assert f(_params(**dict(dec, num_splits=9)), 1) == 2                    # more than 8 splits
    assert f(_params(**dict(dec, batch=40)), 1) == 2                        # 640 CTAs: two waves
    assert f(_params(flags=kvq.ATTN_BITCAST_DECODE, **dec), 1) == 2
    assert f(_params(flags=kvq.ATTN_LONGEST_FIRST, **dec), 1) == 2
    ver = dict(dec, q_len=4, num_splits=4)                                  # 32 rows: the tcgen05 kernel
    assert f(_params(**ver), 1) == 2 and f(_params(**ver), 1, 1) == 3
    assert f(_params(flags=kvq.ATTN_MMA_SYNC, **ver), 1) == 2               # 32 rows on the split kernel
    assert f(_params(batch=0), 1) == 0
    assert f(_params(q_len=0), 1) == -1


def test_python_binding_refuses_fp16_workspace():
    """The split workspace is FP32 by contract; an fp16 buffer is refused before any call
    (the pages' XQA page-4 route broke when handed an fp16 temporary output)."""
    import torch
    with pytest.raises(ValueError):
        # CPU tensors are refused first; the dtype check is exercised on GPU in test_gpu_attention
        kvq._need(torch.zeros(4, dtype=torch.float16), "workspace", torch.float32)


def _pparams(**kw):
    p = dict(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128, max_pages_per_seq=100,
             max_q_len=300, total_q=600, sm_scale=0.0, flags=0)
    p.update(kw)
    return kvq.PrefillParams(**p)


def test_prefill_workspace_size(lib):
    # 100 pages = 400 keys -> 4 tiles of 128 keys; K and V tiles of 32 KiB each
    assert lib.kvq_prefill_workspace_bytes(ctypes.byref(_pparams())) == 2 * 2 * 4 * (2 * 32768 + 16)
    assert lib.kvq_prefill_workspace_bytes(ctypes.byref(_pparams(max_pages_per_seq=32, max_q_len=100))) == 2 * 2 * 1 * (2 * 32768 + 16)


@pytest.mark.parametrize("field,value", [
    ("head_dim", 64), ("num_kv_heads", 3), ("max_q_len", 0), ("max_q_len", 401), ("flags", 1),
    ("batch", -1), ("max_pages_per_seq", 0), ("sm_scale", -1.0), ("total_q", -1),
])
def test_prefill_bad_params_are_refused(lib, field, value):
    assert lib.kvq_prefill_workspace_bytes(ctypes.byref(_pparams(**{field: value}))) == 0


def _prefill(lib, p, k_scale=0.1, v_scale=0.1, ws_bytes=1 << 24, q=FAKE, ws=FAKE, q_start=FAKE):
    return lib.paged_prefill_attn_e4m3(q, FAKE, FAKE, 40, FAKE, FAKE, q_start, ctypes.c_float(k_scale),
                                       ctypes.c_float(v_scale), ws, ws_bytes, FAKE, ctypes.byref(p), None, None)


def test_prefill_host_checks_fail_closed(lib):
    p = _pparams()
    assert _prefill(lib, p, k_scale=0.0) == -2
    assert _prefill(lib, p, v_scale=math.inf) == -2
    assert _prefill(lib, p, ws_bytes=16) == -3
    assert _prefill(lib, p, ws=None) == -3
    assert _prefill(lib, p, q=ctypes.c_void_p(0x10008)) == -6
    assert _prefill(lib, p, q_start=None) == -1
    assert _prefill(lib, _pparams(head_dim=64)) == -4
    assert _prefill(lib, _pparams(batch=0)) == 0          # nothing to do, nothing launched


@pytest.mark.parametrize("longest_first", [False, True])
@pytest.mark.parametrize("name,overrides", [
    ("decode", {}), ("decode32k", {}), ("verify", {}), ("long", {}), ("mixed", {}), ("tiny", {}),
    ("verify", {"num_splits": 0, "split_pages": 256}), ("mixed", {"split_pages": 64}),
    ("mixed", {"batch": 7}), ("decode", {"num_splits": 0}), ("tiny_verify", {}),
])
def test_reference_config_labels_the_library_split_count(lib, name, overrides, longest_first):
    """The reference arm labels its config with the split count of our arm,
    restated in bench.library_splits: it must agree with kvq_attn_num_splits."""
    import bench
    import torch
    from fp8_paged_kv_e4m3_gb300 import inputs
    w = inputs.get(name, **overrides)
    max_pages = inputs.page_layout(w).block_tables.shape[1]
    sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 148
    p = kvq.AttnParams(w.batch, w.q_len, w.num_q_heads, w.num_kv_heads, w.head_dim, w.num_splits, max_pages,
                       w.topk if w.topk > 0 else 0, 0.0, w.split_pages,
                       kvq.ATTN_LONGEST_FIRST if longest_first else 0)
    assert bench.library_splits(w, max_pages, sms, longest_first) == lib.kvq_attn_num_splits(ctypes.byref(p))


def test_bench_output_error_and_saturation_counts():
    """The bench line's E4M3-vs-fp16 report: zero error and unit cosine for
    equal outputs, a known relative RMS for a scaled copy, a turned row
    counted, and elements beyond 448 * scale counted exactly across chunks."""
    torch = pytest.importorskip("torch")
    import bench
    a = torch.randn(3, 2, 4, 16, dtype=torch.float32).to(torch.float16)
    e = bench.output_error([a], [a])
    assert e["max_abs"] == 0.0 and e["rms"] == 0.0 and e["rows_below_0_99_cosine"] == 0
    assert abs(e["min_row_cosine"] - 1.0) < 1e-6 and e["rows"] == 24
    b = a.clone()
    b[0, 0, 0] = -b[0, 0, 0]                      # one row turned around
    e = bench.output_error([a], [b])
    assert e["rows_below_0_99_cosine"] == 1 and e["min_row_cosine"] < -0.99
    e = bench.output_error([a * 1.5], [a])         # E4M3 arm 50 % larger everywhere
    assert abs(e["rel_rms"] - 0.5) < 1e-3
    x = torch.zeros((1 << 26) + 16, dtype=torch.float16)  # spans more than one 2^26-element chunk
    x[5] = 449.0
    x[(1 << 26) + 7] = -500.0
    x[-1] = 448.0                                  # not beyond
    assert bench.count_beyond(x, 448.0) == 2
