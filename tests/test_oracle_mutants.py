"""Mutation check of the oracle's pins (CPU only).

Each case plants one plausible mistake in a copy of the oracle source (a
dropped term, a wrong sign, bias or index, a transposed operand, a wrong tie
rule), builds it, and asserts that the pins used elsewhere in this suite
reject the mutant.  A pin set that accepted a mutant would not be pinning
that part of the oracle.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from tests import _problems as P
from tests import test_oracle_fp8q as F8
from tests.test_oracle_e4m3 import _F16_FINITE, _torch_decode, _torch_quantize, _same, ALL_CODES

MUTANTS = {
    # E4M3 decoder: exponent bias off by one
    "decode_bias": ("v = ldexp(1.0 + m / 8.0, e - 7);", "v = ldexp(1.0 + m / 8.0, e - 8);"),
    # E4M3 decoder: subnormal scale wrong
    "decode_subnormal": ("v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
    # encoder: ties away from zero instead of to even
    "encode_ties": ("if (rem > half || (rem == half && (q & 1u)))", "if (rem >= half)"),
    # encoder: subnormal shift off by one
    "encode_subnormal": ("rne_shift(sig, 23 - (E + 9))", "rne_shift(sig, 22 - (E + 9))"),
    # quantiser multiplies instead of dividing
    "quantize_mul": ("float q = xf / scale;", "float q = xf * scale;"),
    # calibration forgets the 448
    "calib_448": ("return (float)amax / 448.0f;", "return (float)amax / 256.0f;"),
    # pool layout with slot and head transposed
    "pool_transpose": ("return (((page * Hkv + g) * 4 + slot) * (int64_t)D) + d;",
                       "return (((page * 4 + slot) * Hkv + g) * (int64_t)D) + d;"),
    # GQA grouping interleaved instead of contiguous
    "gqa_interleaved": ("int g = h / G; /* contiguous", "int g = h % pr->Hkv; /* contiguous"),
    # the verify window is not causal
    "no_causal": ("int pos = L - pr->q_len + i;\n    int n = 0, j;", "int pos = L - 1;\n    int n = 0, j;"),
    # causal bound off by one (excludes the diagonal)
    "causal_off_by_one": ("for (j = 0; j <= pos; ++j)", "for (j = 0; j < pos; ++j)"),
    # softmax temperature dropped
    "no_sm_scale": ("scores[k] = s * pr->sm_scale;", "scores[k] = s;"),
    # the first channel of every dot product dropped
    "dot_drops_term": ("            s += oracle_f16_to_f64(qrow[d]) * kv;",
                       "            if (d) s += oracle_f16_to_f64(qrow[d]) * kv;"),
    # combine ignores the split sums
    "combine_no_l": ("w = l[r * S + s] * exp(m[r * S + s] - M);", "w = exp(m[r * S + s] - M);"),
    # FP8 score variant: the query scale forgets the 448
    "qscale_448": ("qs = amax > 0.0 ? (float)amax / 448.0f : 1.0f;", "qs = amax > 0.0 ? (float)amax / 256.0f : 1.0f;"),
    # FP8 score variant: the group maximum taken over the first window row only
    "qgroup_scope": ("for (i = 0; i < q_len; ++i)\n                for (h = g * G; h < (g + 1) * G; ++h)\n"
                     "                    for (d = 0; d < D; ++d) {\n                        double a",
                     "for (i = 0; i < 1; ++i)\n                for (h = g * G; h < (g + 1) * G; ++h)\n"
                     "                    for (d = 0; d < D; ++d) {\n                        double a"),
    # FP8 score variant: the decoded query code used without its scale
    "qscale_dropped": ("s += oracle_e4m3_decode(qcode[d]) * qscale * kv;", "s += oracle_e4m3_decode(qcode[d]) * kv;"),
    # FP8 score variant: every group read with the scale of kv head 0
    "qscale_group": ("(double)pr->q_scales[(int64_t)b * pr->Hkv + g]", "(double)pr->q_scales[(int64_t)b * pr->Hkv]"),
    # V scale applied to K
    "swapped_scales": ("return oracle_e4m3_decode(c[idx]) * (is_k ? pr->k_scale : pr->v_scale);",
                       "return oracle_e4m3_decode(c[idx]) * (is_k ? pr->v_scale : pr->k_scale);"),
}


def _pins_pass() -> bool:
    """A compact run of the suite's pins; False as soon as one rejects."""
    # format
    if not _same(oracle.e4m3_decode_array(ALL_CODES), _torch_decode(ALL_CODES)).all():
        return False
    for scale in (1.0, 0.0116, 3.7):
        s32 = float(np.float32(scale))
        if not (oracle.quantize(_F16_FINITE, s32) == _torch_quantize(_F16_FINITE, s32)).all():
            return False
    x = np.random.default_rng(7).standard_normal(512).astype(np.float16)
    x[3] = np.float16(-56.0)
    if oracle.calibrate_scale(x) != 0.125:
        return False
    # attention against the library reference, dense and verify, with the split check
    for name in ("tiny", "tiny_verify"):
        pr = P.host_problem(name)
        kc, vc, ks, vs = P.oracle_pools(pr)
        bt, lens = pr.layout.block_tables, pr.layout.lens
        # appended bytes against the library conversion
        row = pr.hist_rows[5]
        slot = int(pr.hist_slots[5])
        xk = torch.from_numpy(pr.k_tok[row].astype(np.float32)) / torch.tensor(ks, dtype=torch.float32)
        ref_bytes = torch.clamp(xk, -448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        if not np.array_equal(kc[slot // 4, :, slot % 4, :], ref_bytes):
            return False
        out, _ = oracle.attention(pr.q, kc, vc, bt, lens, ks, vs)
        ref = P.torch_reference(pr.q, P.torch_dequant(kc, ks), P.torch_dequant(vc, vs), bt, lens,
                                pr.w.q_len)
        if not np.allclose(out, ref, rtol=1e-10, atol=1e-12):
            return False
        o, m, l, _ = oracle.attention_partials(pr.q, kc, vc, bt, lens, 3, ks, vs)
        if not np.allclose(oracle.combine(o, m, l).transpose(0, 2, 1, 3), out, rtol=1e-10, atol=1e-12):
            return False
        # FP8 score variant: the query codes against the library cast, and a query
        # already on the scaled grid reproduced exactly
        codes, scales = oracle.quantize_q_groups(pr.q, pr.w.num_kv_heads)
        ref_codes, ref_scales = F8._library_route(pr.q, pr.w.num_kv_heads)
        if not (np.array_equal(codes, ref_codes) and np.array_equal(scales, ref_scales)):
            return False
        qg, _, _ = F8._grid_query(pr, np.random.default_rng(11))
        a, _ = oracle.attention(qg, kc, vc, bt, lens, ks, vs)
        b, _ = oracle.attention(qg, kc, vc, bt, lens, ks, vs, fp8_q=True)
        if not np.array_equal(a, b):
            return False
    return True


def test_unmutated_oracle_passes_the_pins():
    assert _pins_pass()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = oracle.build_variant(src.replace(old, new), os.path.join(tmp_path, f"lib_{name}.so"))
    with oracle.use_library(path):
        caught = not _pins_pass()
    assert caught, f"pins accepted the mutant {name}"
