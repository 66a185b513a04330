"""Pins for the oracle's E4M3 format functions (CPU only).

The oracle's decoder, encoder, quantiser and calibration are checked against
things other than themselves: the E4M3FN conversions of two independent
libraries (torch.float8_e4m3fn, ml_dtypes.float8_e4m3fn), an exact-rational
brute-force nearest-value search, the OCP format table in tests/golden/, and
closed-form tie / saturation / error-bound cases.
"""
import fractions
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ALL_CODES = np.arange(256, dtype=np.uint8)


def _torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def _same(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    both_nan = np.isnan(a) & np.isnan(b)
    eq = (a == b) & (np.signbit(a) == np.signbit(b))
    return both_nan | eq


# ---------------------------------------------------------------------------
# decoder

def test_decode_exhaustive_vs_torch():
    ours = oracle.e4m3_decode_array(ALL_CODES)
    assert _same(ours, _torch_decode(ALL_CODES)).all()


def test_decode_exhaustive_vs_ml_dtypes():
    ml_dtypes = pytest.importorskip("ml_dtypes")
    ref = ALL_CODES.view(ml_dtypes.float8_e4m3fn).astype(np.float64)
    assert _same(oracle.e4m3_decode_array(ALL_CODES), ref).all()


def _golden_table():
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_format_points.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            code, value = line.split()
            rows.append((int(code, 16), value))
    return rows


def test_decode_golden_format_points():
    rows = _golden_table()
    assert len(rows) >= 10
    for code, value in rows:
        got = oracle.e4m3_decode(code)
        if value == "nan":
            assert math.isnan(got), hex(code)
        else:
            want = float(fractions.Fraction(value))
            if value.startswith("-"):
                want = -abs(want)  # keeps the sign of -0
            assert got == want and math.copysign(1, got) == math.copysign(1, want), (hex(code), got, want)


def test_decode_structure():
    v = oracle.e4m3_decode_array(ALL_CODES)
    finite = v[np.isfinite(v)]
    assert finite.size == 254                       # 0x7F and 0xFF are the only NaNs
    assert np.unique(finite).size == 253             # +0 and -0 coincide
    pos = v[:0x7F]
    assert (np.diff(pos) > 0).all()                  # 0x00..0x7E strictly increasing
    assert (v[0x80:0xFF] == -v[0x00:0x7F]).all()     # sign-magnitude symmetry
    assert np.nanmax(np.abs(v)) == 448.0


# ---------------------------------------------------------------------------
# encoder: exhaustive over binary16 inputs, against two libraries and brute force

SCALES = [1.0, 2.0 ** -3, 2.0 ** 4, 0.0116, 1.0 / 448.0, 3.7, 0.0123291015625, 0.21875]

_F16 = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
_F16_FINITE = _F16[np.isfinite(_F16)]


def _torch_quantize(x16, scale):
    q = torch.from_numpy(x16.astype(np.float32)) / torch.tensor(scale, dtype=torch.float32)
    q = torch.clamp(q, -448.0, 448.0)  # the library cast maps overflow to NaN; the method saturates
    return q.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@pytest.mark.parametrize("scale", SCALES)
def test_quantize_exhaustive_fp16_vs_torch(scale):
    scale = float(np.float32(scale))
    ours = oracle.quantize(_F16_FINITE, scale)
    ref = _torch_quantize(_F16_FINITE, scale)
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, [(float(_F16_FINITE[i]), hex(ours[i]), hex(ref[i])) for i in bad[:8]]


@pytest.mark.parametrize("scale", [1.0, 0.0116, 3.7])
def test_quantize_exhaustive_fp16_vs_ml_dtypes(scale):
    ml_dtypes = pytest.importorskip("ml_dtypes")
    scale = float(np.float32(scale))
    q = np.clip(_F16_FINITE.astype(np.float32) / np.float32(scale), -448.0, 448.0)
    ref = q.astype(ml_dtypes.float8_e4m3fn).view(np.uint8)
    assert (oracle.quantize(_F16_FINITE, scale) == ref).all()


def _positive_values():
    """Exact rational values of the 127 non-negative finite E4M3 codes 0x00..0x7E."""
    vals = []
    for c in range(0x7F):
        e, m = (c >> 3) & 15, c & 7
        if e == 0:
            vals.append(fractions.Fraction(m, 512))
        else:
            vals.append((1 + fractions.Fraction(m, 8)) * fractions.Fraction(2) ** (e - 7))
    return vals


_POS = _positive_values()


def _brute_force_encode(v32):
    """Nearest E4M3 value by exact rational search; ties to the even code;
    |v| >= 448 saturates; the sign is kept (also for zero)."""
    v = float(v32)
    neg = math.copysign(1.0, v) < 0
    a = fractions.Fraction(abs(v))
    if a >= 448:
        code = 0x7E
    else:
        best = None
        for c, val in enumerate(_POS):
            d = abs(val - a)
            if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
                best = (d, c)
        code = best[1]
    return code | (0x80 if neg else 0)


def test_encode_brute_force_random_f32():
    rng = np.random.default_rng(1234)
    # values spread over every binade that matters, including subnormal E4M3 and overflow
    mags = np.exp2(rng.uniform(-14.0, 10.0, size=4000)).astype(np.float32)
    signs = np.where(rng.random(4000) < 0.5, -1.0, 1.0).astype(np.float32)
    vals = mags * signs
    # add every exact midpoint between adjacent codes (tie cases) and both neighbours
    mids = []
    for lo, hi in zip(_POS[:-1], _POS[1:]):
        mid = float((lo + hi) / 2)
        mids += [mid, float(np.nextafter(np.float32(mid), np.float32(0))),
                 float(np.nextafter(np.float32(mid), np.float32(1e9)))]
    vals = np.concatenate([vals, np.array(mids, np.float32), -np.array(mids, np.float32)])
    for v in vals:
        assert oracle.e4m3_encode_f32(float(v)) == _brute_force_encode(v), float(v)


def test_encode_ties_and_special_cases():
    enc = oracle.e4m3_encode_f32
    assert enc(1.0 + 1.0 / 16) == 0x38        # tie between 1.0 (even) and 1.125
    assert enc(1.0 + 3.0 / 16) == 0x3A        # tie between 1.125 and 1.25 (even)
    assert enc(2.0 ** -10) == 0x00            # half of the smallest subnormal -> 0
    assert enc(3 * 2.0 ** -10) == 0x02        # 1.5 units -> 2 (even)
    assert enc(-0.0) == 0x80 and enc(0.0) == 0x00
    assert enc(-(2.0 ** -11)) == 0x80         # negative values rounding to zero keep the sign
    assert enc(2.0 ** -6) == 0x08 and enc(2.0 ** -9) == 0x01
    assert enc(15 * 2.0 ** -10) == 0x08       # 7.5 units: tie, rounds up to 8 = the smallest normal
    assert enc(13 * 2.0 ** -10) == 0x06       # 6.5 units: tie, rounds down to 6 (even)
    for v in (448.0, 449.0, 463.9, 464.0, 480.0, 1e4, 3.4e38, float("inf")):
        assert enc(v) == 0x7E and enc(-v) == 0xFE, v
    assert enc(float("nan")) & 0x7F == 0x7F   # NaN code


def test_round_trip_every_finite_code():
    for c in range(256):
        v = oracle.e4m3_decode(c)
        if math.isnan(v):
            continue
        assert oracle.e4m3_encode_f32(v) == c
        # power-of-two scales are exact in binary32 and keep the code
        for k in (-3, 2, 5):
            x = np.float32(v * 2.0 ** k)
            assert oracle.e4m3_encode_f32(float(x / np.float32(2.0 ** k))) == c


def test_encode_error_bound_and_monotone():
    x = _F16_FINITE.astype(np.float32)
    x = np.sort(x)
    codes = oracle.quantize(x.astype(np.float16), 1.0)
    dec = oracle.e4m3_decode_array(codes)
    a = np.abs(x.astype(np.float64))
    inside = a < 448.0
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    bound = np.where(a >= 2.0 ** -6, 2.0 ** (e - 4), 2.0 ** -10)
    assert (np.abs(dec[inside] - x[inside]) <= bound[inside]).all()
    assert (dec[~inside] == np.sign(x[~inside]) * 448.0).all()
    assert (np.diff(dec) >= 0).all()          # encode is monotone non-decreasing


# ---------------------------------------------------------------------------
# calibration and the scale gate

def test_calibration_known_amax():
    rng = np.random.default_rng(7)
    x = rng.standard_normal(4096).astype(np.float16)
    x[1234] = np.float16(-56.0)                # amax = 56 = 448 / 8
    assert oracle.calibrate_scale(x) == 0.125
    x[77] = np.float16(448.0 * 2 ** -12)        # does not change amax
    assert oracle.calibrate_scale(x) == 0.125


def test_calibrated_scale_maps_amax_to_448():
    rng = np.random.default_rng(8)
    for _ in range(20):
        x = (rng.standard_normal(2048) * rng.uniform(0.01, 30)).astype(np.float16)
        s = oracle.calibrate_scale(x)
        assert s > 0 and np.isfinite(s)
        codes = oracle.quantize(x, s)
        dec = np.abs(oracle.e4m3_decode_array(codes))
        # the element at amax lands on (or next to) 448; nothing else saturates above it
        assert dec.max() == 448.0 or abs(dec.max() - 448.0) <= 32.0
        assert dec.max() <= 448.0


def test_calibration_rejects_degenerate_input():
    assert oracle.calibrate_scale(np.zeros(16, np.float16)) == 0.0
    x = np.ones(16, np.float16)
    x[3] = np.float16(np.inf)
    assert oracle.calibrate_scale(x) == 0.0


def test_scale_gate():
    ok = np.full(24, 0.01, np.float32)
    assert oracle.count_bad_scales(ok, ok) == 0
    for bad in (0.0, -1.0, np.nan, np.inf, -np.inf):
        k = ok.copy()
        k[5] = bad
        assert oracle.count_bad_scales(k, ok) == 1
        assert oracle.count_bad_scales(ok, k) == 1
    assert oracle.count_bad_scales(ok[:23], ok) == -1   # a missing entry
