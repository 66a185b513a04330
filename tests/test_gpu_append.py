"""GPU parity of calibration and quantise-on-append against the oracle:
bit-exact bytes (and identical scales) on the same fp16 inputs."""
import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_e4m3_gb300 import build, kvq
from tests import _gpu as G
from tests import _problems as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    kvq.load()


ALL_F16 = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)


def _nan_code(c):
    return (c & 0x7F) == 0x7F


@pytest.mark.parametrize("scale", [1.0, 2.0 ** -3, 16.0, 0.0116, 1.0 / 448, 3.7, 0.0123291015625])
def test_quantize_every_fp16_pattern_bit_exact(scale):
    """All 65,536 binary16 patterns (both signs, subnormals, inf, NaN) through
    the append kernel: one token, 1 head, 65536 channels split as 512 x 128."""
    scale = float(np.float32(scale))
    x = ALL_F16.reshape(512, 1, 128)                 # 512 tokens, 1 head, D = 128
    slots = np.arange(512, dtype=np.int32)           # token t -> page t//4, slot t%4
    kc = torch.zeros((128, 1, 4, 128), dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    kvq.kv_append_e4m3(G.to_dev(x), G.to_dev(-x), G.to_dev(slots), kc, vc, scale, scale)
    got_k = kc.reshape(-1).cpu().numpy()
    got_v = vc.reshape(-1).cpu().numpy()
    ref_k = oracle.quantize(x.reshape(-1), scale)
    ref_v = oracle.quantize((-x).reshape(-1), scale)
    for got, ref in ((got_k, ref_k), (got_v, ref_v)):
        nan_ref = _nan_code(ref)
        assert (_nan_code(got) == nan_ref).all()          # NaN inputs give a NaN code
        mism = np.nonzero((got != ref) & ~nan_ref)[0]
        assert mism.size == 0, [(float(ALL_F16[i % 65536]), hex(got[i]), hex(ref[i])) for i in mism[:8]]


@pytest.mark.parametrize("name", ["tiny", "tiny_verify"])
def test_calibrated_scales_equal_oracle(name):
    pr = P.host_problem(name)
    ks = kvq.calibrate_scale(G.to_dev(pr.k_calib))
    vs = kvq.calibrate_scale(G.to_dev(pr.v_calib))
    assert (ks, vs) == P.oracle_scales(pr)


def test_amax_special_values():
    x = torch.randn(10_000, device="cuda").half()
    x[1234] = -300.0
    assert kvq.amax_f16(x).item() == 300.0
    x[77] = float("inf")
    assert kvq.amax_f16(x).item() == float("inf")
    x[78] = float("nan")
    assert np.isnan(kvq.amax_f16(x).item())
    assert kvq.scale_from_amax(float("nan")) == 0.0


@pytest.mark.parametrize("name", ["tiny", "tiny_verify"])
@pytest.mark.parametrize("e4m3", [True, False])
def test_pool_bit_exact_including_untouched_slots(name, e4m3):
    """The whole pool after history + step appends equals the oracle's pool
    byte for byte; slots no sequence owns keep the 0xCC sentinel."""
    pr = P.host_problem(name)
    dp = G.device_problem(pr, e4m3)
    kc_ref, vc_ref, _, _ = P.oracle_pools(pr, e4m3, (dp.k_scale, dp.v_scale) if e4m3 else None)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    got_k = dp.k_cache.cpu().numpy()
    got_v = dp.v_cache.cpu().numpy()
    if not e4m3:
        got_k, got_v = got_k.view(np.uint16), got_v.view(np.uint16)
        kc_ref, vc_ref = kc_ref.view(np.uint16), vc_ref.view(np.uint16)
    assert np.array_equal(got_k, kc_ref)
    assert np.array_equal(got_v, vc_ref)


def test_append_skips_negative_slots_and_flags_bad_ones():
    pr = P.host_problem("tiny")
    dp = G.device_problem(pr)
    before = dp.k_cache.clone()
    slots = pr.step_slots.copy()
    slots[0] = -1
    slots[1] = pr.P * 4 + 5
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    k = G.to_dev(pr.k_tok[pr.step_rows] * np.float16(0.5))
    kvq.kv_append_e4m3(k, k, G.to_dev(slots), dp.k_cache, dp.v_cache, dp.k_scale, dp.v_scale, err)
    torch.cuda.synchronize()
    assert err.item() & kvq.DEV_BAD_SLOT
    # the skipped tokens' slots are unchanged
    s0 = int(pr.step_slots[0])
    assert torch.equal(dp.k_cache[s0 // 4, :, s0 % 4], before[s0 // 4, :, s0 % 4])


def test_append_rejects_bad_scale_before_launch():
    kc = torch.zeros((4, 1, 4, 64), dtype=torch.uint8, device="cuda")
    x = torch.zeros((1, 1, 64), dtype=torch.float16, device="cuda")
    s = torch.zeros(1, dtype=torch.int32, device="cuda")
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(kvq.KvqError):
            kvq.kv_append_e4m3(x, x, s, kc, kc.clone(), bad, 1.0)
