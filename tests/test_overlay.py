"""The revision-bound scale overlay fails closed (CPU: the file logic; GPU:
materialising from calibration draws through the library)."""
import json
import math

import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_e4m3_gb300 import inputs, overlay


def _write(path, revision="rev-abc", n=24, mutate=None):
    layers = []
    for i in range(n):
        ks = float(np.float32(0.01 + i * 1e-4))
        vs = float(np.float32(0.02 + i * 1e-4))
        layers.append({"layer": i, "k_scale_bits": overlay._bits(ks), "v_scale_bits": overlay._bits(vs),
                       "k_scale": ks, "v_scale": vs})
    doc = {"format": overlay.FORMAT, "version": 1, "checkpoint_revision": revision,
           "num_layers": n, "layers": layers}
    if mutate:
        mutate(doc)
    path.write_text(json.dumps(doc))
    return str(path)


def test_round_trip(tmp_path):
    p = _write(tmp_path / "o.json")
    k, v = overlay.load(p, "rev-abc", 24, validate=lambda a, b: None)
    assert len(k) == len(v) == 24
    assert k[3] == float(np.float32(0.01 + 3e-4))


@pytest.mark.parametrize("case", [
    "missing", "revision", "count", "drop_layer", "dup_layer", "zero", "negative", "nan", "inf",
    "bits_mismatch", "format", "garbage"])
def test_refusals(tmp_path, case):
    def drop(d): d["layers"].pop(5)
    def dup(d): d["layers"][6]["layer"] = 5
    def setbits(val):
        def f(d):
            d["layers"][2]["k_scale_bits"] = val
            d["layers"][2].pop("k_scale")
        return f
    def mism(d): d["layers"][1]["v_scale"] = 0.5
    def fmt(d): d["format"] = "something-else"
    muts = {"drop_layer": drop, "dup_layer": dup, "zero": setbits("0x00000000"),
            "negative": setbits(overlay._bits(-0.01)), "nan": setbits("0x7fc00000"),
            "inf": setbits("0x7f800000"), "bits_mismatch": mism, "format": fmt}
    path = tmp_path / "o.json"
    if case == "missing":
        p = str(tmp_path / "absent.json")
    elif case == "garbage":
        path.write_text("{not json")
        p = str(path)
    else:
        p = _write(path, mutate=muts.get(case))
    rev = "rev-other" if case == "revision" else "rev-abc"
    n = 23 if case == "count" else 24
    with pytest.raises(overlay.OverlayError):
        overlay.load(p, rev, n, validate=lambda a, b: None)


@pytest.mark.gpu
def test_materialize_matches_oracle_calibration(tmp_path):
    w = inputs.get("verify")
    draws = [(inputs.calibration_draw(w, l, "k", device="cuda"),
              inputs.calibration_draw(w, l, "v", device="cuda")) for l in range(3)]
    p = str(tmp_path / "overlay.json")
    overlay.materialize(p, "rev-1", draws)
    k, v = overlay.load(p, "rev-1", 3)
    for l, (kd, vd) in enumerate(draws):
        assert k[l] == oracle.calibrate_scale(kd.cpu().numpy())
        assert v[l] == oracle.calibrate_scale(vd.cpu().numpy())
    with pytest.raises(overlay.OverlayError):
        overlay.load(p, "rev-2", 3)
    with pytest.raises(overlay.OverlayError):
        overlay.materialize(str(tmp_path / "bad.json"), "rev-1",
                            [(torch.zeros(64, dtype=torch.float16, device="cuda"),) * 2])
