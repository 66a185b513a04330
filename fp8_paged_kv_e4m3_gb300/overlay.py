"""Revision-bound calibrated scale overlay: materialise and load, failing closed.

PR "[Model][SM70][FP8] Integrate calibrated E4M3 QSA KV capacity path",
sections Changes and Validation boundary: the E4M3 capacity mode needs a
finite, positive K scale and V scale for each layer (24 of 24 on the pages'
model), computed offline by calibration and tied to one checkpoint revision;
without a complete overlay the mode does not start, and a default scale
(such as 1) never stands in for a missing one.  PR
"[Model][SM70] Calibrated E4M3 KV cache for Qwen4Exp QSA with MTP", section
Status and history: the materialiser is revision-checked.

File format (JSON, one object):
    {"format": "kvq-scale-overlay", "version": 1,
     "checkpoint_revision": "<revision string>", "num_layers": N,
     "layers": [{"layer": i, "k_scale_bits": "0x........", "v_scale_bits": "0x........",
                 "k_scale": <decimal, informative>, "v_scale": <decimal, informative>,
                 "k_amax": <float>, "v_amax": <float>}, ...]}
The scales are stored as their exact binary32 bit patterns; the decimals are
for people and must agree with the bits.

Calibration runs on the GPU through the library (amax reduction, then
amax / 448 in binary32); loading is host-only.
"""
from __future__ import annotations

import json
import math
import os
import struct
from typing import Callable, Iterable, Sequence, Tuple

FORMAT = "kvq-scale-overlay"
VERSION = 1


class OverlayError(ValueError):
    """The overlay cannot be used; the caller must refuse to start."""


def _bits(x: float) -> str:
    return "0x%08x" % struct.unpack("<I", struct.pack("<f", x))[0]


def _from_bits(s: str) -> float:
    if not isinstance(s, str) or not s.startswith("0x") or len(s) != 10:
        raise OverlayError(f"malformed scale bits {s!r}")
    try:
        return struct.unpack("<f", struct.pack("<I", int(s, 16)))[0]
    except ValueError as e:
        raise OverlayError(f"malformed scale bits {s!r}") from e


def _good(x: float) -> bool:
    return math.isfinite(x) and x > 0.0


def materialize(path: str, checkpoint_revision: str,
                calibration: Iterable[Tuple["object", "object"]]) -> None:
    """Calibrate every layer and write the overlay.

    calibration yields, per layer in order, (k_draw, v_draw): fp16 CUDA
    tensors of a calibration pass.  Refuses to write an overlay with any
    invalid scale (e.g. an all-zero draw)."""
    from . import kvq
    if not checkpoint_revision:
        raise OverlayError("a checkpoint revision is required")
    layers = []
    for i, (k_draw, v_draw) in enumerate(calibration):
        ka = float(kvq.amax_f16(k_draw).item())
        va = float(kvq.amax_f16(v_draw).item())
        ks, vs = kvq.scale_from_amax(ka), kvq.scale_from_amax(va)
        if not (_good(ks) and _good(vs)):
            raise OverlayError(f"layer {i}: calibration gave no valid scale (amax {ka}, {va})")
        layers.append({"layer": i, "k_scale_bits": _bits(ks), "v_scale_bits": _bits(vs),
                       "k_scale": ks, "v_scale": vs, "k_amax": ka, "v_amax": va})
    if not layers:
        raise OverlayError("no layers calibrated")
    doc = {"format": FORMAT, "version": VERSION, "checkpoint_revision": checkpoint_revision,
           "num_layers": len(layers), "layers": layers}
    tmp = path + ".tmp"
    with open(tmp, "w") as f:
        json.dump(doc, f, indent=1)
    os.replace(tmp, path)


def load(path: str, checkpoint_revision: str, num_layers: int,
         validate: Callable[[Sequence[float], Sequence[float]], None] = None):
    """Return (k_scales, v_scales) for layers 0..num_layers-1, or raise OverlayError.

    Refused: a missing or unreadable file, another format or version, a
    revision other than `checkpoint_revision`, a layer count other than
    `num_layers`, a missing or duplicated layer, bits that disagree with the
    stored decimal, and any scale that is not finite and > 0.  `validate`
    (default: the library's kvq_validate_scales when available) runs last."""
    if not os.path.exists(path):
        raise OverlayError(f"scale overlay {path} is missing")
    try:
        with open(path) as f:
            doc = json.load(f)
    except (OSError, json.JSONDecodeError) as e:
        raise OverlayError(f"scale overlay {path} is unreadable: {e}") from e
    if not isinstance(doc, dict) or doc.get("format") != FORMAT or doc.get("version") != VERSION:
        raise OverlayError("not a kvq scale overlay of a supported version")
    if doc.get("checkpoint_revision") != checkpoint_revision:
        raise OverlayError(f"overlay is for revision {doc.get('checkpoint_revision')!r}, "
                           f"checkpoint is {checkpoint_revision!r}")
    if doc.get("num_layers") != num_layers:
        raise OverlayError(f"overlay has {doc.get('num_layers')} layers, model has {num_layers}")
    entries = doc.get("layers")
    if not isinstance(entries, list):
        raise OverlayError("overlay has no layer list")
    k = [None] * num_layers
    v = [None] * num_layers
    for e in entries:
        i = e.get("layer") if isinstance(e, dict) else None
        if not isinstance(i, int) or not 0 <= i < num_layers:
            raise OverlayError(f"bad layer entry {e!r}")
        if k[i] is not None:
            raise OverlayError(f"layer {i} appears twice")
        ks, vs = _from_bits(e.get("k_scale_bits")), _from_bits(e.get("v_scale_bits"))
        for name, val in (("k_scale", ks), ("v_scale", vs)):
            if not _good(val):
                raise OverlayError(f"layer {i}: {name} {val} is not finite and positive")
            dec = e.get(name)
            if dec is not None and (not isinstance(dec, (int, float)) or
                                    struct.pack("<f", float(dec)) != struct.pack("<f", val)):
                raise OverlayError(f"layer {i}: {name} decimal {dec!r} disagrees with its bits")
        k[i], v[i] = ks, vs
    missing = [i for i in range(num_layers) if k[i] is None]
    if missing:
        raise OverlayError(f"overlay is incomplete: layers {missing} have no scales")
    if validate is None:
        try:
            from . import kvq
            validate = kvq.validate_scales
            kvq.load()
        except Exception:
            validate = None
    if validate is not None:
        validate(k, v)
    return k, v
