"""Pins of the oracle's FP8 codecs (CPU only).

The codec is pinned against things other than itself: hand-derived anchors
(tests/golden/fp8_anchors.txt), an exhaustive nearest-value search over the
format's own 256 codes, and PyTorch's float8 casts (a library routine) for
in-range values.
"""

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import fp8

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fp8_anchors.txt")
FMTS = ["e4m3", "e5m2"]
TORCH_DT = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


def _rows(kind):
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0] == kind:
                yield parts[1:]


def test_golden_decode_anchors():
    n = 0
    for fmt, code, val in _rows("decode"):
        got = fp8.decode(np.array([int(code, 16)], np.uint8), fmt)[0]
        exp = float(val)
        if math.isnan(exp):
            assert math.isnan(got), (fmt, code)
        else:
            assert got == exp and math.copysign(1, got) == math.copysign(1, exp), (fmt, code, got, exp)
        n += 1
    assert n >= 25


def test_golden_encode_anchors():
    n = 0
    for fmt, val, code in _rows("encode"):
        got = int(fp8.encode(np.array([float(val)], np.float32), fmt)[0])
        assert got == int(code, 16), (fmt, val, hex(got), code)
        n += 1
    assert n >= 20


@pytest.mark.parametrize("fmt", FMTS)
def test_code_counts_and_order(fmt):
    t = fp8.decode_table(fmt)
    finite = np.isfinite(t)
    # E4M3fn: 2 NaN codes; E5M2: 2 infinities + 6 NaN codes
    assert finite.sum() == (254 if fmt == "e4m3" else 248)
    pos = t[:128][finite[:128]]
    assert np.all(np.diff(pos) > 0), "positive codes must increase with their value"
    assert np.array_equal(t[128:][finite[128:]], -pos)
    assert pos.max() == (448.0 if fmt == "e4m3" else 57344.0)


@pytest.mark.parametrize("fmt", FMTS)
def test_roundtrip_every_finite_code(fmt):
    t = fp8.decode_table(fmt)
    codes = np.array([c for c in range(256) if np.isfinite(t[c])], np.uint8)
    back = fp8.encode(t[codes].astype(np.float32), fmt)
    assert np.array_equal(back, codes)


def _nearest_even(y, fmt):
    """Exhaustive search: the finite code nearest to y, ties to the even code.

    Independent of ``fp8.encode``: it only uses the value table and compares
    distances in exact rational arithmetic.
    """
    t = fp8.decode_table(fmt)
    codes = [c for c in range(128) if np.isfinite(t[c])]
    a = Fraction(abs(float(y)))
    d = [abs(Fraction(float(t[c])) - a) for c in codes]
    dmin = min(d)
    best = [i for i, x in enumerate(d) if x == dmin]
    if len(best) > 1:
        best = [b for b in best if codes[b] % 2 == 0]
    c = codes[best[0]]
    if math.copysign(1.0, float(y)) < 0:
        c |= 0x80
    return c


def _midpoints(fmt):
    t = fp8.decode_table(fmt)
    pos = np.sort(t[:128][np.isfinite(t[:128])])
    mids = (pos[:-1] + pos[1:]) / 2.0
    mids = mids[mids == mids.astype(np.float32)]  # exact in float32 (all of them are)
    return np.concatenate([mids, -mids, pos, -pos])


@pytest.mark.parametrize("fmt", FMTS)
def test_encode_equals_exhaustive_nearest(fmt):
    rng = np.random.default_rng(7)
    fmax = 448.0 if fmt == "e4m3" else 57344.0
    smallest = 2.0 ** -9 if fmt == "e4m3" else 2.0 ** -16
    ys = np.concatenate([
        _midpoints(fmt),
        rng.standard_normal(2000) * fmax / 4,
        np.exp(rng.uniform(np.log(smallest / 8), np.log(fmax * 2), 3000)) * rng.choice([-1, 1], 3000),
        np.array([fmax * 1.01, fmax * 1.1, -fmax * 3, 1e30, -1e30]),
    ]).astype(np.float32)
    got = fp8.encode(ys, fmt)
    exp = np.array([_nearest_even(y, fmt) for y in ys], np.uint8)
    bad = np.flatnonzero(got != exp)
    assert bad.size == 0, [(float(ys[i]), hex(got[i]), hex(exp[i])) for i in bad[:5]]


@pytest.mark.parametrize("fmt", FMTS)
def test_encode_matches_torch_cast_in_range(fmt):
    rng = np.random.default_rng(11)
    fmax = 448.0 if fmt == "e4m3" else 57344.0
    ys = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * np.float32(fmax / 8),
        _midpoints(fmt).astype(np.float32),
        rng.uniform(-fmax, fmax, 100000).astype(np.float32),
    ])
    ys = ys[np.abs(ys) <= fmax]
    ref = torch.from_numpy(ys).to(TORCH_DT[fmt]).view(torch.uint8).numpy()
    got = fp8.encode(ys, fmt)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("fmt", FMTS)
def test_decode_matches_torch(fmt):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(TORCH_DT[fmt]).to(torch.float64).numpy()
    got = fp8.decode(np.arange(256, dtype=np.uint8), fmt)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(got)
    assert np.array_equal(got[ok], ref[ok])


@pytest.mark.parametrize("fmt", FMTS)
def test_decode_exact_in_fp16(fmt):
    """Every finite FP8 value is an fp16 value (the GPU dequantises to fp16)."""
    t = fp8.decode_table(fmt)
    f = t[np.isfinite(t)]
    assert np.array_equal(f.astype(np.float16).astype(np.float64), f)


FP8_MUTANTS = {
    "exponent bias off by one": ("2.0 ** (e - f.bias)", "2.0 ** (e - f.bias - 1)"),
    "ties away from zero": ("r = np.rint(a / quantum) * quantum", "r = np.floor(a / quantum + 0.5) * quantum"),
    "truncating rounding": ("r = np.rint(a / quantum) * quantum", "r = np.floor(a / quantum) * quantum"),
    "no saturation": ("r = np.minimum(r, f.max_finite)", "r = r"),
    "subnormals flushed": ("np.where(\n        a < f.min_normal, f.subnormal_step,", "np.where(\n        a < 0, f.subnormal_step,"),
    "sign of zero dropped": ("code = np.where(neg, code | 0x80, code)", "code = np.where(neg & (r > 0), code | 0x80, code)"),
}


def _fp8_mutant(old, new):
    import inspect
    import types
    src = inspect.getsource(fp8)
    assert src.count(old) == 1, old
    import sys
    mod = types.ModuleType("fp8_mutant")
    sys.modules["fp8_mutant"] = mod  # dataclasses look their module up here
    exec(compile(src.replace(old, new), "fp8_mutant", "exec"), mod.__dict__)
    return mod


def _codec_pins_pass(mod):
    global fp8
    saved = fp8
    fp8 = mod
    try:
        for test in (test_golden_decode_anchors, test_golden_encode_anchors):
            test()
        for fmt in FMTS:
            test_roundtrip_every_finite_code(fmt)
            test_encode_equals_exhaustive_nearest(fmt)
            test_encode_matches_torch_cast_in_range(fmt)
        return True
    except (AssertionError, Exception):
        return False
    finally:
        fp8 = saved


@pytest.mark.parametrize("name", list(FP8_MUTANTS))
def test_planted_codec_mistake_fails_a_pin(name):
    assert not _codec_pins_pass(_fp8_mutant(*FP8_MUTANTS[name])), name


def test_codec_pins_pass_unmutated():
    assert _codec_pins_pass(fp8)
