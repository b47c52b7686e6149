"""Bitwise FP8 codecs (E4M3 "fn" and E5M2), float64, written from the formats.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Source of the formats. The fork's pages name the two KV-cache formats
(``--kv-cache-dtype fp8_e5m2`` in "1Cat-vLLM", section "Optional experimental
feature: FP8 KV cache"; E4M3 as the qualified KV dtype in "SM70 release
profile and acceleration status", override table) but do not define them. The
definitions used here are the standard 8-bit floating-point layouts:

* E4M3 "fn": 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits. No
  infinities; the only NaN codes are S.1111.111; the largest finite value is
  S.1111.110 = 448. Exponent field 0 encodes subnormals m * 2**-9.
* E5M2: 1 sign bit, 5 exponent bits (bias 15), 2 mantissa bits. S.11111.00 is
  +-infinity, S.11111.{01,10,11} are NaN, the largest finite value is
  S.11110.11 = 57344. Exponent field 0 encodes subnormals m * 2**-16.

Encoding (the reading used for the KV write path): round to nearest, ties to
an even mantissa, including the subnormal range; results whose magnitude
exceeds the largest finite value (and infinities) saturate to it ("satfinite");
the sign of zero is kept (-0.0 -> 0x80).
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class FP8Format:
    name: str
    exp_bits: int
    man_bits: int
    bias: int
    ieee_inf: bool  # True: all-ones exponent is inf/NaN (E5M2); False: only S.1111.111 is NaN (E4M3fn)

    @property
    def max_finite(self) -> float:
        if self.ieee_inf:
            emax = (1 << self.exp_bits) - 2
            mant = (1 << self.man_bits) - 1
        else:
            emax = (1 << self.exp_bits) - 1
            mant = (1 << self.man_bits) - 2
        return (1.0 + mant / (1 << self.man_bits)) * 2.0 ** (emax - self.bias)

    @property
    def min_normal(self) -> float:
        return 2.0 ** (1 - self.bias)

    @property
    def subnormal_step(self) -> float:
        return 2.0 ** (1 - self.bias - self.man_bits)


E4M3 = FP8Format("e4m3fn", exp_bits=4, man_bits=3, bias=7, ieee_inf=False)
E5M2 = FP8Format("e5m2", exp_bits=5, man_bits=2, bias=15, ieee_inf=True)

FORMATS = {"e4m3": E4M3, "e5m2": E5M2}


def _fmt(fmt) -> FP8Format:
    return FORMATS[fmt] if isinstance(fmt, str) else fmt


def decode_code(code: int, fmt) -> float:
    """Value of one FP8 code, from its bit fields (exact in float64)."""
    f = _fmt(fmt)
    sign = -1.0 if (code >> 7) & 1 else 1.0
    e = (code >> f.man_bits) & ((1 << f.exp_bits) - 1)
    m = code & ((1 << f.man_bits) - 1)
    e_all_ones = (1 << f.exp_bits) - 1
    if f.ieee_inf and e == e_all_ones:
        return sign * np.inf if m == 0 else np.nan
    if (not f.ieee_inf) and e == e_all_ones and m == (1 << f.man_bits) - 1:
        return np.nan
    if e == 0:
        return sign * m * f.subnormal_step
    return sign * (1.0 + m / (1 << f.man_bits)) * 2.0 ** (e - f.bias)


def decode_table(fmt) -> np.ndarray:
    """float64[256]: the value of every code (NaN / inf where the format says so)."""
    return np.array([decode_code(c, fmt) for c in range(256)], dtype=np.float64)


_TABLES: dict[str, np.ndarray] = {}


def decode(codes: np.ndarray, fmt) -> np.ndarray:
    """Exact float64 values of an array of uint8 codes."""
    f = _fmt(fmt)
    if f.name not in _TABLES:
        _TABLES[f.name] = decode_table(f)
    return _TABLES[f.name][np.asarray(codes, dtype=np.uint8)]


def encode(y, fmt) -> np.ndarray:
    """uint8 codes of float32 values: round-to-nearest-even, satfinite, signed zero.

    Works from the magnitude: the quantum (spacing of representable values)
    at |y| is 2**(E - man_bits) for a normal binade with exponent E, and the
    subnormal step below the smallest normal. |y| / quantum is exact (a power
    of two scaling of a float32), so ``np.rint`` (round half to even) gives
    the nearest representable magnitude with the even-mantissa tie rule.
    """
    f = _fmt(fmt)
    y = np.asarray(y, dtype=np.float32)
    a = np.abs(y.astype(np.float64))
    neg = np.signbit(y)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)

    # exponent of the binade holding a (a = frac * 2**ex, frac in [0.5, 1))
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    binade = ex.astype(np.int64) - 1
    quantum = np.where(
        a < f.min_normal, f.subnormal_step, np.ldexp(1.0, binade - f.man_bits)
    )
    r = np.rint(a / quantum) * quantum
    r = np.minimum(r, f.max_finite)  # satfinite (covers +inf too)

    # bit fields of the rounded magnitude
    is_sub = r < f.min_normal
    _, rex = np.frexp(np.where(r > 0, r, 1.0))
    rbin = rex.astype(np.int64) - 1
    e_field = np.where(is_sub, 0, rbin + f.bias)
    m_norm = (r / np.ldexp(1.0, rbin) - 1.0) * (1 << f.man_bits)
    m_sub = r / f.subnormal_step
    m_field = np.where(is_sub, m_sub, m_norm)
    assert np.all(m_field == np.floor(m_field)), "mantissa not integral"
    code = (e_field << f.man_bits) | m_field.astype(np.int64)
    code = np.where(neg, code | 0x80, code)
    nan_code = 0x7F  # S.1111.111 (E4M3fn) and S.11111.11 (E5M2) are both NaN
    code = np.where(nan, nan_code, code)
    return code.astype(np.uint8)
