"""Bit-level decoders for the two storage formats the paged KV cache may use.

TEST INFRASTRUCTURE ONLY (see the package docstring).

* bf16: the upper 16 bits of an IEEE-754 binary32.  Decoding is exact: the
  16 bits are shifted into the high half of a 32-bit word and reinterpreted.
* FP8 E4M3 (the OCP 8-bit floating point "E4M3" encoding, the
  ``--kv-cache-dtype fp8_e4m3`` KV-cache format named in the
  model-serving-minefield issue 73 report, "What were you serving"):
  1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0
  encodes subnormals ``(-1)^s * 2^-6 * m/8``; the pattern S.1111.111 is NaN;
  there are no infinities; the largest finite magnitude is 448.

Both decoders are written from those definitions, element by element, with
no library conversion routine; the tests compare them against library casts.
The E4M3 encoder (used to quantise K/V rows appended to an FP8 cache) is
written from the same definition: nearest representable value, ties to the
even code, magnitudes beyond 448 saturated to 448.
"""

from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode raw bf16 storage (any integer dtype holding 16-bit patterns) to float64."""
    b = np.asarray(bits).astype(np.int64) & 0xFFFF
    word = (b << 16).astype(np.uint32)
    with np.errstate(invalid="ignore"):   # NaN payloads widen to NaN
        return word.view(np.float32).astype(np.float64)


def _e4m3_scalar(code: int) -> float:
    sign = -1.0 if (code >> 7) & 1 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return float("nan")
    if exp == 0:
        return sign * (2.0 ** -6) * (man / 8.0)
    return sign * (2.0 ** (exp - 7)) * (1.0 + man / 8.0)


# One value per byte code, built from the scalar definition above.
_E4M3_TABLE = np.array([_e4m3_scalar(c) for c in range(256)], dtype=np.float64)


def e4m3_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode raw FP8 E4M3 storage (uint8 codes) to float64."""
    codes = np.asarray(bits).astype(np.int64) & 0xFF
    return _E4M3_TABLE[codes]


# Non-negative finite E4M3 values in code order (codes 0x00 .. 0x7E); the
# order of the codes is the order of the values.
_E4M3_POS = _E4M3_TABLE[:0x7F]


def f64_to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Encode values as FP8 E4M3 codes (uint8).

    Round to the nearest representable value; a value exactly halfway
    between two takes the code whose mantissa is even (lowest bit 0);
    magnitudes above 448 saturate to +-448 (no infinities exist); NaN becomes
    the positive NaN code 0x7F.  The sign of zero is kept.
    """
    v = np.asarray(x, dtype=np.float64)
    flat = v.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint8)
    mag = np.abs(flat)
    sign = np.signbit(flat).astype(np.uint8) << 7
    nan = np.isnan(flat)
    m = np.where(nan, 0.0, np.minimum(mag, 448.0))
    hi = np.searchsorted(_E4M3_POS, m, side="left")   # first code with value >= m
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_hi = _E4M3_POS[hi] - m
    d_lo = m - _E4M3_POS[lo]
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    code = np.where(pick_lo, lo, hi).astype(np.uint8)
    out[:] = code | sign
    out[nan] = 0x7F
    return out.reshape(v.shape)
