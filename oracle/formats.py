"""Number formats the operation consumes, decoded from their definitions.

Test infrastructure only (see the package docstring).

* e4m3 ("fp8 e4m3" on the aiter PR #5190 page, Motivation; "e4m3fn" on the
  aiter PR #7375 page, Summary): the OCP 8-bit floating-point E4M3 encoding.
  One sign bit, four exponent bits with bias 7, three mantissa bits.  Exponent
  field 0 encodes subnormals m/8 * 2^-6; there are no infinities; the codes
  S.1111.111 are NaN, so the largest finite magnitude is 1.75 * 2^8 = 448.
* bf16 (the query and output type on the same page): the upper 16 bits of an
  IEEE-754 binary32, so decoding is a 16-bit left shift.
"""
from __future__ import annotations

import math

import numpy as np


def e4m3_value(code: int) -> float:
    """Value of one e4m3 code, from the format definition."""
    code &= 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    exp_field = (code >> 3) & 0xF
    mant = code & 0x7
    if exp_field == 0xF and mant == 0x7:
        return math.nan
    if exp_field == 0:
        return sign * (mant / 8.0) * 2.0 ** (1 - 7)
    return sign * (1.0 + mant / 8.0) * 2.0 ** (exp_field - 7)


# Code -> float64 value for all 256 codes.
E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16 / int16) -> float64, by widening to binary32."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits): 2^(floor(log2|x|) - 7).

    Below the smallest normal (2^-126) the spacing is the subnormal step 2^-133.
    """
    ax = np.abs(np.asarray(x, dtype=np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.maximum(e, -126.0)
    return np.ldexp(1.0, (e - 7).astype(np.int64))
