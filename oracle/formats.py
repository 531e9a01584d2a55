"""Number formats, written from their definitions (test infrastructure only).

* fp8 E4M3 ("fn" variant, OCP 8-bit floating point spec): 1 sign bit, 4 exponent bits with
  bias 7, 3 mantissa bits; exponent field 0 encodes subnormals m/8 * 2^-6; the all-ones
  pattern S.1111.111 is NaN; there is no infinity; the largest finite value is 448.
  The per-token scales of the paged KV cache multiply these decoded values.
* bfloat16: the upper 16 bits of an IEEE-754 binary32, rounded to nearest, ties to even.
"""
from __future__ import annotations

import numpy as np


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """uint8 E4M3 codes -> float64 values (NaN for S.1111.111)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = (m / 8.0) * 2.0 ** -6
    val = np.where(e == 0, sub, normal)
    val = np.where((e == 0xF) & ((c & 0x7) == 0x7), np.nan, val)
    return sign * val


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (ties to even), returned as float64.

    Two steps, each exact-or-correctly-rounded: float64 -> float32 (round to nearest even)
    and then float32 -> bfloat16 by rounding the low 16 bits of the binary32 pattern to
    nearest even.  The double rounding can differ from a direct float64 -> bf16 rounding
    only for inputs within 2^-24 relative of a bf16 tie, which the callers never rely on.
    """
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    rounded = ((u + 0x7FFF + lsb) >> 16) << 16
    nan = np.isnan(f)
    rounded = np.where(nan, u, rounded)
    return rounded.astype(np.uint32).view(np.float32).astype(np.float64)
