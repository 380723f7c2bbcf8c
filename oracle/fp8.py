"""The 8-bit floating-point format of an fp8 KV pool (E4M3, "FN" variant).

TEST INFRASTRUCTURE ONLY (see the package docstring). Written from the format
definition: one sign bit, four exponent bits with bias 7, three mantissa
bits; exponent field 0 holds the subnormals m/8 * 2^-6; there is no infinity,
and the all-ones pattern S.1111.111 is NaN, so the largest finite value is
1.75 * 2^8 = 448.

Encoding rounds to the nearest finite value, ties to the even mantissa, and
saturates at +-448 (the reading taken for values past the range); the sign of
a zero or of a value that rounds to zero is kept. NaN encodes as 0x7F.

Pinned by tests/test_oracle_fp8.py against torch's float8_e4m3fn conversions
and hand-worked values.
"""
from __future__ import annotations

import numpy as np

MAX_FINITE = 448.0


def decode_table() -> np.ndarray:
    """float64 value of each of the 256 codes (NaN for the two NaN codes)."""
    out = np.empty(256, np.float64)
    for code in range(256):
        s = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            out[code] = np.nan
        elif e == 0:
            out[code] = s * (m / 8.0) * 2.0 ** -6
        else:
            out[code] = s * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return out


_TABLE = decode_table()
_POS = _TABLE[:0x7F]  # codes 0x00 .. 0x7E: the non-negative finite values, increasing


def decode(codes: np.ndarray) -> np.ndarray:
    return _TABLE[np.asarray(codes, np.uint8)]


def encode(x: np.ndarray) -> np.ndarray:
    """float32 values -> uint8 codes (nearest, ties to even mantissa, saturating)."""
    x = np.asarray(x, np.float32)
    a = np.abs(x.astype(np.float64))
    neg = np.signbit(x)
    a = np.minimum(a, MAX_FINITE)
    hi = np.searchsorted(_POS, a, side="left")  # first value >= a
    hi = np.minimum(hi, len(_POS) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _POS[lo]
    d_hi = _POS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(a == _POS[hi], hi, code).astype(np.uint8)  # exact hits
    code = np.where(neg, code | 0x80, code).astype(np.uint8)
    code = np.where(np.isnan(x), 0x7F, code).astype(np.uint8)
    return code
