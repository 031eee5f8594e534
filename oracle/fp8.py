"""FP8 E4M3 (the "fn" variant: no infinities, one NaN pattern per sign) decoded
from its definition, for the oracle.

TEST INFRASTRUCTURE ONLY (see oracle/gemm.py).

A byte s.eeee.mmm means (-1)^s · 2^(e-7) · (1 + m/8) for e in 1..15, and
(-1)^s · 2^-6 · (m/8) for e = 0 (subnormals); s.1111.111 is NaN.  The largest
finite value is 0.1111.110 = 448.  This is the OCP 8-bit floating point
format's E4M3 encoding; the pages use FP8 only as a tensor-core input type.
"""
from __future__ import annotations

import math

import numpy as np


def e4m3_decode(code: int) -> float:
    """Value of one E4M3 byte (a float, NaN for the NaN patterns)."""
    code &= 0xFF
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return s * math.ldexp(m / 8.0, -6)
    return s * math.ldexp(1.0 + m / 8.0, e - 7)


def e4m3_table() -> np.ndarray:
    """All 256 values, indexed by code, as float32 (every finite E4M3 value is
    exact in float32)."""
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float32)


_TABLE = None


def decode_codes(codes) -> np.ndarray:
    """float32 values of an array of E4M3 codes (uint8)."""
    global _TABLE
    if _TABLE is None:
        _TABLE = e4m3_table()
    return _TABLE[np.asarray(codes, dtype=np.uint8)]
