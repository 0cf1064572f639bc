"""FP4 E2M1 and FP8 E4M3 number formats (oracle side).

The pages fix the storage formats by name only: main KV in FP4 E2M1 with one
E4M3 scale per 16 channels, SWA KV in FP8 (trawling.dev "DeepSeek-V4.1-Flash
공개", section "CSA2와 FP4 KV 캐싱"; origotech.dev deep dive, subsection
"FP4와 SWA Bounded Replay").  The value sets below are the public OCP
Microscaling / OFP8 definitions:

* E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; exponent 0 is
  subnormal (0 or 0.5).  Magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
* E4M3 ("FN" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits;
  exponent 0 is subnormal (m * 2^-9); S.1111.111 is NaN; no infinities;
  largest finite 448.

Encoders round to nearest, ties to the even code, and saturate to the
largest finite magnitude.  The sign bit is copied from the input, so a
negative input that rounds to zero keeps its sign bit.
"""
from __future__ import annotations

import numpy as np


def e2m1_value(code: int) -> float:
    """Value of one 4-bit E2M1 code, from its bit fields."""
    sign = -1.0 if (code >> 3) & 1 else 1.0
    e = (code >> 1) & 3
    m = code & 1
    mag = 0.5 * m if e == 0 else (2.0 ** (e - 1)) * (1.0 + 0.5 * m)
    return sign * mag


def e4m3_value(code: int) -> float:
    """Value of one 8-bit E4M3 code, from its bit fields (NaN for S.1111.111)."""
    sign = -1.0 if (code >> 7) & 1 else 1.0
    e = (code >> 3) & 15
    m = code & 7
    if e == 15 and m == 7:
        return float("nan")
    mag = m * 2.0 ** -9 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return sign * mag


E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
E4M3_MAX = 448.0
# non-negative finite E4M3 magnitudes, codes 0x00..0x7E, strictly increasing
_E4M3_POS = E4M3_TABLE[:127]


def e4m3_encode(x) -> np.ndarray:
    """Round to nearest E4M3 (ties to even code), saturating at 448.

    ``x`` must hold exact values (float32 values, or float64 values that the
    caller guarantees exact); the distances below are exact in float64.
    """
    x = np.asarray(x, dtype=np.float64)
    if np.isnan(x).any():
        raise ValueError("NaN input")
    sign = np.signbit(x)
    a = np.abs(x)
    hi = np.searchsorted(_E4M3_POS, a, side="left")          # _POS[hi-1] < a <= _POS[hi]
    hi = np.minimum(hi, 126)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _E4M3_POS[lo]
    d_hi = _E4M3_POS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a >= _E4M3_POS[126], 126, code)           # saturate
    code = np.where(a <= 0.0, 0, code)
    return (code | np.where(sign, 0x80, 0)).astype(np.uint8)


def e4m3_decode(codes) -> np.ndarray:
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


# Midpoints between consecutive E2M1 magnitudes, in units of the scale, and the
# code chosen at each exact midpoint (the one with an even mantissa bit).
E2M1_MIDPOINTS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def e2m1_code_of_magnitude(mag: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Magnitude code (0..7) of |r| on the grid {0, .5, 1, 1.5, 2, 3, 4, 6} * s.

    Decided by exact comparison of |r| against the midpoints * s (products
    of an E4M3 value and a 3-bit constant are exact).  Below a midpoint goes
    down, above goes up, exactly on it goes to the even code; beyond 5 s the
    code saturates at 6 (code 7).
    """
    mag = np.asarray(mag, dtype=np.float64)
    s = np.asarray(s, dtype=np.float64)
    m = [t * s for t in E2M1_MIDPOINTS]
    code = np.full(np.broadcast(mag, s).shape, 7, dtype=np.uint8)
    # walk the grid from the top down; each test is exact
    code = np.where(mag <= m[6], 6, code)   # tie at 5 s -> 4 (code 6, even)
    code = np.where(mag < m[5], 5, code)    # tie at 3.5 s -> 4 (code 6)
    code = np.where(mag <= m[4], 4, code)   # tie at 2.5 s -> 2 (code 4)
    code = np.where(mag < m[3], 3, code)    # tie at 1.75 s -> 2 (code 4)
    code = np.where(mag <= m[2], 2, code)   # tie at 1.25 s -> 1 (code 2)
    code = np.where(mag < m[1], 1, code)    # tie at 0.75 s -> 1 (code 2)
    code = np.where(mag <= m[0], 0, code)   # tie at 0.25 s -> 0 (code 0)
    code = np.where(s == 0.0, 0, code)
    return code.astype(np.uint8)
