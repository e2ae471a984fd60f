"""Round-to-nearest-even from FP64 to FP16 and BF16 -- oracle, test infrastructure only.

The library casts its FP32 accumulators to the output type exactly once
(FalconGEMM write-up, numerics paragraph: the fused kernel keeps C in FP32 on
chip and casts back to the target precision only at the end).  The oracle
forms the same single rounding from the FP64 result.

One routine serves both formats.  A binary floating-point format with ``p``
significant bits and minimum normal exponent ``emin`` has, for a value whose
leading bit has weight ``2^e``, a unit in the last place of
``2^(max(e, emin) - p + 1)``; rounding is ``ulp * rint(x / ulp)`` with ties to
even (both scalings are exact powers of two).  Values whose rounded magnitude
exceeds the largest finite number become infinity.

* FP16 (IEEE 754 binary16): p = 11, emin = -14, emax = 15.
* BF16: p = 8, emin = -126, emax = 127 (the FP32 exponent range).

Pins: the FP16 instance is compared with numpy's float64 -> float16 cast and
the BF16 instance with torch's float32 -> bfloat16 cast, on random values and
on every tie, subnormal and overflow edge (``tests/test_oracle_rounding.py``).
"""
from __future__ import annotations

import numpy as np

F16 = 0
BF16 = 1

_FORMATS = {
    F16: (11, -14, 15),
    BF16: (8, -126, 127),
}


def rne_values(x, dtype: int) -> np.ndarray:
    """Round float64 values to the nearest ``dtype`` value (ties to even).

    Returns float64 values that are exactly representable in ``dtype``
    (or +-inf / nan).
    """
    p, emin, emax = _FORMATS[dtype]
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, dtype=np.float64, copy=True)
    fin = np.isfinite(x)
    ax = np.abs(x[fin])
    _, e = np.frexp(ax)              # ax = m * 2^e with 0.5 <= m < 1, so the leading bit is 2^(e-1)
    lead = np.maximum(e - 1, emin)   # below the normal range the ulp stays at 2^(emin-p+1)
    ulp_exp = lead - (p - 1)
    r = np.ldexp(np.rint(np.ldexp(ax, -ulp_exp)), ulp_exp)
    largest = np.ldexp(2.0 - 2.0 ** (1 - p), emax)
    r = np.where(r > largest, np.inf, r)
    out[fin] = np.copysign(r, x[fin])
    return out


def rne_bits(x, dtype: int) -> np.ndarray:
    """Round float64 values to ``dtype`` and return the uint16 bit patterns."""
    v = rne_values(x, dtype)
    if dtype == F16:
        return v.astype(np.float16).view(np.uint16)   # exact: v is representable
    b = v.astype(np.float32).view(np.uint32)          # exact: BF16 values are FP32 values
    b = np.where(np.isnan(v), np.uint32(0x7FC00000), b)
    return (b >> 16).astype(np.uint16)
