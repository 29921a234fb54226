"""bfloat16 as numpy ``uint16`` bit patterns (oracle; test infrastructure only).

bfloat16 is IEEE-754 binary32 with the low 16 bits of the significand
dropped: 1 sign bit, 8 exponent bits (bias 127), 7 stored significand bits.
The pages store every tensor of the bf16 workloads in this format; they do
not say how values are rounded into it, so the oracle takes the IEEE default,
round-to-nearest, ties-to-even, applied ONCE to the exact value.

Rounding is written from that definition rather than from bit tricks: the
value is split into a significand and a power of two, scaled so that one unit
in the last bf16 place is 1, rounded half-to-even with ``numpy.rint`` and
scaled back.  All scalings are by powers of two, so they are exact in fp64.
"""
from __future__ import annotations

import numpy as np

# Smallest normal bf16 exponent (same as binary32): values below 2**-126 are
# subnormal and share the fixed spacing 2**(-126-7) = 2**-133.
_EMIN = -126
_PREC = 8  # significand bits including the implicit leading one
_MAX_FINITE = float.fromhex("0x1.fep127")  # (2 - 2**-7) * 2**127


def widen(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact: bf16 is a prefix of binary32)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def widen64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 values (exact)."""
    return widen(bits).astype(np.float64)


def round_rne(values: np.ndarray) -> np.ndarray:
    """Round real values (float32 or float64 array) to bf16, nearest-even.

    Returns uint16 bit patterns.  One rounding from the given value: an fp64
    input is NOT first rounded to fp32.  Overflow past the largest finite
    bf16 gives +-inf, as IEEE round-to-nearest does.  NaN maps to the quiet
    NaN 0x7FC0 with the input's sign.
    """
    v = np.asarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.float64)
    finite = np.isfinite(v)
    fv = v[finite]
    # fv = m * 2**e with 0.5 <= |m| < 1, so the leading bit has weight 2**(e-1)
    # and the last of the 8 significand bits has weight 2**(e-1-7) = 2**(e-8).
    _, e = np.frexp(fv)
    e = np.maximum(e, _EMIN + 1)          # below the normal range the spacing is fixed
    ulp_exp = e - _PREC
    q = np.ldexp(fv, -ulp_exp)            # exact: power-of-two scaling
    r = np.rint(q)                        # round half to even
    rounded = np.ldexp(r, ulp_exp)        # exact again
    rounded = np.where(np.abs(rounded) > _MAX_FINITE, np.copysign(np.inf, fv), rounded)
    out[finite] = rounded
    out[~finite] = v[~finite]
    f32 = out.astype(np.float32)          # exact: every bf16 value is a binary32 value
    bits = (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(v)
    if nan.any():
        sign = np.signbit(v[nan]).astype(np.uint16) << np.uint16(15)
        bits[nan] = np.uint16(0x7FC0) | sign
    return bits


def from_float(values: np.ndarray) -> np.ndarray:
    """Alias of :func:`round_rne` for readability at call sites."""
    return round_rne(values)
