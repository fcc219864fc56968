"""Storage formats read and written by the decode step, decoded to / encoded from
exact float64 values.

Test infrastructure only (see the package docstring).

* BF16: IEEE-754 binary32 with the low 16 mantissa bits dropped (1 sign bit,
  8 exponent bits, 7 stored mantissa bits).
* FP8-e4m3 ("FP8 Formats for Deep Learning", the e4m3 variant that the
  reference list of "Kernel Fusion for Large-Scale LLM Inference" cites):
  1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0
  encodes subnormals m/8 * 2^-6; there are no infinities; S.1111.111 is NaN, so
  the largest finite magnitude is 1.75 * 2^8 = 448.

Both encoders round to nearest with ties to even, written from the definition
of the value grid (quantum of the binade), not from any bit-twiddling recipe.
The e4m3 encoder saturates to +-448 ("satfinite").
"""
from __future__ import annotations

import numpy as np

__all__ = ["bf16_decode", "round_bf16", "e4m3_decode", "E4M3_VALUES", "round_e4m3",
           "E4M3_MAX"]

E4M3_MAX = 448.0


def bf16_decode(bits: np.ndarray) -> np.ndarray:
    """uint16 BF16 bit patterns -> exact float64 values."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):          # NaN patterns stay NaN
        return b.view(np.float32).astype(np.float64)


def _round_to_grid(x: np.ndarray, sig_bits: int, min_exp: int) -> np.ndarray:
    """Round float64 values to the nearest number with `sig_bits` significant
    bits (ties to even), with the quantum floored at 2^(min_exp - sig_bits + 1)
    (the subnormal spacing)."""
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                        # x = m * 2^e, 0.5 <= |m| < 1
    e = np.maximum(e - 1, min_exp)            # exponent of the leading bit
    quantum = np.ldexp(1.0, e - (sig_bits - 1))
    return np.rint(x / quantum) * quantum     # x / quantum exact; rint = ties-to-even


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float64 -> uint16 BF16 bits, round to nearest even (single rounding)."""
    x = np.asarray(x, dtype=np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("non-finite value")
    y = _round_to_grid(x, 8, -126)
    if np.any(np.abs(y) > np.float64(np.finfo(np.float32).max)):
        raise OverflowError("value beyond the BF16 range")
    # y has at most 8 significant bits, so it is exact in float32 with a zero low half.
    f = y.astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _e4m3_table() -> np.ndarray:
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        exp = (code >> 3) & 0xF
        man = code & 0x7
        if exp == 0xF and man == 0x7:
            vals[code] = np.nan
        elif exp == 0:
            vals[code] = sign * (man / 8.0) * 2.0 ** (1 - 7)
        else:
            vals[code] = sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)
    return vals


E4M3_VALUES = _e4m3_table()
_POS_VALUES = E4M3_VALUES[:0x7F]          # codes 0x00..0x7E, strictly increasing; 0x7F is NaN


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """uint8 e4m3 codes -> exact float64 values (NaN for the two NaN codes)."""
    return E4M3_VALUES[np.asarray(codes).astype(np.uint8)]


def round_e4m3(x: np.ndarray) -> np.ndarray:
    """float64 -> uint8 e4m3 codes, round to nearest even, saturating at +-448."""
    x = np.asarray(x, dtype=np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("non-finite value")
    y = _round_to_grid(x, 4, -6)
    y = np.clip(y, -E4M3_MAX, E4M3_MAX)
    mag = np.abs(y)
    codes = np.searchsorted(_POS_VALUES, mag)
    if not np.array_equal(_POS_VALUES[np.minimum(codes, 0x7E)], mag):
        raise AssertionError("rounded value is not on the e4m3 grid")
    codes = np.where(np.signbit(y), codes | 0x80, codes)     # keeps the sign of zero
    return codes.astype(np.uint8)
