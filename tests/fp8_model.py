"""Numpy model of round-to-nearest-even into the OCP FP8 formats (e4m3:
bias 7, 3 mantissa bits, max 448; e5m2: bias 15, 2 mantissa bits), written
from the format definitions; used by the tests of the 8-bit operand path."""
import numpy as np


def round_fp8(y, mant_bits, emin, max_finite):
    """Round float64 values to the nearest representable FP8 value (ties to
    even), saturating at +-max_finite; emin is the smallest normal exponent."""
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, emin)  # subnormals share the quantum of the smallest normal
    q = np.exp2(e - mant_bits)
    r = np.round(a / q) * q  # numpy rounds half to even
    r = np.minimum(r, max_finite)
    return np.sign(y) * r


def e4m3(y):
    return round_fp8(y, 3, -6, 448.0)


def e5m2(y):
    return round_fp8(y, 2, -14, 57344.0)


def row_sigma(mx):
    """sigma = 2^(8 - e) with mx = f 2^e, f in [0.5, 1): mx sigma in [128, 256)
    (1 for a zero maximum)."""
    mx = np.asarray(mx, dtype=np.float64)
    _, e = np.frexp(np.where(mx > 0, mx, 1.0))
    return np.where(mx > 0, np.exp2(8.0 - e), 1.0)


def planes(y, n):
    """Split y into n e4m3 planes, each the rounding of what the earlier ones
    left; returns their sum."""
    out = np.zeros_like(y, dtype=np.float64)
    r = np.asarray(y, dtype=np.float64).copy()
    for _ in range(n):
        p = e4m3(r)
        out += p
        r -= p
    return out
