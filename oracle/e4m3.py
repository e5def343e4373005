"""OCP 8-bit floating point, E4M3 variant: the byte format of the fp8 KV cache.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages name the fp8 KV cache ("vLLM 部署深度指南", 量化支持 table, FP8 row;
section FP8 部署, ``--kv-cache-dtype fp8``) but not its bit layout.  The layout
used is OCP OFP8 E4M3, restated here from its definition:

  * 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
  * exponent field 0 encodes subnormals ``(-1)^s * 2^-6 * (m / 8)``;
  * exponent fields 1..15 encode normals ``(-1)^s * 2^(e-7) * (1 + m/8)``,
    except ``e = 15, m = 7`` (codes 0x7F and 0xFF), which is NaN;
  * there are no infinities; the largest finite magnitude is 448 (code 0x7E).

Encoding (the write side of the fp8 cache) rounds to the nearest finite
value, ties to the code whose mantissa is even, and saturates magnitudes
above 448 to 448 (saturating conversion, the only one that keeps a
per-tensor-scaled cache finite).  NaN encodes to 0x7F; the sign of a NaN is
not fixed by the format, so callers compare NaN codes by their low 7 bits.
"""

import numpy as np

#: Largest finite E4M3 magnitude.
MAX_FINITE = 448.0

#: Canonical NaN code produced by :func:`encode`.
NAN_CODE = 0x7F


def _magnitude_of_code(code):
    """Value of the 7 low bits of an E4M3 code (sign cleared), as a Python float."""
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return (m / 8.0) * 2.0 ** (1 - 7)
    return (1.0 + m / 8.0) * 2.0 ** (e - 7)


#: ``DECODE_TABLE[c]`` is the float64 value of byte ``c``.
DECODE_TABLE = np.array(
    [(-1.0 if c & 0x80 else 1.0) * _magnitude_of_code(c & 0x7F) for c in range(256)],
    dtype=np.float64,
)

# The 127 finite non-negative magnitudes, in code order 0x00..0x7E.  Code order
# is value order for non-negative codes, which the nearest-value search uses.
_FINITE_MAGNITUDES = DECODE_TABLE[:0x7F].copy()


def decode(codes):
    """Map uint8 E4M3 codes to float64 values (exact)."""
    codes = np.asarray(codes, dtype=np.uint8)
    return DECODE_TABLE[codes]


def encode(x):
    """Encode real values to E4M3 codes: nearest finite value, ties to even, saturating.

    ``x`` is any float array; each element is taken exactly (float64 holds every
    float32).  Returns a uint8 array of the same shape.
    """
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(a)
    a_clean = np.where(nan, 0.0, a)

    # Index of the largest representable magnitude <= a, and its successor.
    lo = np.searchsorted(_FINITE_MAGNITUDES, a_clean, side="right") - 1
    lo = np.clip(lo, 0, 0x7E)
    hi = np.minimum(lo + 1, 0x7E)
    v_lo = _FINITE_MAGNITUDES[lo]
    v_hi = _FINITE_MAGNITUDES[hi]
    d_lo = a_clean - v_lo
    d_hi = v_hi - a_clean
    # Nearest; on a tie the even code (even mantissa) wins.
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0) & (hi != lo))
    mag_code = np.where(pick_hi, hi, lo)
    # Saturation: everything at or beyond the largest finite value (including +inf).
    mag_code = np.where(a_clean >= MAX_FINITE, 0x7E, mag_code)

    code = mag_code.astype(np.uint8) | np.where(sign, 0x80, 0x00).astype(np.uint8)
    code = np.where(nan, NAN_CODE, code).astype(np.uint8)
    return code


def is_nan_code(codes):
    """True where a code is an E4M3 NaN (either sign)."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes & 0x7F) == 0x7F
