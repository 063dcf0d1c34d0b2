"""Oracle FP8 E4M3 codec, written from the OCP 8-bit floating point format.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The "ToPG framework" page (section 3.3 tuning YAML) stores the KV cache
"compressed" as FP8; the "LLM inference tutorial" (section 3.1) gives the
symmetric per-channel rule ``scale = absmax / qmax``, ``q = round(x / scale)``,
``x' = q * scale``.  With E4M3 as the 8-bit type, qmax is its largest finite
value.  The format (OCP OFP8, E4M3 variant):

* 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits;
* exponent field 0 holds subnormals ``m/8 * 2**-6`` (smallest 2**-9);
* exponent fields 1..15 hold normals ``(1 + m/8) * 2**(e-7)``;
* there are no infinities; ``S.1111.111`` is NaN, so the largest finite value
  is ``1.75 * 2**8 = 448``.

Encoding rounds to nearest, ties to even, and saturates: every finite value
(and infinity) beyond 448 in magnitude becomes +-448; NaN stays NaN.
"""
from __future__ import annotations

import math

import numpy as np

E4M3_MAX = 448.0


def decode_code(code: int) -> float:
    """Value of one E4M3 code as a Python float (exact)."""
    code &= 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


# The 127 non-negative finite magnitudes, ascending with their code.
_POS_CODES = list(range(0x00, 0x7F))
_POS_VALUES = [decode_code(c) for c in _POS_CODES]


def _round_magnitude(a: float) -> float:
    """Round a finite non-negative magnitude to the E4M3 grid (RNE, saturating)."""
    if a >= E4M3_MAX:
        return E4M3_MAX
    if a == 0.0:
        return 0.0
    e = math.floor(math.log2(a))
    # guard against log2 rounding at exact powers of two
    if 2.0 ** e > a:
        e -= 1
    elif 2.0 ** (e + 1) <= a:
        e += 1
    quantum = 2.0 ** (max(e, -6) - 3)          # spacing of the grid near a
    q = a / quantum                             # exact: quantum is a power of 2
    lo = math.floor(q)
    frac = q - lo
    if frac > 0.5 or (frac == 0.5 and lo % 2 == 1):
        lo += 1
    r = lo * quantum
    return min(r, E4M3_MAX)


def encode_value(x: float) -> int:
    """E4M3 code of a real value: round to nearest even, saturate to +-448."""
    if math.isnan(x):
        return 0x7F
    sign = 0x80 if math.copysign(1.0, x) < 0 else 0x00
    a = abs(x)
    r = E4M3_MAX if math.isinf(a) else _round_magnitude(a)
    idx = _POS_VALUES.index(r)
    return sign | _POS_CODES[idx]


_DECODE_TABLE = np.array([decode_code(c) for c in range(256)], dtype=np.float64)


def decode(codes: np.ndarray) -> np.ndarray:
    """Vectorised decode of uint8 codes to float64."""
    return _DECODE_TABLE[np.asarray(codes, dtype=np.uint8)]


def encode_f32(x: np.ndarray) -> np.ndarray:
    """Vectorised ``encode_value`` over a float32 array.

    Same rule as ``encode_value``: the grid spacing near ``|x|`` is
    ``2**(max(floor(log2|x|), -6) - 3)``; ``np.rint`` rounds the exact quotient
    ``|x| / spacing`` half-to-even; magnitudes at or above 448 (and infinity)
    saturate to 448; NaN encodes as 0x7F.
    """
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x.astype(np.float64))
    nan = np.isnan(a)
    a_safe = np.where(nan | np.isinf(a), 0.0, a)
    _, ex = np.frexp(a_safe)                       # a = f * 2**ex, f in [0.5, 1)
    e = np.where(a_safe > 0, ex - 1, -6)
    quantum = np.ldexp(1.0, np.maximum(e, -6) - 3)
    r = np.rint(a_safe / quantum) * quantum
    r = np.where(a >= E4M3_MAX, E4M3_MAX, np.minimum(r, E4M3_MAX))
    r = np.where(nan, 0.0, r)
    mag = np.searchsorted(np.asarray(_POS_VALUES), r).astype(np.uint8)
    sign = np.where(np.signbit(x), 0x80, 0x00).astype(np.uint8)
    out = (mag | sign).astype(np.uint8)
    out[nan] = 0x7F
    return out
