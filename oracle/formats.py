"""Number formats of the MX family, restated from their bit fields.

Test infrastructure (see ``oracle/__init__``).  Every decode table is built
from the sign / exponent / mantissa field definitions, never from a cast
library, so that a cast library can serve as an independent check.

Sources:
* UE8M0 FP8 / MXFP8 explainer, section 1: E4M3 has a maximum of about
  1.75 * 2^8 and a minimum of about 2^-9 (about 17.8 binades) and a single NaN
  bit pattern; E5M2 follows IEEE-754 special values; the UE8M0 scale has
  8 exponent bits, no sign and no mantissa, and encodes 2^-127 .. 2^127 or NaN;
  MXFP4 elements are E2M1.
* Where the page only names a format (E2M1), the field layout follows from the
  name with the IEEE-style bias 2^(E-1) - 1 and no Inf/NaN codes: parity for
  E2M1 rests on that reading plus the invariants in the tests.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class ElemFormat:
    """An element format: 1 sign bit, ``ebits`` exponent bits, ``mbits``
    mantissa bits, exponent bias ``2^(ebits-1) - 1``.

    ``specials`` says how the all-ones exponent is used:
      * ``"fn"``   -- only the all-ones exponent with all-ones mantissa is NaN
                      (E4M3: a single NaN pattern, no infinities);
      * ``"ieee"`` -- all-ones exponent is Inf (mantissa 0) or NaN (E5M2);
      * ``"none"`` -- every code is a finite number (E2M1).
    """

    name: str
    code: int          # the library's enum value (0 E4M3, 1 E5M2, 2 E2M1)
    ebits: int
    mbits: int
    specials: str
    table: np.ndarray = field(init=False, repr=False, compare=False)

    def __post_init__(self):
        object.__setattr__(self, "table", _build_table(self))

    @property
    def nbits(self) -> int:
        return 1 + self.ebits + self.mbits

    @property
    def bias(self) -> int:
        return (1 << (self.ebits - 1)) - 1

    @property
    def ncodes(self) -> int:
        return 1 << self.nbits

    @property
    def max_finite(self) -> float:
        t = self.table
        return float(np.max(t[np.isfinite(t)]))

    @property
    def min_subnormal(self) -> float:
        t = self.table
        return float(np.min(t[np.isfinite(t) & (t > 0)]))


def _decode_code(f: ElemFormat, code: int) -> float:
    """Value of one code of format ``f`` from its bit fields."""
    sign = (code >> (f.ebits + f.mbits)) & 1
    exp = (code >> f.mbits) & ((1 << f.ebits) - 1)
    man = code & ((1 << f.mbits) - 1)
    emax_field = (1 << f.ebits) - 1
    mman = (1 << f.mbits) - 1
    if f.specials == "fn" and exp == emax_field and man == mman:
        return math.nan
    if f.specials == "ieee" and exp == emax_field:
        return (-math.inf if sign else math.inf) if man == 0 else math.nan
    if exp == 0:   # subnormal: 0.m * 2^(1 - bias)
        mag = math.ldexp(man, 1 - f.bias - f.mbits)
    else:          # normal: 1.m * 2^(exp - bias)
        mag = math.ldexp((1 << f.mbits) + man, exp - f.bias - f.mbits)
    return -mag if sign else mag


def _build_table(f: ElemFormat) -> np.ndarray:
    return np.array([_decode_code(f, c) for c in range(1 << f.nbits)],
                    dtype=np.float64)


E4M3 = ElemFormat("e4m3", 0, 4, 3, "fn")
E5M2 = ElemFormat("e5m2", 1, 5, 2, "ieee")
E2M1 = ElemFormat("e2m1", 2, 2, 1, "none")
FORMATS = {0: E4M3, 1: E5M2, 2: E2M1, "e4m3": E4M3, "e5m2": E5M2, "e2m1": E2M1}


def fmt(f) -> ElemFormat:
    return f if isinstance(f, ElemFormat) else FORMATS[f]


# ---------------------------------------------------------------- E8M0 scale
E8M0_NAN = 0xFF


def e8m0_decode(code) -> np.ndarray:
    """UE8M0 scale: code c in 0..254 means 2^(c - 127); 0xFF is NaN
    (explainer, section 1)."""
    c = np.asarray(code, dtype=np.int64)
    out = np.ldexp(1.0, c - 127).astype(np.float64)
    return np.where(c == E8M0_NAN, np.nan, out)


# ---------------------------------------------------------------- bf16 input
def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16): bf16 is the upper half of
    an IEEE binary32, so the value is that of the float32 ``bits << 16``."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f32_bits_to_f64(bits) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint32).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- decode / encode
def decode(f, codes) -> np.ndarray:
    """Value (float64) of each element code."""
    f = fmt(f)
    return f.table[np.asarray(codes, dtype=np.int64)]


def _positive_grid(f: ElemFormat):
    """Non-negative finite values in ascending order with their codes."""
    half = f.ncodes // 2
    codes = np.arange(half)
    vals = f.table[:half]
    keep = np.isfinite(vals)
    return vals[keep], codes[keep]


def encode_rne_sat(f, y) -> np.ndarray:
    """Round real values ``y`` (float64, taken as exact) to format ``f``:
    round-to-nearest, ties to the code with an even mantissa (its LSB 0),
    saturating to +-max_finite when |y| exceeds it (explainer, section 4:
    values beyond the upper limit are clamped).  The sign is always kept, so
    -0 and negative values that round to zero give the negative-zero code.
    NaN is outside the domain of this function (blocks holding NaN or Inf are
    handled by the block quantizer)."""
    f = fmt(f)
    y = np.asarray(y, dtype=np.float64)
    sign = np.signbit(y).astype(np.int64)
    a = np.minimum(np.abs(y), f.max_finite)
    vals, codes = _positive_grid(f)
    hi_i = np.searchsorted(vals, a, side="left")          # vals[hi_i] >= a
    hi_i = np.minimum(hi_i, len(vals) - 1)
    lo_i = np.where(vals[hi_i] == a, hi_i, np.maximum(hi_i - 1, 0))
    lo, hi = vals[lo_i], vals[hi_i]
    d_lo, d_hi = a - lo, hi - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((codes[hi_i] & 1) == 0)
                               & (lo_i != hi_i))
    pos = np.where(pick_hi, codes[hi_i], codes[lo_i])
    return (pos | (sign << (f.nbits - 1))).astype(np.uint8)


def neighbours(f, a):
    """For non-negative values ``a`` <= max_finite return (lo, hi): the
    largest grid value <= a and the smallest grid value >= a."""
    f = fmt(f)
    a = np.asarray(a, dtype=np.float64)
    vals, _ = _positive_grid(f)
    hi_i = np.minimum(np.searchsorted(vals, a, side="left"), len(vals) - 1)
    lo_i = np.where(vals[hi_i] == a, hi_i, np.maximum(hi_i - 1, 0))
    return vals[lo_i], vals[hi_i]


# ---------------------------------------------------------------- FP4 packing
def pack_fp4(codes: np.ndarray) -> np.ndarray:
    """Two E2M1 codes per byte along the last axis: element 2i in the low
    nibble, element 2i+1 in the high nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    assert c.shape[-1] % 2 == 0
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack_fp4(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out
