"""Per-tensor FP8 quantize with fused amax and the delayed-scaling history fold.

Test infrastructure (see ``oracle/__init__``).

Definitions followed (AstrAI ``astrai/extension/ops/fp8.py``):
* ``quantize`` docstring: ``scale`` is the quantization multiplier, ``fmt`` is
  E4M3 or E5M2, the tensor amax is returned; ``transposed`` gives x8T, the
  [cols][rows] row-major transpose of the quantized input.
* ``quantize_dual`` docstring: one read gives both x8 and x8T (and amax).
* ``quantize`` docstring and the commit message: with a ring buffer laid out
  [hist n | scale | legacy | amax | done], the kernel's last block folds the
  amax into hist[hist_idx] and publishes the next scale
  max(hist) / fp8_max / pow2_margin; the amax slot is then self-cleaned and
  reads zero.

Readings (the page leaves these open):
* x8 = RNE-saturating encode of RN32(x * m): the bf16 x fp32 product is
  exact in float64 and rounded once to float32.
* The ``scale`` slot holds the published value max(hist)/fp8_max/pow2_margin
  (a dequantization scale), each division correctly rounded to float32; the
  ``legacy`` slot holds RN32(1 / scale), the multiplier form the next step
  passes in.  ``pow2_margin`` is a plain divisor.  When max(hist) is 0 or not
  finite nothing is published.  amax and done are reset to 0.
"""

from __future__ import annotations

import numpy as np

from . import formats as F


def quantize_pertensor(x: np.ndarray, m: float, f):
    """x float64 (exact bf16 values), m float32 multiplier.
    Returns (x8 [R][C] uint8, x8T [C][R] uint8, amax float)."""
    f = F.fmt(f)
    assert f.nbits == 8
    x = np.asarray(x, dtype=np.float64)
    amax = float(np.max(np.abs(x))) if x.size else 0.0
    p = (x * np.float64(np.float32(m))).astype(np.float32).astype(np.float64)
    x8 = F.encode_rne_sat(f, p)
    return x8, np.ascontiguousarray(x8.T), amax


def ring_new(n: int) -> np.ndarray:
    """Initial ring: hist = 0, scale = 1, legacy = 1, amax = 0, done = 0."""
    r = np.zeros(n + 4, dtype=np.float32)
    r[n] = 1.0
    r[n + 1] = 1.0
    return r


def _div32(a: float, b: float) -> np.float32:
    # float64 quotient rounded to float32 equals the correctly rounded
    # float32 quotient (53 >= 2*24 + 2)
    return np.float32(np.float64(np.float32(a)) / np.float64(np.float32(b)))


def ring_fold(ring: np.ndarray, amax: float, hist_idx: int,
              fp8_max: float = 448.0, pow2_margin: float = 1.0) -> np.ndarray:
    """Fold one step's amax into the ring and publish the next scale."""
    r = np.array(ring, dtype=np.float32, copy=True)
    n = r.size - 4
    r[hist_idx] = np.float32(amax)
    M = float(np.max(r[:n]))
    if M > 0 and np.isfinite(M):
        sc = _div32(float(_div32(M, fp8_max)), pow2_margin)
        r[n] = sc
        r[n + 1] = np.float32(np.float64(1.0) / np.float64(sc))
    r[n + 2] = 0.0
    r[n + 3] = 0.0
    return r
