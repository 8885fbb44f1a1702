"""MX (microscaling) block quantization, dequantization and the fixed-sign
32-point Hadamard preconditioner.

Test infrastructure (see ``oracle/__init__``).

Definitions followed:
* UE8M0 FP8 / MXFP8 explainer, section 1: an MX block is k = 32 elements that
  share one UE8M0 scale X; quantizing source values V_i means finding X and
  element codes q_i with q_i * X ~= V_i, and storing X and the q_i.
* Same page, section 4: the scale's exponent comes from the block amax and
  elements are quantized with saturation (clamped at the format maximum).
* Same page, gap section 1: two scale-rounding rules exist -- the OCP v1.0
  "round down" rule (here ``floor``: X = 2^(floor(log2 amax) -
  floor(log2 destmax))) and the NVIDIA training recipe that rounds up
  (here ``ceil``: X = 2^ceil(log2(amax / destmax))).
* Same page, gap section 2: tensors consumed along both axes need a row-wise
  (1x32) and a column-wise (32x1) copy; the column copy is stored transposed
  so its blocks run along the contiguous dimension.
* Format-aware fusion article (MXFP4 recipe): row-gradient stochastic
  rounding and a fixed-sign 32-point Hadamard on each 32-block.

Readings where the pages are silent (each listed in the design notes):
* amax == 0 gives the smallest scale code (e = -127); a block holding NaN or
  Inf gets the NaN scale code 0xFF and zero codes.
* Scale exponents are clamped to [-127, 127].
* Stochastic rounding: r = word 0 of Philox-4x32-10(key = seed,
  counter = flat element index); with y' = min(|y|, max) strictly between
  grid neighbours lo < y' < hi, t = floor((y' - lo) / (hi - lo) * 2^32) and
  the magnitude rounds up to hi iff r < t.  The sign is reattached.
  Option ``SR4``: the same rounding with r = word (index & 3) of the call
  with counter = index >> 2 (one generator call per four elements).
* Hadamard: u_j = s_j v_j; butterflies h = 1, 2, 4, 8, 16 in that order in
  float32 round-to-nearest, (u_i, u_{i+h}) <- (u_i + u_{i+h}, u_i - u_{i+h})
  for (i & h) == 0; then y_j = RN32(u_j * c) with c = RN32(1 / sqrt(32)).
"""

from __future__ import annotations

import numpy as np

from . import formats as F
from .philox import hadamard_signs, sr_draw, sr_draw4

K = 32  # MX block size, the same for every MX element type (explainer, section 1)

FLOOR = 0
CEIL = 1
RNE = 0
SR = 1
SR4 = 2
ROW = 1
COL = 2
DUAL = 3


# ------------------------------------------------------------------ scales
def exponent_mantissa(a: np.ndarray):
    """a = m * 2^E with m in [1, 2) for finite a > 0 (exact; subnormals
    included).  Returns (E, m)."""
    fr, ex = np.frexp(np.asarray(a, dtype=np.float64))
    return ex.astype(np.int64) - 1, fr * 2.0


def scale_exponent(amax: np.ndarray, f, mode: int) -> np.ndarray:
    """Shared-scale exponent e of each block from its amax (float64, >= 0,
    finite).  floor: e = E(amax) - E(destmax).  ceil: the smallest e with
    amax * 2^-e <= destmax, i.e. E(amax) - E(destmax) + [m(amax) > m(destmax)].
    amax == 0 gives -127.  Clamped to [-127, 127]."""
    f = F.fmt(f)
    amax = np.asarray(amax, dtype=np.float64)
    Ed, md = exponent_mantissa(np.float64(f.max_finite))
    safe = np.where(amax > 0, amax, 1.0)
    Ea, ma = exponent_mantissa(safe)
    e = Ea - Ed
    if mode == CEIL:
        e = e + (ma > md).astype(np.int64)
    e = np.where(amax > 0, e, -127)
    return np.clip(e, -127, 127)


# ------------------------------------------------------------------ Hadamard
def rn32(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32)


HADAMARD_C = np.float32(1.0 / np.sqrt(np.float64(32.0)))  # RN32(1/sqrt(32)); pinned in tests


def hadamard32_blocks(v32: np.ndarray, seed: int) -> np.ndarray:
    """Apply the fixed-sign 32-point Hadamard to each block along the last
    axis (length 32).  Input float32 (or exactly-float32 values); output
    float32.  Follows the float32 butterfly order stated in the module
    docstring."""
    s = hadamard_signs(seed).astype(np.float32)
    u = (np.asarray(v32, dtype=np.float32) * s).astype(np.float32)
    assert u.shape[-1] == 32
    h = 1
    while h < 32:
        nu = u.copy()
        for i in range(32):
            if i & h == 0:
                a, b = u[..., i], u[..., i + h]
                nu[..., i] = a + b            # float32 add, round-to-nearest
                nu[..., i + h] = a - b
        u = nu
        h *= 2
    return (u * HADAMARD_C).astype(np.float32)


def sylvester(n: int = 32) -> np.ndarray:
    """Dense Sylvester Hadamard matrix H_ij = (-1)^popcount(i & j)."""
    i = np.arange(n)
    pc = np.vectorize(lambda v: bin(v).count("1"))(i[:, None] & i[None, :])
    return np.where(pc % 2 == 0, 1, -1).astype(np.int64)


# ------------------------------------------------------------------ element step
def quantize_blocks(vals: np.ndarray, f, mode: int, rounding: int = RNE,
                    sr_seed: int = 0, flat_idx: np.ndarray | None = None):
    """Quantize blocks along the last axis (length 32).

    vals: float64 values that are exactly those the method scales (bf16
    inputs, or the float32 Hadamard outputs).  Returns (codes uint8 [..., 32],
    scale codes uint8 [...]).  ``flat_idx`` gives each element's index in the
    input tensor (needed for stochastic rounding)."""
    f = F.fmt(f)
    v = np.asarray(vals, dtype=np.float64)
    bad = ~np.all(np.isfinite(v), axis=-1)
    amax = np.max(np.abs(np.where(np.isfinite(v), v, 0.0)), axis=-1)
    e = scale_exponent(amax, f, mode)
    y = v * np.ldexp(1.0, -e)[..., None]            # exact in float64
    y = np.where(np.isfinite(y), y, 0.0)
    if rounding == RNE:
        q = F.encode_rne_sat(f, y)
    elif rounding == SR4:
        q = stochastic_round(f, y, sr_draw4(sr_seed, flat_idx))
    else:
        q = stochastic_round(f, y, sr_draw(sr_seed, flat_idx))
    q = np.where(bad[..., None], np.uint8(0), q)
    s = np.where(bad, np.uint8(F.E8M0_NAN), (e + 127).astype(np.uint8))
    return q.astype(np.uint8), s.astype(np.uint8)


def sr_threshold(f, y: np.ndarray):
    """For stochastic rounding of float64 y: returns (lo, hi, t) where
    lo <= min(|y|, max) <= hi are grid neighbours and t the 32-bit threshold
    floor((y' - lo) / (hi - lo) * 2^32) (0 when y' is on the grid)."""
    f = F.fmt(f)
    a = np.minimum(np.abs(y), f.max_finite)
    lo, hi = F.neighbours(f, a)
    span = np.where(hi > lo, hi - lo, 1.0)
    t = np.floor((a - lo) / span * 4294967296.0)
    t = np.where(hi > lo, t, 0.0).astype(np.uint64)
    return lo, hi, t


def stochastic_round(f, y: np.ndarray, r: np.ndarray) -> np.ndarray:
    """Stochastic rounding of float64 y with 32-bit draws r (see module
    docstring).  The magnitude rounds up iff r < t."""
    f = F.fmt(f)
    lo, hi, t = sr_threshold(f, y)
    up = np.asarray(r, dtype=np.uint64) < t
    mag = np.where(up, hi, lo)
    mag = np.where(np.signbit(y), -mag, mag)
    # mag is on the grid; encode keeps it and keeps the sign (also of zero)
    sgn = np.signbit(y)
    mag = np.where(mag == 0, np.where(sgn, -0.0, 0.0), mag)
    return F.encode_rne_sat(f, mag)


# ------------------------------------------------------------------ tensor quantizer
def quantize(x: np.ndarray, f, orient: int = ROW, mode: int = FLOOR,
             rounding: int = RNE, hadamard32: bool = False,
             sr_seed: int = 0, hadamard_seed: int = 7,
             row_index=None, total_cols: int | None = None):
    """MX-quantize a 2-D tensor ``x`` (float64 holding exact bf16 values).

    Row orientation: blocks x[r, 32j:32j+32]; codes q_row [R][C] and scales
    s_row [R][C/32].  Column orientation: blocks x[32i:32i+32, c]; the copy is
    stored transposed, codes q_col [C][R] and scales s_col [C][R/32], so that
    q_col is the row-wise quantization of x^T.  E2M1 codes are packed two per
    byte (low nibble = even index along the contiguous axis).

    ``row_index`` / ``total_cols`` let a caller quantize sampled rows of a
    larger tensor: element (i, c) then has flat index
    row_index[i] * total_cols + c (the stochastic-rounding counter).

    Returns a dict with the requested outputs."""
    f = F.fmt(f)
    x = np.asarray(x, dtype=np.float64)
    R, C = x.shape
    if orient in (ROW, DUAL):
        assert C % K == 0
    if orient in (COL, DUAL):
        assert R % K == 0
    out = {}
    if row_index is None:
        idx = np.arange(R * C, dtype=np.int64).reshape(R, C)
    else:
        tc = C if total_cols is None else int(total_cols)
        idx = np.asarray(row_index, dtype=np.int64)[:, None] * tc + np.arange(C, dtype=np.int64)[None, :]

    def one(xx, ii):
        rr, cc = xx.shape
        qs, ss = [], []
        for a in range(0, rr, 512):          # row slices bound the temporaries
            vb = xx[a:a + 512].reshape(-1, cc // K, K)
            ib = ii[a:a + 512].reshape(-1, cc // K, K)
            if hadamard32:
                vb = hadamard32_blocks(rn32(vb), hadamard_seed).astype(np.float64)
            q, s = quantize_blocks(vb, f, mode, rounding, sr_seed, ib)
            q = q.reshape(-1, cc)
            if f.nbits == 4:
                q = F.pack_fp4(q)
            qs.append(q)
            ss.append(s)
        return np.concatenate(qs), np.concatenate(ss)

    if orient in (ROW, DUAL):
        out["q_row"], out["s_row"] = one(x, idx)
    if orient in (COL, DUAL):
        out["q_col"], out["s_col"] = one(x.T, idx.T)
    return out


def dequantize(q: np.ndarray, s: np.ndarray, f) -> np.ndarray:
    """v_hat = decode(q) * 2^(s - 127), exact in float64; scale 0xFF gives
    NaN.  ``q`` is [R][C] codes (E2M1 packed [R][C/2]), ``s`` [R][C/32]."""
    f = F.fmt(f)
    q = np.asarray(q, dtype=np.uint8)
    if f.nbits == 4:
        q = F.unpack_fp4(q)
    v = F.decode(f, q)
    X = F.e8m0_decode(s)
    return v * np.repeat(X, K, axis=-1)


# ------------------------------------------------------------------ MMA scale layout
def sf_to_mma(s: np.ndarray) -> np.ndarray:
    """Permute canonical scales s [rows][kb] (rows % 128 == 0, kb % 4 == 0)
    into the tensor-core layout: 512-byte chunks, one per 128 rows x 4 scale
    columns (128 K-elements), chunk (rb, kc) at byte (rb * kb/4 + kc) * 512;
    inside a chunk, the scale of row r and k-block k sits at byte
    (r % 32) * 16 + ((r // 32) % 4) * 4 + (k % 4).  Returns a flat uint8
    array."""
    s = np.asarray(s, dtype=np.uint8)
    rows, kb = s.shape
    assert rows % 128 == 0 and kb % 4 == 0
    out = np.empty(rows * kb, dtype=np.uint8)
    r = np.arange(rows)[:, None]
    k = np.arange(kb)[None, :]
    pos = ((r // 128) * (kb // 4) + k // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (k % 4)
    out[pos.ravel()] = s.ravel()
    return out


def sf_from_mma(flat: np.ndarray, rows: int, kb: int) -> np.ndarray:
    flat = np.asarray(flat, dtype=np.uint8).ravel()
    r = np.arange(rows)[:, None]
    k = np.arange(kb)[None, :]
    pos = ((r // 128) * (kb // 4) + k // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (k % 4)
    return flat[pos]
