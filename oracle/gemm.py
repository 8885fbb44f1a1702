"""Block-scaled GEMM reference: the float64 product of the dequantized
operands, and the comparison gate.

Test infrastructure (see ``oracle/__init__``).

Definition followed: UE8M0 FP8 / MXFP8 explainer, section 1 -- tensor cores
consume the scale X and the codes q_i of both operands of each block and
form the dot product, accumulating in FP32; the same page (section on the
8B / 15T study) emulates MX by casting GEMM inputs to MX and back before a
higher-precision GEMM.  So the reference is

    C[m, n] = sum_k  dec(a[m, k]) * Xa[m, k/32] * dec(b[n, k]) * Xb[n, k/32]

in float64 (every product is exact), with A [M][K] and B [N][K] both
K-contiguous (C = A * B^T).  Each operand is decoded with its own element
format: the explainer's FP8 section sets E4M3 (more precise) beside E5M2
(wider range), so a product may pair an E5M2 gradient with an E4M3 operand.

Gate (reading; the target "max relative error 2e-3 against the float64
product" made attainable for a bf16 output): for each element,
    e_i = max(0, |c_i - ref_i| - ulp_bf16(max(|c_i|, |ref_i|)) / 2)
          / max(|ref_i|, rms(ref))
and the gate passes when max_i e_i <= 2e-3.  The half-ulp term removes the
output rounding itself; the rms floor keeps elements that cancel to near zero
from dividing by ~0.
"""

from __future__ import annotations

import numpy as np

from .mx import dequantize


def reference(a_q, a_s, b_q, b_s, f, fb=None) -> np.ndarray:
    """float64 C = dequant(A) @ dequant(B)^T; A in format f, B in fb (default f)."""
    A = dequantize(a_q, a_s, f)
    B = dequantize(b_q, b_s, f if fb is None else fb)
    return A @ B.T


def reference_rows_cols(a_q, a_s, b_q, b_s, f, rows, cols, fb=None) -> np.ndarray:
    """Sampled reference: C[rows][:, cols] only (rows/cols index arrays)."""
    A = dequantize(np.asarray(a_q)[rows], np.asarray(a_s)[rows], f)
    B = dequantize(np.asarray(b_q)[cols], np.asarray(b_s)[cols], f if fb is None else fb)
    return A @ B.T


def mm_fp8_reference(a8, b8, f, scale: float, bias=None) -> np.ndarray:
    """Per-tensor FP8 product (AstrAI fp8.py, mm_fp8: "a @ b * scale
    (+ bias)", scale the combined dequantization scale, bias added per output
    column): float64 C = (dec(a8) @ dec(b8)^T) * scale + bias with a8 [.., M, K]
    and b8 [.., N, K] FP8 codes of format f (both K-contiguous; a leading batch
    axis broadcasts like matmul) and bias [N] or None."""
    from .formats import decode
    A = decode(f, np.asarray(a8)).astype(np.float64)
    B = decode(f, np.asarray(b8)).astype(np.float64)
    C = np.matmul(A, np.swapaxes(B, -1, -2)) * float(scale)
    if bias is not None:
        C = C + np.asarray(bias, dtype=np.float64)
    return C


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits; subnormal floor
    2^-133)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    safe = np.where(a > 0, a, 1.0)
    _, ex = np.frexp(safe)
    u = np.ldexp(1.0, np.maximum(ex - 8, -133))
    return np.where(a > 0, u, np.ldexp(1.0, -133))


def gate_error(c: np.ndarray, ref: np.ndarray, out_is_bf16: bool = True) -> float:
    """Largest normalized element error e_i (see module docstring)."""
    c = np.asarray(c, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    slack = 0.5 * ulp_bf16(np.maximum(np.abs(c), np.abs(ref))) if out_is_bf16 else 0.0
    err = np.maximum(0.0, np.abs(c - ref) - slack)
    den = np.maximum(np.abs(ref), rms if rms > 0 else 1.0)
    return float(np.max(err / den)) if ref.size else 0.0


def frobenius_rel(c: np.ndarray, ref: np.ndarray) -> float:
    c = np.asarray(c, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(c - ref) / max(np.linalg.norm(ref), 1e-300))
