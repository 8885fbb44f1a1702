"""Seeded synthetic inputs for the quantizers and the GEMM.

This module holds no quantization arithmetic: it draws float32 values with
numpy's ``default_rng(seed)`` and rounds them once to bf16 (round to nearest
even, by torch).  The same bf16 bytes feed the CUDA path and the CPU
oracle.  ``N(0, s^2)`` in the workload descriptions is a variance.

Workloads (shapes and laws of the five configurations this library is
measured on):

* ``small_rowwise``   256 x 512, N(0,1) * 2^u_r with u_r ~ U[-8, 8] per row,
  0.5 % of entries set to +-0, 4 entries set to +-1e4.  Seed 0.
* ``activations``     R x C, N(0,1) with 0.1 % of the columns (at least one)
  scaled by 100 (outlier channels).  Seed 0 (8192 x 4096 by default).
* ``gradients``       R x C, N(0, 1e-3).  Seed 1.
* ``pertensor_base``  4096 x 14336, N(0, 0.02^2).  Seed 2; the 16 per-step
  power-of-two factors 2^v, v ~ U{-4..4}, come from seed 3 (a power of two
  keeps every bf16 value exact).
* ``weights``         N x K, N(0, 0.02^2).  Seed 4 (4096 x 4096), 5 (14336 x 4096).
* ``heavy_gradient``  4096 x 14336, 1e-2 * t_3 / sqrt(3) (Student-t, nu = 3,
  normalised to variance 1e-4).  Seed 6.
* ``fp4_operand``     4096 x 14336, N(0, 1).  Seed 8.
* ``tiled_large``     beyond 2^31 elements: tiles of a seeded block, each
  scaled by 2^e, e ~ U{-3..3} (seed 9), for the 64-bit indexing cases.
"""

from __future__ import annotations

import numpy as np
import torch


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """float32 numpy -> bf16 torch CPU tensor (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bf16 tensor (CPU copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def normal(rows: int, cols: int, std: float, seed: int) -> torch.Tensor:
    rng = np.random.default_rng(seed)
    return to_bf16(rng.standard_normal((rows, cols), dtype=np.float32) * np.float32(std))


def small_rowwise(rows: int = 256, cols: int = 512, seed: int = 0) -> torch.Tensor:
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, cols), dtype=np.float32)
    u = rng.uniform(-8.0, 8.0, size=(rows, 1)).astype(np.float32)
    x = x * np.exp2(u).astype(np.float32)
    n = rows * cols
    nz = int(round(0.005 * n))
    zi = rng.choice(n, size=nz, replace=False)
    zs = rng.integers(0, 2, size=nz)
    flat = x.reshape(-1)
    flat[zi] = np.where(zs == 1, np.float32(-0.0), np.float32(0.0))
    rest = np.setdiff1d(np.arange(n), zi)
    bi = rng.choice(rest, size=min(4, rest.size), replace=False)
    bs = rng.integers(0, 2, size=bi.size)
    flat[bi] = np.where(bs == 1, np.float32(-1e4), np.float32(1e4))
    return to_bf16(x)


def activations(rows: int = 8192, cols: int = 4096, seed: int = 0) -> torch.Tensor:
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, cols), dtype=np.float32)
    nout = max(1, int(round(0.001 * cols)))
    oc = rng.choice(cols, size=nout, replace=False)
    x[:, oc] *= np.float32(100.0)
    return to_bf16(x)


def gradients(rows: int = 8192, cols: int = 4096, seed: int = 1) -> torch.Tensor:
    return normal(rows, cols, float(np.sqrt(1e-3)), seed)


def pertensor_base(rows: int = 4096, cols: int = 14336, seed: int = 2) -> torch.Tensor:
    return normal(rows, cols, 0.02, seed)


def pertensor_step_exponents(steps: int = 16, seed: int = 3) -> list[int]:
    rng = np.random.default_rng(seed)
    return [int(v) for v in rng.integers(-4, 5, size=steps)]


def pertensor_step(base: torch.Tensor, v: int) -> torch.Tensor:
    """Step input x_t = base * 2^v (bf16, on base's device).  A power-of-two
    factor is exact in bf16 for these magnitudes, so every step's values are
    the base's, shifted in exponent."""
    return (base.float() * (2.0 ** v)).to(torch.bfloat16)


def weights(rows: int = 4096, cols: int = 4096, seed: int = 4) -> torch.Tensor:
    return normal(rows, cols, 0.02, seed)


def heavy_gradient(rows: int = 4096, cols: int = 14336, seed: int = 6) -> torch.Tensor:
    rng = np.random.default_rng(seed)
    t = rng.standard_t(3, size=(rows, cols)).astype(np.float32)
    return to_bf16(t * np.float32(1e-2 / np.sqrt(3.0)))


def fp4_operand(rows: int = 4096, cols: int = 14336, seed: int = 8) -> torch.Tensor:
    return normal(rows, cols, 1.0, seed)


def tiled_large(rows: int, cols: int, block: torch.Tensor, seed: int = 9) -> torch.Tensor:
    """A tensor larger than 2^31 elements built on ``block``'s device from a
    small block: tile (i, j) of the result is ``block * 2^e_ij`` with e_ij ~
    U{-3..3} (seed ``seed``; a power of two keeps every bf16 value exact),
    so neighbouring tiles differ in scale.  ``tiled_large_rows`` rebuilds
    any rows of it on the CPU."""
    br, bc = block.shape
    e = tiled_large_exponents(rows // br, cols // bc, seed)
    f = torch.from_numpy(np.exp2(e).astype(np.float32)).to(block.device)
    out = torch.empty(rows, cols, dtype=torch.bfloat16, device=block.device)
    for i in range(rows // br):
        for j in range(cols // bc):
            out[i * br:(i + 1) * br, j * bc:(j + 1) * bc] = (block.float() * f[i, j]).to(torch.bfloat16)
    return out


def tiled_large_exponents(ti: int, tj: int, seed: int = 9) -> np.ndarray:
    return np.random.default_rng(seed).integers(-3, 4, size=(ti, tj)).astype(np.float64)


def tiled_large_rows(rows_idx, cols: int, block: torch.Tensor, nrows: int, seed: int = 9) -> torch.Tensor:
    """Rows ``rows_idx`` of ``tiled_large(nrows, cols, block, seed)``, on the CPU."""
    br, bc = block.shape
    e = tiled_large_exponents(nrows // br, cols // bc, seed)
    b = block.cpu().float()
    rows = []
    for r in rows_idx:
        i = r // br
        f = torch.from_numpy(np.repeat(np.exp2(e[i]).astype(np.float32), bc))
        rows.append((b[r % br].repeat(cols // bc) * f).to(torch.bfloat16))
    return torch.stack(rows)


def special_values_bf16() -> np.ndarray:
    """A row of 32 awkward bf16 values (zeros of both signs, a subnormal,
    large and small magnitudes) as float32, for edge-case tests."""
    v = np.array([0.0, -0.0, 1.0, -1.0, 2.0 ** -133, -(2.0 ** -130), 3.0e38, -1.5,
                  448.0, 449.0, 464.0, 480.0, 57344.0, 6.0, 5.0, 0.25,
                  1e-3, -1e-3, 7.0, -7.5, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -11, 0.75,
                  1.75, 1.875, -2.5, 3.5, 0.125, -0.0625, 100.0, -1e4], dtype=np.float64)
    return v.astype(np.float32)
