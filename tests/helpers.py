"""Shared test helpers: move seeded inputs to the oracle's float64 view and
report the first mismatch of two byte arrays."""

import numpy as np
import torch

from block_scaled_precision_02_gb300 import inputs
from oracle import formats as F


def f64(x: torch.Tensor) -> np.ndarray:
    """Exact float64 values of a bf16 tensor, via its bit patterns."""
    return F.bf16_bits_to_f64(inputs.bf16_bits(x))


def np_(t):
    return None if t is None else t.detach().cpu().numpy()


def assert_bytes_equal(got, want, what: str, inp=None):
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, f"{what}: shape {got.shape} != {want.shape}"
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        i = tuple(bad[0])
        extra = f", input {inp[i]!r}" if inp is not None and inp.shape == got.shape else ""
        raise AssertionError(f"{what}: {len(bad)} mismatches, first at {i}: got {got[i]:#x}, want {want[i]:#x}{extra}")
