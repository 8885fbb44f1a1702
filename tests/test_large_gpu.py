"""Beyond 2^31 elements: the quantizer's 64-bit offsets (scale arrays,
transposed copies) on a 49152 x 49152 bf16 tensor (2.4e9 elements), bit for
bit against the oracle on sampled rows and 32-row slabs.  The input is tiles
of a seeded 4096 x 4096 block, each scaled by its own power of two, so a row
or tile mapped to the wrong place changes the bytes."""

import numpy as np
import pytest
import torch

from block_scaled_precision_02_gb300 import inputs
from oracle import formats as F
from oracle import mx as omx
from tests.helpers import assert_bytes_equal, f64, np_

pytestmark = pytest.mark.gpu

R = C = 49152


@pytest.fixture(scope="module")
def big():
    blk = inputs.activations(4096, 4096, seed=10).to("cuda")
    x = inputs.tiled_large(R, C, blk)
    yield blk, x
    del x
    torch.cuda.empty_cache()


def test_dual_beyond_2_31_elements(lib, big):
    blk, x = big
    assert x.numel() > 2 ** 31
    qr, sr, qc, sc = lib.mx_quantize(x, "e4m3", "dual", "floor")
    rows = [0, 4095, 4096, 30001, R - 1]
    xv = f64(inputs.tiled_large_rows(rows, C, blk, R))
    ref = omx.quantize(xv, F.E4M3, omx.ROW, omx.FLOOR)
    assert_bytes_equal(np_(qr[rows]), ref["q_row"], "q_row rows")
    assert_bytes_equal(np_(sr[rows]), ref["s_row"], "s_row rows")
    for sl in (0, 777, R // 32 - 1):
        r0 = sl * 32
        xs = f64(inputs.tiled_large_rows(range(r0, r0 + 32), C, blk, R))
        refc = omx.quantize(xs, F.E4M3, omx.COL, omx.FLOOR)
        assert_bytes_equal(np_(qc[:, r0:r0 + 32]), refc["q_col"], "q_col slab")
        assert_bytes_equal(np_(sc[:, sl:sl + 1]), refc["s_col"], "s_col slab")
    del qr, sr, qc, sc


def test_row_mma_layout_beyond_2_31_elements(lib, big):
    blk, x = big
    qr, sr, _, _ = lib.mx_quantize(x, "e5m2", "row", "ceil", sf_layout="mma")
    rows = [1, 20000, R - 2]
    xv = f64(inputs.tiled_large_rows(rows, C, blk, R))
    ref = omx.quantize(xv, F.E5M2, omx.ROW, omx.CEIL)
    assert_bytes_equal(np_(qr[rows]), ref["q_row"], "q_row rows")
    # MMA layout: row r, k-block k at chunk (r // 128, k // 4), byte (r % 32) * 16 + ((r // 32) % 4) * 4 + k % 4
    s = np_(sr).reshape(-1)
    kb = C // 32
    for n, r in enumerate(rows):
        k = np.arange(kb)
        off = ((r // 128) * (kb // 4) + k // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + k % 4
        assert_bytes_equal(s[off], ref["s_row"][n], "s_row (MMA layout)")
    del qr, sr


def test_gemm_outputs_beyond_2_31_elements(lib):
    """A 65536 x 33024 product (2.16e9 outputs) with K = 256: float32 C and
    the MX row and column-block outputs, on operands whose products and sums
    are exact in float32 (A = +-2^j per row, B small integers), so sampled
    rows, columns and 32-row slabs must equal the oracle bit for bit."""
    from oracle import gemm as og
    M, N, K = 65536, 33024, 256
    rng = np.random.default_rng(40)
    a = rng.choice([-1.0, 1.0], (M, K)) * np.exp2(rng.integers(-8, 9, size=(M, 1)))
    b = rng.integers(-4, 5, (N, K)).astype(np.float64)
    ra = omx.quantize(a, F.E4M3, omx.ROW, omx.FLOOR)
    rb = omx.quantize(b, F.E4M3, omx.ROW, omx.FLOOR)
    t = lambda v: torch.from_numpy(np.ascontiguousarray(v)).to("cuda")
    aq, as_ = t(ra["q_row"]), t(omx.sf_to_mma(ra["s_row"]))
    bq, bs = t(rb["q_row"]), t(omx.sf_to_mma(rb["s_row"]))
    rows = [0, 32767, 40000, M - 1]
    cols = [0, 12345, N - 1]
    c = lib.mx_gemm(aq, as_, bq, bs, "e4m3", torch.float32)
    assert c.numel() > 2 ** 31
    ref_rows = a[rows] @ b.T
    assert np.array_equal(np_(c[rows]).astype(np.float64), ref_rows)
    assert np.array_equal(np_(c[:, cols]).astype(np.float64), a @ b[cols].T)
    del c
    cq, cs, cqT, csT = lib.mx_gemm_mx_out(aq, as_, bq, bs, "e4m3", out_fmt="e4m3", orientation="dual")
    want = omx.quantize(ref_rows, F.E4M3, omx.ROW, omx.FLOOR)
    assert_bytes_equal(np_(cq[rows]), want["q_row"], "row codes")
    assert_bytes_equal(np_(cs[rows]), want["s_row"], "row scales")
    for sl in (0, 1500, M // 32 - 1):
        r0 = sl * 32
        ref = og.reference_rows_cols(ra["q_row"], ra["s_row"], rb["q_row"], rb["s_row"], F.E4M3,
                                     np.arange(r0, r0 + 32), np.arange(N))
        wc = omx.quantize(ref, F.E4M3, omx.COL, omx.FLOOR)
        assert_bytes_equal(np_(cqT[:, r0:r0 + 32]), wc["q_col"], "column-block codes")
        assert_bytes_equal(np_(csT[:, sl:sl + 1]), wc["s_col"], "column-block scales")
    del cq, cs, cqT, csT
