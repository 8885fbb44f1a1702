"""GPU parity of the block-scaled GEMM against the oracle's float64 product.

Operands are quantized by the CPU oracle (never by the CUDA path), their
scales permuted into the tensor-core layout by the oracle, then multiplied
on the GPU.  Structured cases whose result is exactly representable must
match bit for bit; general cases must pass the 2e-3 gate (oracle.gemm).
"""

import numpy as np
import pytest
import torch

from block_scaled_precision_02_gb300 import inputs
from oracle import formats as F
from oracle import gemm as og
from oracle import mx as omx
from tests.helpers import f64

pytestmark = pytest.mark.gpu

FMTS = {"e4m3": F.E4M3, "e5m2": F.E5M2, "e2m1": F.E2M1}
TOL = 2e-3


def oracle_operand(x_f64, fmt, mode=omx.FLOOR):
    r = omx.quantize(x_f64, FMTS[fmt], omx.ROW, mode)
    return r["q_row"], r["s_row"]


def gpu_gemm(lib, aq, as_, bq, bs, fmt, out_dtype=torch.bfloat16, b_fmt=None):
    dev = torch.device("cuda")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    c = lib.mx_gemm(t(aq), t(omx.sf_to_mma(as_)), t(bq), t(omx.sf_to_mma(bs)), fmt, out_dtype, b_fmt=b_fmt)
    return c.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2", "e2m1"])
@pytest.mark.parametrize("mn", [(128, 256), (256, 512), (512, 256)])
def test_unit_rows_select_columns_exactly(lib, fmt, mn):
    """B row n holds a single non-zero at column perm[n]: C[:, n] is a scaled
    copy of one dequantized column of A (exact in bf16), so the scale mapping
    of both operands is checked bit for bit.  M = 128 runs the single-CTA
    kernel; M, N multiples of 256 run the CTA-pair kernel (both CTAs' rows,
    both halves of B)."""
    f = FMTS[fmt]
    rng = np.random.default_rng(1)
    M, N = mn
    K = 512
    a = rng.standard_normal((M, K)) * np.exp2(rng.integers(-6, 6, size=(M, K // 32))).repeat(32, 1)
    aq, as_ = oracle_operand(a, fmt)
    perm = rng.permutation(K)[:N]
    b = np.zeros((N, K))
    b[np.arange(N), perm] = np.exp2(rng.integers(-3, 4, size=N)) * (1.5 if fmt != "e2m1" else 1.0)
    bq, bs = oracle_operand(b, fmt)
    ref = og.reference(aq, as_, bq, bs, f)
    got = gpu_gemm(lib, aq, as_, bq, bs, fmt)
    assert np.array_equal(got, ref), f"max abs diff {np.max(np.abs(got - ref))}"


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2", "e2m1"])
@pytest.mark.parametrize("mnk", [(128, 256, 256), (256, 512, 1024), (384, 384, 512), (128, 128, 2048),
                                 (768, 512, 768), (256, 256, 4096), (128, 128, 256), (256, 256, 256)])
def test_random_gemm_gate(lib, fmt, mnk):
    M, N, K = mnk
    a = f64(inputs.activations(M, K, seed=0))
    b = f64(inputs.weights(N, K, seed=4))
    aq, as_ = oracle_operand(a, fmt)
    bq, bs = oracle_operand(b, fmt)
    ref = og.reference(aq, as_, bq, bs, FMTS[fmt])
    got = gpu_gemm(lib, aq, as_, bq, bs, fmt)
    err = og.gate_error(got, ref)
    assert err <= TOL, (err, og.frobenius_rel(got, ref))


MIXED = [("e4m3", "e5m2"), ("e5m2", "e4m3")]


@pytest.mark.parametrize("fa,fb", MIXED)
@pytest.mark.parametrize("mn", [(128, 256), (256, 512)])
def test_mixed_formats_unit_rows_exactly(lib, fa, fb, mn):
    """A in one 8-bit format, B (unit rows) in the other: C[:, n] is a
    scaled copy of one dequantized A column, exact in bf16, so each
    operand's element type in the instruction descriptor is checked."""
    rng = np.random.default_rng(3)
    M, N = mn
    K = 512
    a = rng.standard_normal((M, K)) * np.exp2(rng.integers(-6, 6, size=(M, K // 32))).repeat(32, 1)
    aq, as_ = oracle_operand(a, fa)
    perm = rng.permutation(K)[:N]
    b = np.zeros((N, K))
    b[np.arange(N), perm] = np.exp2(rng.integers(-3, 4, size=N)) * 1.5
    bq, bs = oracle_operand(b, fb)
    ref = og.reference(aq, as_, bq, bs, FMTS[fa], FMTS[fb])
    got = gpu_gemm(lib, aq, as_, bq, bs, fa, b_fmt=fb)
    assert np.array_equal(got, ref), f"max abs diff {np.max(np.abs(got - ref))}"


@pytest.mark.parametrize("fa,fb", MIXED)
@pytest.mark.parametrize("mnk", [(256, 512, 1024), (384, 384, 512), (512, 768, 2048)])
def test_mixed_formats_gate(lib, fa, fb, mnk):
    """E5M2 gradients times E4M3 weights (and the reverse) against the
    float64 product of the dequantized operands."""
    M, N, K = mnk
    a = f64(inputs.gradients(M, K, seed=1) if fa == "e5m2" else inputs.activations(M, K, seed=0))
    b = f64(inputs.gradients(N, K, seed=2) if fb == "e5m2" else inputs.weights(N, K, seed=4))
    aq, as_ = oracle_operand(a, fa)
    bq, bs = oracle_operand(b, fb)
    ref = og.reference(aq, as_, bq, bs, FMTS[fa], FMTS[fb])
    got = gpu_gemm(lib, aq, as_, bq, bs, fa, b_fmt=fb)
    assert og.gate_error(got, ref) <= TOL, (og.gate_error(got, ref), og.frobenius_rel(got, ref))


MIXED_FP4 = [("e4m3", "e2m1"), ("e5m2", "e2m1"), ("e2m1", "e4m3")]


@pytest.mark.parametrize("fa,fb", MIXED_FP4)
@pytest.mark.parametrize("mn", [(128, 256), (256, 512), (128, 128)])
def test_fp8_x_fp4_unit_rows_exactly(lib, fa, fb, mn):
    """An 8-bit operand beside a packed E2M1 one (kind::mxf8f6f4 with the
    E2M1 codes widened in shared memory): B's unit rows make C[:, n] a
    scaled copy of one dequantized A column, exact in bf16, so the widened
    layout, both element types and both operands' scales are checked bit for
    bit on the single-CTA kernel (M = 128) and the CTA pair."""
    rng = np.random.default_rng(5)
    M, N = mn
    K = 512
    a = rng.standard_normal((M, K)) * np.exp2(rng.integers(-6, 6, size=(M, K // 32))).repeat(32, 1)
    aq, as_ = oracle_operand(a, fa)
    perm = rng.permutation(K)[:N]
    b = np.zeros((N, K))
    b[np.arange(N), perm] = np.exp2(rng.integers(-3, 4, size=N)) * 1.5
    bq, bs = oracle_operand(b, fb)
    ref = og.reference(aq, as_, bq, bs, FMTS[fa], FMTS[fb])
    got = gpu_gemm(lib, aq, as_, bq, bs, fa, b_fmt=fb)
    assert np.array_equal(got, ref), f"max abs diff {np.max(np.abs(got - ref))}"


def _mixed_input(fmt, rows, K, seed):
    if fmt == "e2m1":
        return f64(inputs.fp4_operand(rows, K, seed=seed))
    if fmt == "e5m2":
        return f64(inputs.gradients(rows, K, seed=seed))
    return f64(inputs.activations(rows, K, seed=seed))


@pytest.mark.parametrize("fa,fb", MIXED_FP4)
@pytest.mark.parametrize("mnk", [(256, 512, 1024), (384, 384, 640), (128, 256, 128), (512, 768, 2048)])
def test_fp8_x_fp4_gate(lib, fa, fb, mnk):
    """MXFP8 activations (or E5M2 gradients) times MXFP4 weights, and the
    reverse, against the float64 product of the dequantized operands; K
    down to one 128-element step and K not a multiple of 256."""
    M, N, K = mnk
    a = _mixed_input(fa, M, K, 0)
    b = _mixed_input(fb, N, K, 4)
    aq, as_ = oracle_operand(a, fa)
    bq, bs = oracle_operand(b, fb)
    ref = og.reference(aq, as_, bq, bs, FMTS[fa], FMTS[fb])
    got = gpu_gemm(lib, aq, as_, bq, bs, fa, b_fmt=fb)
    assert og.gate_error(got, ref) <= TOL, (og.gate_error(got, ref), og.frobenius_rel(got, ref))


def test_fp32_output_and_many_tiles(lib):
    """float32 epilogue, and more output tiles than SMs (the persistent loop)."""
    M, N, K = 2048, 4096, 256
    a = f64(inputs.activations(M, K, seed=5))
    b = f64(inputs.weights(N, K, seed=6))
    aq, as_ = oracle_operand(a, "e4m3", omx.CEIL)
    bq, bs = oracle_operand(b, "e4m3", omx.CEIL)
    ref = og.reference(aq, as_, bq, bs, F.E4M3)
    got32 = gpu_gemm(lib, aq, as_, bq, bs, "e4m3", torch.float32)
    assert og.gate_error(got32, ref, out_is_bf16=False) <= 1e-5
    got16 = gpu_gemm(lib, aq, as_, bq, bs, "e4m3")
    assert og.gate_error(got16, ref) <= TOL


def test_pm_one_operands_integer_sums(lib):
    """All-+-1 E2M1 operands: every product and partial sum is a small
    integer, exact in float32, so C equals a @ b^T exactly."""
    rng = np.random.default_rng(2)
    M, N, K = 256, 256, 512
    a = rng.choice([-1.0, 1.0], (M, K))
    b = rng.choice([-1.0, 1.0], (N, K))
    aq, as_ = oracle_operand(a, "e2m1")
    bq, bs = oracle_operand(b, "e2m1")
    got = gpu_gemm(lib, aq, as_, bq, bs, "e2m1", torch.float32)
    assert np.array_equal(got, a @ b.T)


@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_fp4_many_tiles_exact(lib, out):
    """MXFP4 with bf16 and float32 output over 256 pair tiles (several per
    CTA pair, so the epilogue's one staging buffer is reused across tiles
    and chunks): +-1 operands give even integer sums of magnitude at most
    512, exact in float32 and in bf16, so C equals a @ b^T exactly."""
    rng = np.random.default_rng(12)
    M, N, K = 4096, 4096, 512
    a = rng.choice([-1.0, 1.0], (M, K))
    b = rng.choice([-1.0, 1.0], (N, K))
    aq, as_ = oracle_operand(a, "e2m1")
    bq, bs = oracle_operand(b, "e2m1")
    got = gpu_gemm(lib, aq, as_, bq, bs, "e2m1", out)
    assert np.array_equal(got, a @ b.T)


def _sampled(lib, M, N, K, fmt, gen_a, gen_b, nrows=64, ncols=64):
    a = f64(gen_a(M, K))
    b = f64(gen_b(N, K))
    aq, as_ = oracle_operand(a, fmt)
    bq, bs = oracle_operand(b, fmt)
    got = gpu_gemm(lib, aq, as_, bq, bs, fmt)
    rng = np.random.default_rng(7)
    rows = np.sort(rng.choice(M, nrows, replace=False))
    cols = np.sort(rng.choice(N, ncols, replace=False))
    ref = og.reference_rows_cols(aq, as_, bq, bs, FMTS[fmt], rows, cols)
    err = og.gate_error(got[np.ix_(rows, cols)], ref)
    assert err <= TOL, err


def test_full_size_square_sampled(lib):
    """8192 x 4096 activations times 4096 x 4096 weights (MXFP8 E4M3)."""
    _sampled(lib, 8192, 4096, 4096, "e4m3", lambda m, k: inputs.activations(m, k, seed=0),
             lambda n, k: inputs.weights(n, k, seed=4))


def test_full_size_ffn_sampled(lib):
    """8192 x 4096 activations times 14336 x 4096 weights (MXFP8 E4M3)."""
    _sampled(lib, 8192, 14336, 4096, "e4m3", lambda m, k: inputs.activations(m, k, seed=0),
             lambda n, k: inputs.weights(n, k, seed=5))


def test_full_size_mixed_sampled(lib):
    """The bench's mixed-format product: the 8192 x 4096 E5M2 gradient times
    the 4096 x 4096 E4M3 weights."""
    M, N, K = 8192, 4096, 4096
    a = f64(inputs.gradients(M, K, seed=1))
    b = f64(inputs.weights(N, K, seed=4))
    aq, as_ = oracle_operand(a, "e5m2")
    bq, bs = oracle_operand(b, "e4m3")
    got = gpu_gemm(lib, aq, as_, bq, bs, "e5m2", b_fmt="e4m3")
    rng = np.random.default_rng(8)
    rows = np.sort(rng.choice(M, 64, replace=False))
    cols = np.sort(rng.choice(N, 64, replace=False))
    ref = og.reference_rows_cols(aq, as_, bq, bs, F.E5M2, rows, cols, F.E4M3)
    assert og.gate_error(got[np.ix_(rows, cols)], ref) <= TOL


def test_full_size_fp8_x_fp4_sampled(lib):
    """The bench's MXFP8 x MXFP4 product: 8192 x 4096 E4M3 activations times
    4096 x 4096 E2M1 weights."""
    M, N, K = 8192, 4096, 4096
    a = f64(inputs.activations(M, K, seed=0))
    b = f64(inputs.fp4_operand(N, K, seed=8))
    aq, as_ = oracle_operand(a, "e4m3")
    bq, bs = oracle_operand(b, "e2m1")
    got = gpu_gemm(lib, aq, as_, bq, bs, "e4m3", b_fmt="e2m1")
    rng = np.random.default_rng(9)
    rows = np.sort(rng.choice(M, 64, replace=False))
    cols = np.sort(rng.choice(N, 64, replace=False))
    ref = og.reference_rows_cols(aq, as_, bq, bs, F.E4M3, rows, cols, F.E2M1)
    assert og.gate_error(got[np.ix_(rows, cols)], ref) <= TOL


def test_full_size_fp4_sampled(lib):
    """4096 x 14336 gradient times 4096 x 14336 operand (MXFP4 E2M1)."""
    _sampled(lib, 4096, 4096, 14336, "e2m1", lambda m, k: inputs.heavy_gradient(m, k, seed=6),
             lambda n, k: inputs.fp4_operand(n, k, seed=8))


def test_device_status_clean_after_gemm(lib):
    assert lib.last_device_status() == 0
