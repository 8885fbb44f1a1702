"""GPU parity of the GEMM's other outputs: the MX-quantized output (codes and
UE8M0 scales of 1x32 row blocks written from the accumulator) and the
per-tensor FP8 product with scale and bias (mm_fp8).

Operands come from the CPU oracle.  Where the float32 accumulation is exact
(small-integer sums), the MX output must equal the oracle's MX quantization
of the float64 product bit for bit; elsewhere the decisions are taken on the
kernel's float32 accumulator, which the oracle cannot reproduce, so the
check is a property that holds at any size: the dequantized output sits
within one element step of the float64 product and nearly every code
agrees.  The per-tensor product passes the 2e-3 gate (oracle.gemm).
"""

import numpy as np
import pytest
import torch

from block_scaled_precision_02_gb300 import inputs
from oracle import formats as F
from oracle import gemm as og
from oracle import mx as omx
from tests.helpers import assert_bytes_equal, f64, np_

pytestmark = pytest.mark.gpu

FMTS = {"e4m3": F.E4M3, "e5m2": F.E5M2, "e2m1": F.E2M1}
MODES = {"floor": omx.FLOOR, "ceil": omx.CEIL}
dev = torch.device("cuda")


def t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def mx_operand(x, fmt):
    r = omx.quantize(x, FMTS[fmt], omx.ROW, omx.FLOOR)
    return r["q_row"], r["s_row"]


def run_mx_out(lib, aq, as_, bq, bs, fmt, out_fmt, mode, layout, orientation="row"):
    """Codes and canonical scales of the row blocks and of the (transposed)
    column blocks; None for an orientation not requested."""
    out = lib.mx_gemm_mx_out(t(aq), t(omx.sf_to_mma(as_)), t(bq), t(omx.sf_to_mma(bs)), fmt,
                             out_fmt=out_fmt, out_scale_mode=mode, out_sf_layout=layout, orientation=orientation)
    res = []
    for q, s in (out[0:2], out[2:4]):
        if q is None:
            res += [None, None]
            continue
        q = q.cpu().numpy()
        s = s.cpu().numpy()
        if layout == "mma":
            s = omx.sf_from_mma(s.reshape(-1), q.shape[0], s.size // q.shape[0])
        res += [q, s]
    return res


@pytest.mark.parametrize("out_fmt", ["e4m3", "e5m2", "e2m1"])
@pytest.mark.parametrize("mode", ["floor", "ceil"])
@pytest.mark.parametrize("layout", ["canonical", "mma"])
@pytest.mark.parametrize("mnk", [(128, 256, 512), (256, 512, 1024), (128, 384, 256)])
@pytest.mark.parametrize("orientation", ["row", "col", "dual"])
def test_mx_output_exact_on_integer_products(lib, out_fmt, mode, layout, mnk, orientation):
    """A = +-2^j per row (exact in E4M3 with the row scale), B = small
    integers: every product and partial sum is exact in float32, so the
    accumulator equals the float64 product and the MX output must equal the
    oracle's quantization of it, codes and scales, for the row blocks and
    for the transposed column blocks."""
    M, N, K = mnk
    rng = np.random.default_rng(21)
    a = rng.choice([-1.0, 1.0], (M, K)) * np.exp2(rng.integers(-8, 9, size=(M, 1)))
    b = rng.integers(-4, 5, (N, K)).astype(np.float64)
    aq, as_ = mx_operand(a, "e4m3")
    bq, bs = mx_operand(b, "e4m3")
    ref = og.reference(aq, as_, bq, bs, F.E4M3)
    assert np.array_equal(ref, a @ b.T)                          # the operands quantize exactly
    want = omx.quantize(ref, FMTS[out_fmt], omx.DUAL, MODES[mode])
    cq, cs, cqT, csT = run_mx_out(lib, aq, as_, bq, bs, "e4m3", out_fmt, mode, layout, orientation)
    if orientation in ("row", "dual"):
        assert_bytes_equal(cq, want["q_row"], "codes")
        assert_bytes_equal(cs, want["s_row"], "scales")
    else:
        assert cq is None
    if orientation in ("col", "dual"):
        assert_bytes_equal(cqT, want["q_col"], "column-block codes")
        assert_bytes_equal(csT, want["s_col"], "column-block scales")
    else:
        assert cqT is None


@pytest.mark.parametrize("out_fmt", ["e4m3", "e2m1"])
@pytest.mark.parametrize("layout", ["canonical", "mma"])
@pytest.mark.parametrize("mnk", [(128, 256, 512), (256, 512, 256)])
def test_mx_output_nonfinite_blocks(lib, out_fmt, layout, mnk):
    """Accumulator rows that are not finite: row m0 takes a NaN scale (UE8M0
    0xFF) on its first k-block, row m1 the scale 2^127, which drives every
    product of that k-block past float32's range (the first k-block's A and
    B values are all positive, so no cancellation can bring the sum back).
    Every 1x32 row block of those rows and every 32x1 column block of their
    32-row bands must carry scale 0xFF and zero codes; all other blocks are
    the oracle's quantization of the exact integer product.  The float32
    overflow is written into the float64 reference by hand (the oracle's sum
    is finite in float64)."""
    M, N, K = mnk
    rng = np.random.default_rng(33)
    a = rng.choice([-1.0, 1.0], (M, K)) * np.exp2(rng.integers(-8, 9, size=(M, 1)))
    a[:, :32] = np.abs(a[:, :32])
    b = rng.integers(-4, 5, (N, K)).astype(np.float64)
    b[:, :32] = rng.integers(1, 5, (N, 32))
    aq, as_ = mx_operand(a, "e4m3")
    bq, bs = mx_operand(b, "e4m3")
    m0, m1 = 5, M - 40
    as_ = as_.copy()
    as_[m0, 0] = 0xFF
    as_[m1, 0] = 0xFE
    ref = og.reference(aq, as_, bq, bs, F.E4M3)
    assert np.isnan(ref[m0]).all() and np.isfinite(np.delete(ref, [m0], axis=0)).all()
    assert (np.abs(ref[m1]) > 2.0 ** 128).all()
    ref[m1] = np.inf
    want = omx.quantize(ref, FMTS[out_fmt], omx.DUAL, omx.FLOOR)
    cq, cs, cqT, csT = run_mx_out(lib, aq, as_, bq, bs, "e4m3", out_fmt, "floor", layout, "dual")
    for m in (m0, m1):
        assert (cs[m] == 0xFF).all() and (want["s_row"][m] == 0xFF).all()
        assert (cq[m] == 0).all()
        assert (csT[:, m // 32] == 0xFF).all() and (want["s_col"][:, m // 32] == 0xFF).all()
    assert_bytes_equal(cq, want["q_row"], "codes")
    assert_bytes_equal(cs, want["s_row"], "scales")
    assert_bytes_equal(cqT, want["q_col"], "column-block codes")
    assert_bytes_equal(csT, want["s_col"], "column-block scales")


@pytest.mark.parametrize("fa,fb", [("e4m3", "e2m1"), ("e2m1", "e4m3")])
@pytest.mark.parametrize("mnk", [(128, 256, 512), (256, 512, 384)])
def test_mx_output_exact_fp8_x_fp4(lib, fa, fb, mnk):
    """The MX output of a mixed MXFP8 x MXFP4 product: A = +-2^j per row and
    B = integers in [-4, 4] are exact in E4M3 and in E2M1 alike, every sum is
    exact in float32, so the row and column blocks must equal the oracle's
    quantization of the float64 product bit for bit."""
    M, N, K = mnk
    rng = np.random.default_rng(23)
    a = rng.choice([-1.0, 1.0], (M, K)) * np.exp2(rng.integers(-8, 9, size=(M, 1)))
    b = rng.integers(-4, 5, (N, K)).astype(np.float64)
    fmts = {"e4m3": F.E4M3, "e2m1": F.E2M1}
    ra = omx.quantize(a, fmts[fa], omx.ROW, omx.FLOOR)
    rb = omx.quantize(b, fmts[fb], omx.ROW, omx.FLOOR)
    aq, as_, bq, bs = ra["q_row"], ra["s_row"], rb["q_row"], rb["s_row"]
    ref = og.reference(aq, as_, bq, bs, fmts[fa], fmts[fb])
    assert np.array_equal(ref, a @ b.T)                          # the operands quantize exactly
    want = omx.quantize(ref, F.E4M3, omx.DUAL, omx.FLOOR)
    out = lib.mx_gemm_mx_out(t(aq), t(omx.sf_to_mma(as_)), t(bq), t(omx.sf_to_mma(bs)), fa, b_fmt=fb,
                             out_fmt="e4m3", out_scale_mode="floor", out_sf_layout="canonical",
                             orientation="dual")
    cq, cs, cqT, csT = (x.cpu().numpy() for x in out)
    assert_bytes_equal(cq, want["q_row"], "codes")
    assert_bytes_equal(cs, want["s_row"], "scales")
    assert_bytes_equal(cqT, want["q_col"], "column-block codes")
    assert_bytes_equal(csT, want["s_col"], "column-block scales")


@pytest.mark.parametrize("orientation", ["row", "col", "dual"])
@pytest.mark.parametrize("layout", ["canonical", "mma"])
@pytest.mark.parametrize("mnk", [(128, 256, 256), (256, 512, 512)])
def test_mx_output_exact_mxfp4_operands(lib, orientation, layout, mnk):
    """The MX output of an MXFP4 x MXFP4 product (kind::mxf4): A = +-2^j per
    row and B = integers in [-4, 4] are exact in E2M1, every sum is exact in
    float32, so the output blocks equal the oracle's quantization of the
    float64 product bit for bit, on the single-CTA kernel (M = 128) and the
    CTA pair."""
    M, N, K = mnk
    rng = np.random.default_rng(29)
    a = rng.choice([-1.0, 1.0], (M, K)) * np.exp2(rng.integers(-8, 9, size=(M, 1)))
    b = rng.integers(-4, 5, (N, K)).astype(np.float64)
    ra = omx.quantize(a, F.E2M1, omx.ROW, omx.FLOOR)
    rb = omx.quantize(b, F.E2M1, omx.ROW, omx.FLOOR)
    aq, as_, bq, bs = ra["q_row"], ra["s_row"], rb["q_row"], rb["s_row"]
    ref = og.reference(aq, as_, bq, bs, F.E2M1)
    assert np.array_equal(ref, a @ b.T)                          # the operands quantize exactly
    want = omx.quantize(ref, F.E4M3, omx.DUAL, omx.FLOOR)
    cq, cs, cqT, csT = run_mx_out(lib, aq, as_, bq, bs, "e2m1", "e4m3", "floor", layout, orientation)
    if orientation in ("row", "dual"):
        assert_bytes_equal(cq, want["q_row"], "codes")
        assert_bytes_equal(cs, want["s_row"], "scales")
    if orientation in ("col", "dual"):
        assert_bytes_equal(cqT, want["q_col"], "column-block codes")
        assert_bytes_equal(csT, want["s_col"], "column-block scales")


@pytest.mark.parametrize("layout", ["canonical", "mma"])
@pytest.mark.parametrize("mnk", [(128, 256, 256), (256, 512, 512)])
def test_mxfp4_output_exact_and_feeds_the_next_mxfp4_gemm(lib, layout, mnk):
    """MXFP4 x MXFP4 product written as MX E2M1 row and column blocks
    (format-aware fusion for FP4): bit for bit the oracle's quantization of
    the exact float64 product; the MMA-layout row output is then the A
    operand of a second MXFP4 product, checked against the oracle too."""
    M, N, K = mnk
    rng = np.random.default_rng(31)
    a = rng.choice([-1.0, 1.0], (M, K)) * np.exp2(rng.integers(-8, 9, size=(M, 1)))
    b = rng.integers(-4, 5, (N, K)).astype(np.float64)
    ra = omx.quantize(a, F.E2M1, omx.ROW, omx.FLOOR)
    rb = omx.quantize(b, F.E2M1, omx.ROW, omx.FLOOR)
    aq, as_, bq, bs = ra["q_row"], ra["s_row"], rb["q_row"], rb["s_row"]
    ref = og.reference(aq, as_, bq, bs, F.E2M1)
    assert np.array_equal(ref, a @ b.T)
    want = omx.quantize(ref, F.E2M1, omx.DUAL, omx.FLOOR)
    cq, cs, cqT, csT = run_mx_out(lib, aq, as_, bq, bs, "e2m1", "e2m1", "floor", layout, "dual")
    assert_bytes_equal(cq, want["q_row"], "E2M1 codes")
    assert_bytes_equal(cs, want["s_row"], "scales")
    assert_bytes_equal(cqT, want["q_col"], "E2M1 column-block codes")
    assert_bytes_equal(csT, want["s_col"], "column-block scales")
    if layout == "mma" and N % 256 == 0:
        # the row output [M][N] is the next product's A operand (K' = N)
        N2 = 256
        b2 = rng.integers(-2, 3, (N2, N)).astype(np.float64)
        r2 = omx.quantize(b2, F.E2M1, omx.ROW, omx.FLOOR)
        out = lib.mx_gemm_mx_out(t(aq), t(omx.sf_to_mma(as_)), t(bq), t(omx.sf_to_mma(bs)), "e2m1",
                                 out_fmt="e2m1", out_scale_mode="floor", out_sf_layout="mma", orientation="row")
        c2 = lib.mx_gemm(out[0], out[1], t(r2["q_row"]), t(omx.sf_to_mma(r2["s_row"])), "e2m1", torch.float32)
        ref2 = og.reference(want["q_row"], want["s_row"], r2["q_row"], r2["s_row"], F.E2M1)
        assert og.gate_error(c2.cpu().numpy().astype(np.float64), ref2, out_is_bf16=False) <= 1e-5


def test_mx_output_e2m1_random_within_one_step(lib):
    """Random MXFP8 operands, E2M1 output: scales within one binade of the
    oracle's quantization of the float64 product, and at least 99 % of the
    codes identical (decisions differ only at rounding boundaries)."""
    M, N, K = 256, 512, 1024
    a = f64(inputs.activations(M, K, seed=0))
    b = f64(inputs.weights(N, K, seed=4))
    aq, as_ = mx_operand(a, "e4m3")
    bq, bs = mx_operand(b, "e4m3")
    ref = og.reference(aq, as_, bq, bs, F.E4M3)
    want = omx.quantize(ref, F.E2M1, omx.DUAL, omx.FLOOR)
    cq, cs, cqT, csT = run_mx_out(lib, aq, as_, bq, bs, "e4m3", "e2m1", "floor", "canonical", "dual")
    for got_q, got_s, wq, ws in ((cq, cs, want["q_row"], want["s_row"]), (cqT, csT, want["q_col"], want["s_col"])):
        assert np.max(np.abs(got_s.astype(int) - ws.astype(int))) <= 1
        gn = F.unpack_fp4(got_q)
        wn = F.unpack_fp4(wq)
        assert np.mean(gn == wn) >= 0.99


def e4m3_spacing(y):
    """Grid spacing of E4M3 at magnitude y (3 mantissa bits; subnormal step 2^-9)."""
    a = np.abs(y)
    safe = np.where(a >= 2.0 ** -6, a, 1.0)
    return np.where(a >= 2.0 ** -6, np.exp2(np.floor(np.log2(safe)) - 3), 2.0 ** -9)


@pytest.mark.parametrize("mnk", [(256, 512, 1024), (384, 256, 2048)])
def test_mx_output_random_within_one_step(lib, mnk):
    """Random activations x weights: the kernel quantizes its float32
    accumulator, the oracle the float64 product, so decisions may differ
    where a value sits on a rounding or binade boundary.  Scales differ by
    at most one binade; where they agree the element codes differ by at most
    one grid step; elsewhere the dequantized values differ by at most one
    top-binade step; and at least 99 % of the codes are equal."""
    M, N, K = mnk
    a = f64(inputs.activations(M, K, seed=0))
    b = f64(inputs.weights(N, K, seed=4))
    aq, as_ = mx_operand(a, "e4m3")
    bq, bs = mx_operand(b, "e4m3")
    ref = og.reference(aq, as_, bq, bs, F.E4M3)
    want = omx.quantize(ref, F.E4M3, omx.ROW, omx.FLOOR)
    cq, cs, _, _ = run_mx_out(lib, aq, as_, bq, bs, "e4m3", "e4m3", "floor", "canonical")
    ek = cs.astype(int) - 127
    eo = want["s_row"].astype(int) - 127
    assert np.max(np.abs(ek - eo)) <= 1
    same = np.repeat(ek == eo, 32, axis=1)
    yk = F.decode(F.E4M3, cq)
    yo = F.decode(F.E4M3, want["q_row"])
    tol = e4m3_spacing(np.maximum(np.abs(yk), np.abs(yo)))
    assert np.all(np.abs(yk - yo)[same] <= tol[same])
    dk = omx.dequantize(cq, cs, F.E4M3)
    do = omx.dequantize(want["q_row"], want["s_row"], F.E4M3)
    top = np.repeat(np.exp2(np.maximum(ek, eo) + 5.0), 32, axis=1)
    assert np.all(np.abs(dk - do)[~same] <= top[~same])
    assert np.mean(cq == want["q_row"]) >= 0.99


def test_mx_output_feeds_the_next_gemm(lib):
    """Producer writes its consumer's layout: the MMA-layout output of one
    GEMM is the A operand of the next, with no conversion in between."""
    M, N, K, N2 = 256, 512, 512, 256
    rng = np.random.default_rng(22)
    a = rng.choice([-1.0, 1.0], (M, K))
    b = rng.integers(-2, 3, (N, K)).astype(np.float64)
    w = rng.choice([-1.0, 1.0], (N2, N))
    aq, as_ = mx_operand(a, "e4m3")
    bq, bs = mx_operand(b, "e4m3")
    wq, ws = mx_operand(w, "e4m3")
    cq, cs, _, _ = lib.mx_gemm_mx_out(t(aq), t(omx.sf_to_mma(as_)), t(bq), t(omx.sf_to_mma(bs)), "e4m3",
                                      out_sf_layout="mma")
    d = lib.mx_gemm(cq, cs, t(wq), t(omx.sf_to_mma(ws)), "e4m3", torch.float32)
    c_ref = omx.quantize(a @ b.T, F.E4M3, omx.ROW, omx.FLOOR)
    d_ref = og.reference(c_ref["q_row"], c_ref["s_row"], wq, ws, F.E4M3)
    assert og.gate_error(d.cpu().numpy().astype(np.float64), d_ref, out_is_bf16=False) <= 1e-5


# ---------------------------------------------------------------- mm_fp8
def fp8_codes(x, fmt):
    return F.encode_rne_sat(FMTS[fmt], x)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("mnk", [(128, 256, 256), (256, 512, 512)])
def test_mm_fp8_one_hot_rows_exact(lib, fmt, mnk):
    """One-hot A rows pick B's columns; with scale 0.5 and no bias every
    output is an FP8 value times 0.5, exact in bf16."""
    M, N, K = mnk
    rng = np.random.default_rng(23)
    a8 = np.zeros((M, K), dtype=np.uint8)
    a8[np.arange(M), rng.integers(0, K, M)] = fp8_codes(np.array([1.0]), fmt)[0]
    b8 = fp8_codes(rng.standard_normal((N, K)) * 8, fmt)
    scale = torch.tensor([0.5], dtype=torch.float32, device=dev)
    c = lib.mm_fp8(t(a8), t(b8), scale, trans_b=True, fmt=fmt)
    ref = og.mm_fp8_reference(a8, b8, FMTS[fmt], 0.5)
    assert np.array_equal(c.float().cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("shape", [(1, 256, 512, 1024), (3, 256, 256, 512), (2, 128, 384, 256)])
@pytest.mark.parametrize("b_batched", [False, True])
def test_mm_fp8_gate_with_bias_and_batches(lib, fmt, shape, b_batched):
    batch, M, N, K = shape
    rng = np.random.default_rng(24)
    a8 = fp8_codes(rng.standard_normal((batch, M, K)), fmt)
    b8 = fp8_codes(rng.standard_normal((batch, N, K) if b_batched else (N, K)) * 2, fmt)
    bias = inputs.to_bf16(rng.standard_normal(N).astype(np.float32))
    sc = np.float32(0.0123)
    scale = torch.tensor([sc], dtype=torch.float32, device=dev)
    c = lib.mm_fp8(t(a8), t(b8).transpose(-1, -2), scale, bias=bias.to(dev), fmt=fmt)
    ref = og.mm_fp8_reference(a8, b8, FMTS[fmt], float(sc), f64(bias))
    got = c.float().cpu().numpy().astype(np.float64)
    assert got.shape == ref.shape
    assert og.gate_error(got, ref) <= 2e-3


def test_mm_fp8_more_tiles_than_pairs(lib):
    """4 x 2048 x 2048 outputs are 256 tiles of 256 x 256, more than the CTA
    pairs, so each pair alternates between its two accumulators."""
    rng = np.random.default_rng(26)
    batch, M, N, K = 4, 2048, 2048, 256
    a8 = fp8_codes(rng.standard_normal((batch, M, K)), "e4m3")
    b8 = fp8_codes(rng.standard_normal((N, K)), "e4m3")
    bias = inputs.to_bf16(rng.standard_normal(N).astype(np.float32))
    scale = torch.tensor([0.5], dtype=torch.float32, device=dev)
    c = lib.mm_fp8(t(a8), t(b8), scale, trans_b=True, bias=bias.to(dev), fmt="e4m3")
    ref = og.mm_fp8_reference(a8, b8, F.E4M3, 0.5, f64(bias))
    assert og.gate_error(c.float().cpu().numpy().astype(np.float64), ref) <= 2e-3


def _stored(x, trans):
    """The operand as the library reads it: x itself, or the transpose of a
    row-major copy of x^T (the same matrix, other-axis contiguous)."""
    if not trans:
        return t(x)
    return t(np.ascontiguousarray(np.swapaxes(x, -1, -2))).transpose(-1, -2)


@pytest.mark.parametrize("a_mn", [False, True])
@pytest.mark.parametrize("b_mn", [False, True])
@pytest.mark.parametrize("mnk", [(128, 384, 256), (256, 512, 512), (384, 256, 384)])
def test_mm_fp8_every_layout_one_hot_exact(lib, a_mn, b_mn, mnk):
    """Operands K-contiguous or M/N-contiguous (a row-major [K][M] a used as
    a^T, a row-major [K][N] b), read in place: one-hot rows of op(a) pick
    columns of op(b) exactly, on the CTA-pair kernel (M, N multiples of 256)
    and the single-CTA one (the other shapes)."""
    M, N, K = mnk
    rng = np.random.default_rng(31)
    a8 = np.zeros((M, K), dtype=np.uint8)
    a8[np.arange(M), rng.integers(0, K, M)] = fp8_codes(np.array([1.0]), "e4m3")[0]
    b8 = fp8_codes(rng.standard_normal((N, K)) * 8, "e4m3")            # logical B^T [N][K]
    scale = torch.tensor([0.5], dtype=torch.float32, device=dev)
    A = _stored(a8, a_mn)                                                  # op(a) [M][K]
    B = _stored(b8, b_mn).transpose(-1, -2)                            # op(b) [K][N]
    assert (A.stride(-2) == 1) == a_mn and (B.stride(-1) == 1) == b_mn
    c = lib.mm_fp8(A, B, scale, fmt="e4m3")
    ref = og.mm_fp8_reference(a8, b8, F.E4M3, 0.5)
    assert np.array_equal(c.float().cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("a_mn", [False, True])
@pytest.mark.parametrize("b_mn", [False, True])
@pytest.mark.parametrize("shape,a_batched,b_batched", [((2, 256, 512, 384), True, False),
                                                       ((3, 256, 256, 256), True, True),
                                                       ((2, 128, 256, 256), False, True),
                                                       ((1, 512, 768, 1024), True, True)])
def test_mm_fp8_every_layout_gate(lib, fmt, a_mn, b_mn, shape, a_batched, b_batched):
    """Random FP8 operands in all four layouts, batched or broadcast, with
    bias: within the GEMM gate of the float64 product."""
    batch, M, N, K = shape
    rng = np.random.default_rng(32)
    a8 = fp8_codes(rng.standard_normal((batch, M, K) if a_batched else (M, K)), fmt)
    b8 = fp8_codes(rng.standard_normal((batch, N, K) if b_batched else (N, K)) * 2, fmt)
    bias = inputs.to_bf16(rng.standard_normal(N).astype(np.float32))
    sc = np.float32(0.0371)
    scale = torch.tensor([sc], dtype=torch.float32, device=dev)
    A = _stored(a8, a_mn)
    B = _stored(b8, b_mn).transpose(-1, -2)
    c = lib.mm_fp8(A, B, scale, bias=bias.to(dev), fmt=fmt)
    a_full = np.broadcast_to(a8, (batch, M, K))
    b_full = np.broadcast_to(b8, (batch, N, K))
    ref = og.mm_fp8_reference(a_full, b_full, FMTS[fmt], float(sc), f64(bias))
    got = c.float().cpu().numpy().astype(np.float64).reshape(ref.shape)
    assert og.gate_error(got, ref) <= 2e-3


def test_mm_fp8_trans_flags_and_bad_layouts(lib):
    """trans_a / trans_b transpose the stored operands (AstrAI mm_fp8
    semantics); a strided slice that is neither layout raises."""
    rng = np.random.default_rng(25)
    a8 = t(fp8_codes(rng.standard_normal((256, 512)), "e4m3"))             # [M][K]
    w8 = t(fp8_codes(rng.standard_normal((384, 512)), "e4m3"))             # [N][K]
    scale = torch.tensor([1.0], dtype=torch.float32, device=dev)
    c1 = lib.mm_fp8(a8, w8, scale, trans_b=True)
    c2 = lib.mm_fp8(a8, w8.t(), scale)
    c3 = lib.mm_fp8(a8, w8.t().contiguous(), scale)                        # b stored [K][N]
    c4 = lib.mm_fp8(a8.t().contiguous(), w8.t().contiguous(), scale, trans_a=True)
    assert torch.equal(c1, c2)
    ref = og.mm_fp8_reference(np_(a8), np_(w8), F.E4M3, 1.0)
    for c in (c1, c3, c4):
        assert og.gate_error(c.float().cpu().numpy().astype(np.float64), ref) <= 2e-3
    big = t(fp8_codes(rng.standard_normal((256, 1024)), "e4m3"))
    with pytest.raises(ValueError):
        lib.mm_fp8(big[:, ::2], w8, scale, trans_b=True)                   # every other column


# ---------------------------------------------------------------- full sizes, sampled
def _rows(n, k, seed):
    return np.sort(np.random.default_rng(seed).choice(n, k, replace=False))


def test_full_size_mx_output_sampled(lib):
    """8192 x 4096 activations times 4096 x 4096 weights (MXFP8 E4M3), as the
    bench runs it, with row and column-block E4M3 outputs: sampled output
    rows and output columns against the oracle's MX quantization of the
    float64 product (the property bar of the random test)."""
    M, N, K = 8192, 4096, 4096
    a = f64(inputs.activations(M, K, seed=0))
    b = f64(inputs.weights(N, K, seed=4))
    aq, as_ = mx_operand(a, "e4m3")
    bq, bs = mx_operand(b, "e4m3")
    cq, cs, cqT, csT = run_mx_out(lib, aq, as_, bq, bs, "e4m3", "e4m3", "floor", "mma", "dual")
    rows = _rows(M, 16, 1)
    ref = og.reference_rows_cols(aq, as_, bq, bs, F.E4M3, rows, np.arange(N))
    want = omx.quantize(ref, F.E4M3, omx.ROW, omx.FLOOR)
    assert np.max(np.abs(cs[rows].astype(int) - want["s_row"].astype(int))) <= 1
    assert np.mean(cq[rows] == want["q_row"]) >= 0.99
    # column blocks: 32-row groups of sampled output columns
    cols = _rows(N, 8, 2)
    groups = _rows(M // 32, 8, 3)
    rr = (groups[:, None] * 32 + np.arange(32)[None, :]).reshape(-1)
    refc = og.reference_rows_cols(aq, as_, bq, bs, F.E4M3, rr, cols)          # [8*32][8]
    wantc = omx.quantize(refc.T.reshape(len(cols), len(groups), 32).reshape(len(cols), -1), F.E4M3, omx.ROW,
                         omx.FLOOR)
    got_codes = cqT[cols][:, rr]
    got_scales = csT[cols][:, groups]
    assert np.max(np.abs(got_scales.astype(int) - wantc["s_row"].astype(int))) <= 1
    assert np.mean(got_codes == wantc["q_row"]) >= 0.99


def test_full_size_mx_row_output_sampled(lib):
    """The bench's MX E4M3 row-output product at full size (the rows-only
    kernel variant): sampled output rows against the oracle's MX
    quantization of the float64 product (the property bar)."""
    M, N, K = 8192, 4096, 4096
    a = f64(inputs.activations(M, K, seed=0))
    b = f64(inputs.weights(N, K, seed=4))
    aq, as_ = mx_operand(a, "e4m3")
    bq, bs = mx_operand(b, "e4m3")
    cq, cs, cqT, _ = run_mx_out(lib, aq, as_, bq, bs, "e4m3", "e4m3", "floor", "mma", "row")
    assert cqT is None
    rows = _rows(M, 16, 12)
    ref = og.reference_rows_cols(aq, as_, bq, bs, F.E4M3, rows, np.arange(N))
    want = omx.quantize(ref, F.E4M3, omx.ROW, omx.FLOOR)
    assert np.max(np.abs(cs[rows].astype(int) - want["s_row"].astype(int))) <= 1
    assert np.mean(cq[rows] == want["q_row"]) >= 0.99


def test_full_size_mxfp4_e2m1_output_sampled(lib):
    """The bench's MXFP4 product with MX E2M1 output (4096 x 14336 gradient
    times 4096 x 14336 operand, MMA-layout scales): sampled output rows
    against the oracle's E2M1 quantization of the float64 product."""
    M, N, K = 4096, 4096, 14336
    a = f64(inputs.heavy_gradient(M, K, seed=6))
    b = f64(inputs.fp4_operand(N, K, seed=8))
    aq, as_ = mx_operand(a, "e2m1")
    bq, bs = mx_operand(b, "e2m1")
    cq, cs, _, _ = run_mx_out(lib, aq, as_, bq, bs, "e2m1", "e2m1", "floor", "mma", "row")
    assert cq.shape == (M, N // 2)
    rows = _rows(M, 16, 13)
    ref = og.reference_rows_cols(aq, as_, bq, bs, F.E2M1, rows, np.arange(N))
    want = omx.quantize(ref, F.E2M1, omx.ROW, omx.FLOOR)
    assert np.max(np.abs(cs[rows].astype(int) - want["s_row"].astype(int))) <= 1
    assert np.mean(F.unpack_fp4(cq[rows]) == F.unpack_fp4(want["q_row"])) >= 0.99


@pytest.mark.parametrize("kn", [False, True])
def test_full_size_mm_fp8_sampled(lib, kn):
    """The bench's per-tensor FP8 products at full size and launch
    configuration: 8192 x 4096 E4M3 operand times a 4096 x 4096 weight with
    bias, the weight stored [N][K] (transposed view) or [K][N] (the default
    layout, read N-contiguous); sampled rows and columns within the gate."""
    M, N, K = 8192, 4096, 4096
    rng = np.random.default_rng(27)
    # seeded finite E4M3 codes (every code but the NaN patterns 0x7F / 0xFF)
    x8n = (rng.integers(0, 0x7F, (M, K), dtype=np.uint8) | (rng.integers(0, 2, (M, K), dtype=np.uint8) << 7))
    w8n = (rng.integers(0, 0x7F, (N, K), dtype=np.uint8) | (rng.integers(0, 2, (N, K), dtype=np.uint8) << 7))
    bias = inputs.weights(1, N, seed=9).reshape(N)
    sc = torch.tensor([0.75], dtype=torch.float32, device=dev)
    if kn:
        c = lib.mm_fp8(t(x8n), t(w8n.T), sc, bias=bias.to(dev), fmt="e4m3").float().cpu().numpy()
    else:
        c = lib.mm_fp8(t(x8n), t(w8n), sc, trans_b=True, bias=bias.to(dev), fmt="e4m3").float().cpu().numpy()
    rows, cols = _rows(M, 64, 4), _rows(N, 64, 5)
    ref = og.mm_fp8_reference(x8n[rows], w8n[cols], F.E4M3, 0.75, f64(bias)[cols])
    assert og.gate_error(c[np.ix_(rows, cols)].astype(np.float64), ref) <= 2e-3


def test_device_status_clean_after_epilogues(lib):
    assert lib.last_device_status() == 0
