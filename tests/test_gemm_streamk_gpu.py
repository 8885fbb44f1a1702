"""GPU parity of the stream-K schedule of the block-scaled GEMM
(mxq_gemm_ws): shapes whose 256 x 256 tiles do not fill whole waves of the
GPU's CTA pairs, so the last tiles are cut into k-ranges and finished by
adding the parked float32 sums of the other piece.  Every output is checked
against the oracle: bit for bit where the products are exact, within the
gate elsewhere; the schedule is also checked to agree with the plain one
within float32 rounding and to repeat bit for bit."""

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
dev = torch.device("cuda")


def t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def operand(x, fmt):
    r = omx.quantize(x, FMTS[fmt], omx.ROW, omx.FLOOR)
    return r["q_row"], r["s_row"]


def pairs_on_device():
    # the pair kernel runs one 2-CTA cluster per two SMs at most
    return torch.cuda.get_device_properties(dev).multi_processor_count // 2


def run(lib, aq, as_, bq, bs, fa, fb, stream_k, out_dtype=torch.bfloat16):
    c = lib.mx_gemm(t(aq), t(omx.sf_to_mma(as_)), t(bq), t(omx.sf_to_mma(bs)), fa, out_dtype, b_fmt=fb,
                    stream_k=stream_k)
    return c.float().cpu().numpy().astype(np.float64)


def shape_with_tail(waves):
    """(M, N): 256 x 256 tiles = `waves` full waves of CTA pairs plus a
    sparse last one (eight tiles), the case the stream-K schedule takes."""
    p = pairs_on_device()
    nt_n = 8
    nt_m = -(-(waves * p + 8) // nt_n)
    assert 0 < nt_m * nt_n - waves * p <= p // 4
    return 256 * nt_m, 256 * nt_n


@pytest.mark.parametrize("fa,fb", [("e4m3", "e4m3"), ("e5m2", "e5m2"), ("e2m1", "e2m1"), ("e4m3", "e2m1")])
def test_stream_k_unit_rows_exact(lib, fa, fb):
    """One non-zero per B row: every output is one dequantized A entry, exact
    whichever piece of a cut tile holds it."""
    M, N = shape_with_tail(1)
    K = 512
    rng = np.random.default_rng(3)
    a = rng.standard_normal((M, K)) * np.exp2(rng.integers(-6, 6, size=(M, K // 32))).repeat(32, 1)
    aq, as_ = operand(a, fa)
    perm = rng.integers(0, K, N)
    b = np.zeros((N, K))
    b[np.arange(N), perm] = np.exp2(rng.integers(-3, 4, N))
    bq, bs = operand(b, fb)
    ref = og.reference(aq, as_, bq, bs, FMTS[fa], FMTS[fb])
    got = run(lib, aq, as_, bq, bs, fa, fb, True, torch.float32)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("fa,fb,K", [("e4m3", "e4m3", 1024), ("e5m2", "e4m3", 640), ("e2m1", "e2m1", 1536),
                                     ("e4m3", "e2m1", 768)])
@pytest.mark.parametrize("waves", [1, 2])
def test_stream_k_gate_and_agreement(lib, fa, fb, K, waves):
    M, N = shape_with_tail(waves)
    a = f64(inputs.activations(M, K, seed=0))
    b = f64(inputs.weights(N, K, seed=4) if fb != "e2m1" else inputs.fp4_operand(N, K, seed=8))
    aq, as_ = operand(a, fa)
    bq, bs = operand(b, fb)
    ref = og.reference(aq, as_, bq, bs, FMTS[fa], FMTS[fb])
    sk = run(lib, aq, as_, bq, bs, fa, fb, True)
    assert og.gate_error(sk, ref) <= 2e-3
    # the float32 sums of a cut tile are added once more: within a few
    # float32 roundings of the plain schedule's float32 output
    sk32 = run(lib, aq, as_, bq, bs, fa, fb, True, torch.float32)
    plain32 = run(lib, aq, as_, bq, bs, fa, fb, False, torch.float32)
    scale = np.maximum(np.abs(plain32), np.sqrt(np.mean(plain32 ** 2)))
    assert np.max(np.abs(sk32 - plain32) / scale) <= 1e-5
    if "e2m1" not in (fa, fb):
        # 8-bit products round in float32: the cut tiles, summed in two
        # pieces, differ somewhere (E2M1 products here are exact either way)
        assert not np.array_equal(sk32, plain32)
    assert og.gate_error(sk32, ref, out_is_bf16=False) <= 1e-5
    # the same launch again: identical bits
    assert np.array_equal(run(lib, aq, as_, bq, bs, fa, fb, True, torch.float32), sk32)


def test_full_size_sparse_tail_sampled(lib):
    """The bench's sparse-tail product at full size: 2560 x 2048 x 16384
    MXFP8 (80 tiles on the CTA pairs), stream-K and plain schedules.
    Sampled rows and columns within the gate, and the two schedules'
    float32 outputs within a few float32 roundings of each other."""
    M, N, K = 2560, 2048, 16384
    a = f64(inputs.activations(M, K, seed=0))
    b = f64(inputs.weights(N, K, seed=4))
    aq, as_ = operand(a, "e4m3")
    bq, bs = operand(b, "e4m3")
    sk = run(lib, aq, as_, bq, bs, "e4m3", "e4m3", True)
    plain = run(lib, aq, as_, bq, bs, "e4m3", "e4m3", False)
    rng = np.random.default_rng(11)
    rows = np.sort(rng.choice(M, 48, replace=False))
    cols = np.sort(rng.choice(N, 48, replace=False))
    ref = og.reference_rows_cols(aq, as_, bq, bs, F.E4M3, rows, cols)
    assert og.gate_error(sk[np.ix_(rows, cols)], ref) <= 2e-3
    assert og.gate_error(plain[np.ix_(rows, cols)], ref) <= 2e-3
    # Both schedules add K/32 float32 MMA partial sums; splitting the
    # running sum in two changes at most a few roundings per step, each at
    # most 2^-24 of the running sum's size (bounded by the scale below).
    # With K = 16384 that is a looser bound than the 1e-5 of the short-K
    # shapes above.
    sk32 = run(lib, aq, as_, bq, bs, "e4m3", "e4m3", True, torch.float32)
    plain32 = run(lib, aq, as_, bq, bs, "e4m3", "e4m3", False, torch.float32)
    scale = np.maximum(np.abs(plain32), np.sqrt(np.mean(plain32 ** 2)))
    assert np.max(np.abs(sk32 - plain32) / scale) <= 2 * 2.0 ** -24 * (K // 32)


def test_stream_k_without_workspace_is_the_plain_schedule(lib):
    M, N = shape_with_tail(1)
    K = 256
    rng = np.random.default_rng(5)
    aq, as_ = operand(rng.standard_normal((M, K)), "e4m3")
    bq, bs = operand(rng.standard_normal((N, K)), "e4m3")
    A, As, B, Bs = t(aq), t(omx.sf_to_mma(as_)), t(bq), t(omx.sf_to_mma(bs))
    c_plain = lib.mx_gemm(A, As, B, Bs, "e4m3", torch.float32, stream_k=False)
    c_null = torch.empty_like(c_plain)
    L = lib.load()
    st = torch.cuda.current_stream().cuda_stream
    rc = L.mxq_gemm_ws(lib._ptr(A), lib._ptr(As), 0, lib._ptr(B), lib._ptr(Bs), 0, M, N, K, 1, lib._ptr(c_null), 1,
                       None, 0, st)
    assert rc == 0
    c_small = torch.empty_like(c_plain)
    ws = torch.zeros(4096, dtype=torch.uint8, device=dev)
    rc = L.mxq_gemm_ws(lib._ptr(A), lib._ptr(As), 0, lib._ptr(B), lib._ptr(Bs), 0, M, N, K, 1, lib._ptr(c_small), 1,
                       lib._ptr(ws), ws.numel(), st)
    assert rc == 0
    assert torch.equal(c_plain, c_null) and torch.equal(c_plain, c_small)


def test_device_status_clean_after_stream_k(lib):
    assert lib.last_device_status() == 0
