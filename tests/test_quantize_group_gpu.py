"""GPU parity of the grouped MX quantize (mxq_quantize_group): several tensors
of one format and orientation in one launch.  Every job's bytes must equal
the oracle's quantization of that tensor (and so the single-tensor call's),
whatever the mix of shapes, ragged edges and scale modes in the group."""

import numpy as np
import pytest
import torch

from block_scaled_precision_02_gb300 import inputs
from oracle import formats as F
from oracle import mx as omx
from tests.helpers import assert_bytes_equal, f64, np_

pytestmark = pytest.mark.gpu

FMTS = {"e4m3": F.E4M3, "e5m2": F.E5M2, "e2m1": F.E2M1}
ORI = {"row": omx.ROW, "col": omx.COL, "dual": omx.DUAL}
MODE = {"floor": omx.FLOOR, "ceil": omx.CEIL}
dev = torch.device("cuda")


def check_job(out, x, fmt, orient, mode, sf="canonical"):
    qr, sr, qc, sc = [None if t is None else np_(t) for t in out]
    ref = omx.quantize(f64(x), FMTS[fmt], ORI[orient], MODE[mode])
    if ORI[orient] & omx.ROW:
        assert_bytes_equal(qr, ref["q_row"], "q_row")
        s = ref["s_row"] if sf == "canonical" else omx.sf_to_mma(ref["s_row"])
        assert_bytes_equal(sr.reshape(s.shape), s, "s_row")
    else:
        assert qr is None and sr is None
    if ORI[orient] & omx.COL:
        assert_bytes_equal(qc, ref["q_col"], "q_col")
        s = ref["s_col"] if sf == "canonical" else omx.sf_to_mma(ref["s_col"])
        assert_bytes_equal(sc.reshape(s.shape), s, "s_col")
    else:
        assert qc is None and sc is None


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2", "e2m1"])
@pytest.mark.parametrize("orient", ["row", "col", "dual"])
def test_group_of_ragged_shapes_and_mixed_modes(lib, fmt, orient):
    """Four tensors whose tile counts differ (ragged row and column tiles),
    floor and ceil scales mixed: each job bit for bit the oracle's."""
    shapes = [(288, 416), (64, 96), (160, 544), (32, 32)]
    modes = ["floor", "ceil", "ceil", "floor"]
    xs = [inputs.small_rowwise(r, c, seed=20 + k) for k, (r, c) in enumerate(shapes)]
    outs = lib.mx_quantize_group([x.to(dev) for x in xs], fmt, orient, modes)
    assert len(outs) == 4
    for out, x, mode in zip(outs, xs, modes):
        check_job(out, x, fmt, orient, mode)


@pytest.mark.parametrize("n", [1, 2, 3])
def test_smaller_groups_and_mma_layout(lib, n):
    """Groups of one to three tensors, MMA-layout scales."""
    xs = [inputs.activations(256, 384, seed=30 + k) for k in range(n)]
    outs = lib.mx_quantize_group([x.to(dev) for x in xs], "e4m3", "dual", "floor", sf_layout="mma")
    for out, x in zip(outs, xs):
        check_job(out, x, "e4m3", "dual", "floor", sf="mma")


def test_group_equals_single_calls_on_strided_input(lib):
    """A strided view (row stride above the column count) inside a group:
    the same bytes as the single-tensor call and as the oracle."""
    base = inputs.activations(256, 512, seed=41).to(dev)
    view = base[:, :384]
    other = inputs.gradients(128, 256, seed=42).to(dev)
    outs = lib.mx_quantize_group([view, other], "e5m2", "dual", ["ceil", "floor"])
    single = lib.mx_quantize(view, "e5m2", "dual", "ceil")
    for a, b in zip(outs[0], single):
        assert torch.equal(a, b)
    check_job(outs[1], other.cpu(), "e5m2", "dual", "floor")


@pytest.mark.parametrize("fmt,gen,seed", [("e4m3", inputs.activations, 0), ("e5m2", inputs.gradients, 1)])
def test_bench_group_full_size_sampled(lib, fmt, gen, seed):
    """The launches the benchmark times for its headline: the 8192 x 4096
    activations (E4M3) and gradients (E5M2), dual, floor and ceil scales of
    one tensor in one group (two input copies), MMA-layout scales.  Sampled
    rows and 32-row slabs against the oracle, and every byte against the
    single-tensor calls (whose full-size parity is tested on their own)."""
    x = gen(8192, 4096, seed=seed)
    xd = x.to(dev)
    x2 = xd.clone()
    outs = lib.mx_quantize_group([xd, x2], fmt, "dual", ["floor", "ceil"], sf_layout="mma")
    for out, mode in zip(outs, ["floor", "ceil"]):
        single = lib.mx_quantize(xd, fmt, "dual", mode, sf_layout="mma")
        for a, b in zip(out, single):
            assert torch.equal(a, b)
        qr, sr = np_(out[0]), omx.sf_from_mma(np_(out[1]), 8192, 4096 // 32)
        rows = np.sort(np.random.default_rng(5).choice(8192, 48, replace=False))
        ref = omx.quantize(f64(x)[rows], FMTS[fmt], omx.ROW, MODE[mode])
        assert_bytes_equal(qr[rows], ref["q_row"], "q_row sample")
        assert_bytes_equal(sr[rows], ref["s_row"], "s_row sample")
        qc, sc = np_(out[2]), omx.sf_from_mma(np_(out[3]), 4096, 8192 // 32)
        for sl in (3, 200):
            refc = omx.quantize(f64(x)[sl * 32:(sl + 1) * 32], FMTS[fmt], omx.COL, MODE[mode])
            assert_bytes_equal(qc[:, sl * 32:(sl + 1) * 32], refc["q_col"], "q_col slab")
            assert_bytes_equal(sc[:, sl:sl + 1], refc["s_col"], "s_col slab")


def test_group_argument_errors(lib):
    x = inputs.small_rowwise(64, 64, seed=1).to(dev)
    with pytest.raises(ValueError):
        lib.mx_quantize_group([], "e4m3")
    with pytest.raises(ValueError):
        lib.mx_quantize_group([x] * 5, "e4m3")
    with pytest.raises(ValueError):
        lib.mx_quantize_group([x, x], "e4m3", "row", ["floor"])
    bad = inputs.small_rowwise(64, 64, seed=2).to(dev)[:48]           # 48 rows: not a multiple of 32
    with pytest.raises(lib.MXQError):
        lib.mx_quantize_group([x, bad], "e4m3")
    assert lib.last_device_status() == 0
