"""Failure detection on the GPU without a fault: a test hook leaves one
pipeline barrier phase incomplete, so a bounded wait expires (about one
second); the kernel records MXQ_ERR_TIMEOUT and winds down; the context stays
usable and the next calls are exact again."""

import numpy as np
import pytest
import torch

from block_scaled_precision_02_gb300 import inputs
from oracle import formats as F
from oracle import gemm as og
from oracle import mx as omx
from tests.helpers import assert_bytes_equal, f64, np_

pytestmark = pytest.mark.gpu

MXQ_ERR_TIMEOUT = -6


def test_quantizer_wait_expires_and_context_survives(lib):
    L = lib.load()
    dev = torch.device("cuda")
    x = inputs.activations(512, 512, seed=3)
    assert lib.last_device_status() == 0
    assert L.mxq_test_stall_next_launch(1) == 0
    lib.mx_quantize(x.to(dev), "e4m3", "dual", "floor")       # launches; one stage never lands
    assert lib.last_device_status() == MXQ_ERR_TIMEOUT
    assert lib.last_device_status() == 0                        # read clears it
    out = lib.mx_quantize(x.to(dev), "e4m3", "dual", "floor")
    ref = omx.quantize(f64(x), F.E4M3, omx.DUAL, omx.FLOOR)
    assert_bytes_equal(np_(out[0]), ref["q_row"], "q_row after recovery")
    assert_bytes_equal(np_(out[2]), ref["q_col"], "q_col after recovery")
    assert lib.last_device_status() == 0


def test_column_only_wait_expires_and_context_survives(lib):
    """A column-only launch splits each CTA's tiles between two warp groups
    (even and odd tiles, each on its own stages).  With one group's first
    stage never landing, that group times out, the other group's tiles and
    the loads still in flight end normally, the status reads TIMEOUT, and
    the next call is exact.  4096 x 4096 gives every CTA many tiles."""
    L = lib.load()
    dev = torch.device("cuda")
    x = inputs.activations(4096, 4096, seed=3)
    xd = x.to(dev)
    assert lib.last_device_status() == 0
    assert L.mxq_test_stall_next_launch(1) == 0
    lib.mx_quantize(xd, "e4m3", "col", "floor")
    assert lib.last_device_status() == MXQ_ERR_TIMEOUT
    out = lib.mx_quantize(xd, "e4m3", "col", "floor")
    for r0 in (0, 2048, 3840):                       # 256-row slabs: their column blocks
        ref = omx.quantize(f64(x)[r0:r0 + 256], F.E4M3, omx.COL, omx.FLOOR)
        assert_bytes_equal(np_(out[2])[:, r0:r0 + 256], ref["q_col"], f"q_col after recovery, rows {r0}+")
        assert_bytes_equal(np_(out[3])[:, r0 // 32:r0 // 32 + 8], ref["s_col"], f"s_col after recovery, rows {r0}+")
    assert lib.last_device_status() == 0


def test_gemm_wait_expires_and_context_survives(lib):
    L = lib.load()
    dev = torch.device("cuda")
    a = omx.quantize(f64(inputs.activations(256, 512, seed=0)), F.E4M3, omx.ROW)
    b = omx.quantize(f64(inputs.weights(256, 512, seed=4)), F.E4M3, omx.ROW)
    t = lambda v: torch.from_numpy(np.ascontiguousarray(v)).to(dev)
    args = (t(a["q_row"]), t(omx.sf_to_mma(a["s_row"])), t(b["q_row"]), t(omx.sf_to_mma(b["s_row"])), "e4m3")
    assert L.mxq_test_stall_next_launch(2) == 0
    lib.mx_gemm(*args)
    assert lib.last_device_status() == MXQ_ERR_TIMEOUT
    c = lib.mx_gemm(*args)
    ref = og.reference(a["q_row"], a["s_row"], b["q_row"], b["s_row"], F.E4M3)
    assert og.gate_error(c.float().cpu().numpy(), ref) <= 2e-3
    assert lib.last_device_status() == 0


def test_disarm(lib):
    L = lib.load()
    assert L.mxq_test_stall_next_launch(1) == 0
    assert L.mxq_test_stall_next_launch(0) == 0
    assert L.mxq_test_stall_next_launch(7) == -1
    x = inputs.activations(128, 128, seed=1).cuda()
    lib.mx_quantize(x, "e4m3", "row", "floor")
    assert lib.last_device_status() == 0
