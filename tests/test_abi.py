"""The C-ABI library builds for sm_103a, loads, exports every entry point that
include/*.h declares, and rejects bad arguments before touching a GPU.
CPU only: no call here launches a kernel."""

import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def so():
    import block_scaled_precision_02_gb300 as mxq
    from block_scaled_precision_02_gb300 import build
    if not os.path.exists(mxq.LIB_PATH):
        build.build()
    return mxq.load()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("defined",)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("mxq_quantize", "mxq_quantize_group", "mxq_dequantize", "fp8_quantize_pertensor", "fp8_ring_fold",
              "mxq_gemm",
              "mxq_gemm_mixed", "mxq_gemm_ws", "mxq_gemm_workspace_size",
              "mxq_gemm_mx_out", "mxq_mm_fp8", "mxq_sf_to_mma",
              "mxq_last_device_status", "mxq_strerror", "mxq_version"):
        assert n in names


def test_library_exports_every_declared_symbol(so):
    for n in declared_functions():
        assert hasattr(so, n), n


def test_strerror_and_version(so):
    for code in range(0, -7, -1):
        assert so.mxq_strerror(code)
    assert so.mxq_version() >= 100


FAKE = ctypes.c_void_p(0x10000)           # 16-byte aligned, never dereferenced
ODD = ctypes.c_void_p(0x10008)
FAKE16 = ctypes.c_void_p(0x10010)         # 16-byte but not 32-byte aligned


def test_argument_checks_need_no_gpu(so):
    q = so.mxq_quantize
    # NULL input, bad format / orientation / scale mode / rounding / layout
    assert q(None, 64, 64, 64, 0, 1, 0, 0, 0, 0, 7, 0, FAKE, FAKE, None, None, None) == -1
    assert q(FAKE, 64, 64, 64, 9, 1, 0, 0, 0, 0, 7, 0, FAKE, FAKE, None, None, None) == -1
    assert q(FAKE, 64, 64, 64, 0, 4, 0, 0, 0, 0, 7, 0, FAKE, FAKE, None, None, None) == -1
    assert q(FAKE, 64, 64, 64, 0, 1, 2, 0, 0, 0, 7, 0, FAKE, FAKE, None, None, None) == -1
    assert q(FAKE, 64, 64, 64, 0, 1, 0, 3, 0, 0, 7, 0, FAKE, FAKE, None, None, None) == -1
    assert q(FAKE, 64, 64, 64, 0, 1, 0, 0, 0, 0, 7, 5, FAKE, FAKE, None, None, None) == -1
    # missing column outputs for DUAL
    assert q(FAKE, 64, 64, 64, 0, 3, 0, 0, 0, 0, 7, 0, FAKE, FAKE, None, None, None) == -1
    # shapes: not multiples of 32, ld < cols, MMA layout needs multiples of 128
    assert q(FAKE, 48, 64, 64, 0, 1, 0, 0, 0, 0, 7, 0, FAKE, FAKE, None, None, None) == -2
    assert q(FAKE, 64, 64, 32, 0, 1, 0, 0, 0, 0, 7, 0, FAKE, FAKE, None, None, None) == -2
    assert q(FAKE, 64, 64, 64, 0, 1, 0, 0, 0, 0, 7, 1, FAKE, FAKE, None, None, None) == -2
    # empty tensors are a shape error, checked before any launch
    assert q(FAKE, 0, 64, 64, 0, 1, 0, 0, 0, 0, 7, 0, FAKE, FAKE, None, None, None) == -2
    assert q(FAKE, 64, 0, 64, 0, 1, 0, 0, 0, 0, 7, 0, FAKE, FAKE, None, None, None) == -2
    assert so.mxq_gemm(FAKE, FAKE, FAKE, FAKE, 0, 128, 128, 0, 1, FAKE, 0, None) == -2
    assert so.mxq_gemm(FAKE, FAKE, FAKE, FAKE, 128, 128, 0, 0, 1, FAKE, 0, None) == -2
    assert so.fp8_quantize_pertensor(FAKE, 0, 64, FAKE, 0, 1, None, 0, 0, 448.0, 1.0, FAKE, None, FAKE, None) == -2
    # misaligned input or leading dimension
    assert q(ODD, 64, 64, 64, 0, 1, 0, 0, 0, 0, 7, 0, FAKE, FAKE, None, None, None) == -3
    assert q(FAKE, 64, 64, 68, 0, 1, 0, 0, 0, 0, 7, 0, FAKE, FAKE, None, None, None) == -3

    p = so.fp8_quantize_pertensor
    assert p(FAKE, 64, 64, FAKE, 2, 1, None, 0, 0, 448.0, 1.0, FAKE, None, FAKE, None) == -1   # E2M1
    assert p(FAKE, 64, 64, FAKE, 0, 1, None, 0, 0, 448.0, 1.0, FAKE, None, None, None) == -1   # no amax sink
    assert p(FAKE, 64, 64, FAKE, 0, 1, FAKE, 16, 16, 448.0, 1.0, FAKE, None, None, None) == -1 # hist_idx
    assert p(FAKE, 64, 40, FAKE, 0, 1, None, 0, 0, 448.0, 1.0, FAKE, None, FAKE, None) == -2
    assert p(FAKE, 40, 64, FAKE, 0, 3, None, 0, 0, 448.0, 1.0, FAKE, FAKE, FAKE, None) == -2

    g = so.mxq_gemm
    assert g(None, FAKE, FAKE, FAKE, 128, 128, 128, 0, 1, FAKE, 0, None) == -1
    assert g(FAKE, FAKE, FAKE, FAKE, 128, 128, 128, 0, 0, FAKE, 0, None) == -4   # canonical scales
    assert g(FAKE, FAKE, FAKE, FAKE, 100, 128, 128, 0, 1, FAKE, 0, None) == -2
    assert g(FAKE, FAKE, FAKE, FAKE, 128, 128, 128, 2, 1, FAKE, 0, None) == -2   # E2M1 needs K % 256
    assert g(ODD, FAKE, FAKE, FAKE, 128, 128, 128, 0, 1, FAKE, 0, None) == -3

    mg = so.mxq_gemm_mixed
    # E2M1 beside an 8-bit operand: K % 128 as for 8-bit pairs, and the E2M1
    # codes 32-byte aligned (a 16-byte aligned pointer is enough for the other)
    assert mg(FAKE, FAKE, 0, FAKE, FAKE, 2, 128, 128, 192, 1, FAKE, 0, None) == -2   # E4M3 x E2M1
    assert mg(FAKE, FAKE, 0, FAKE, FAKE, 2, 128, 128, 128, 1, None, 0, None) == -1   # shape passed; no C
    assert mg(FAKE, FAKE, 0, FAKE16, FAKE, 2, 128, 128, 256, 1, FAKE, 0, None) == -3
    assert mg(FAKE16, FAKE, 2, FAKE, FAKE, 1, 128, 128, 256, 1, FAKE, 0, None) == -3   # E2M1 x E5M2
    assert mg(FAKE16, FAKE, 0, FAKE, FAKE, 2, 128, 128, 256, 1, None, 0, None) == -1   # alignment passed
    assert mg(FAKE, FAKE, 2, FAKE, FAKE, 2, 128, 128, 128, 1, FAKE, 0, None) == -2   # E2M1 x E2M1: K % 256
    assert mg(FAKE, FAKE, 0, FAKE, FAKE, 5, 128, 128, 256, 1, FAKE, 0, None) == -1   # unknown format
    assert mg(FAKE, FAKE, 0, FAKE, FAKE, 1, 100, 128, 256, 1, FAKE, 0, None) == -2
    assert mg(FAKE, FAKE, 0, FAKE, FAKE, 1, 128, 128, 256, 0, FAKE, 0, None) == -4   # canonical scales

    mo = so.mxq_gemm_mx_out
    row = (FAKE, FAKE, None, None)
    assert mo(FAKE, FAKE, 0, FAKE, FAKE, 0, 128, 128, 128, 1, 5, 0, 0, *row, None) == -1   # output format
    assert mo(FAKE, FAKE, 0, FAKE, FAKE, 0, 128, 128, 128, 1, 0, 2, 0, *row, None) == -1   # scale mode
    assert mo(FAKE, FAKE, 0, FAKE, FAKE, 0, 128, 128, 128, 1, 0, 0, 2, *row, None) == -1   # scale layout
    assert mo(FAKE, FAKE, 0, FAKE, FAKE, 0, 128, 128, 128, 1, 0, 0, 0, FAKE, None, None, None, None) == -1
    assert mo(FAKE, FAKE, 0, FAKE, FAKE, 0, 128, 128, 128, 1, 0, 0, 0, None, None, FAKE, None, None) == -1
    assert mo(FAKE, FAKE, 0, FAKE, FAKE, 0, 128, 128, 128, 1, 0, 0, 0, None, None, None, None, None) == -1
    assert mo(FAKE, FAKE, 0, FAKE, FAKE, 0, 128, 128, 128, 1, 0, 0, 0, ODD, FAKE, None, None, None) == -3
    assert mo(FAKE, FAKE, 0, FAKE, FAKE, 0, 128, 128, 128, 1, 0, 0, 0, None, None, FAKE, ODD, None) == -3
    assert mo(FAKE, FAKE, 0, FAKE, FAKE, 0, 128, 100, 128, 1, 0, 0, 0, *row, None) == -2

    mm = so.mxq_mm_fp8
    assert mm(FAKE, FAKE, 1, 128, 128, 128, 0, 0, 0, 1, 2, FAKE, None, FAKE, None) == -4   # E2M1
    assert mm(FAKE, FAKE, 1, 128, 128, 128, 0, 0, 0, 1, 0, None, None, FAKE, None) == -1   # no scale
    assert mm(FAKE, FAKE, 1, 128, 128, 128, 2, 0, 0, 1, 0, FAKE, None, FAKE, None) == -1   # batched flag
    assert mm(FAKE, FAKE, 1, 128, 128, 128, 0, 0, 2, 1, 0, FAKE, None, FAKE, None) == -1   # trans_a flag
    assert mm(FAKE, FAKE, 1, 128, 128, 128, 0, 0, 0, -1, 0, FAKE, None, FAKE, None) == -1  # trans_b flag
    assert mm(FAKE, FAKE, 0, 128, 128, 128, 0, 0, 0, 1, 0, FAKE, None, FAKE, None) == -2   # batch 0
    assert mm(FAKE, FAKE, 1, 100, 128, 128, 0, 0, 1, 0, 0, FAKE, None, FAKE, None) == -2
    assert mm(FAKE, FAKE, 1, 128, 128, 128, 0, 0, 0, 0, 0, FAKE, ODD, FAKE, None) == -3   # bias alignment

    assert so.mxq_gemm_workspace_size(None) == -1
    ws = so.mxq_gemm_ws
    assert ws(FAKE, FAKE, 0, FAKE, FAKE, 0, 256, 256, 128, 1, FAKE, 0, ODD, 1 << 20, None) == -3   # workspace alignment
    assert ws(FAKE, FAKE, 0, FAKE, FAKE, 0, 256, 100, 128, 1, FAKE, 0, FAKE, 1 << 20, None) == -2

    rf = so.fp8_ring_fold
    assert rf(None, FAKE, 16, 0, 448.0, 1.0, None) == -1           # no amax
    assert rf(FAKE, None, 16, 0, 448.0, 1.0, None) == -1           # no ring
    assert rf(FAKE, FAKE, 16, 16, 448.0, 1.0, None) == -1          # hist_idx out of range
    assert rf(FAKE, FAKE, 0, 0, 448.0, 1.0, None) == -1            # empty history
    assert rf(ctypes.c_void_p(0x10002), FAKE, 16, 0, 448.0, 1.0, None) == -3

    assert so.mxq_dequantize(FAKE, FAKE, 64, 48, 0, 1, FAKE, None) == -2
    assert so.mxq_sf_to_mma(FAKE, 100, 4, FAKE, None) == -2


def test_package_has_no_fallback(monkeypatch, tmp_path):
    """Without the built library every entry point raises (no CPU path)."""
    import block_scaled_precision_02_gb300 as mxq
    monkeypatch.setattr(mxq, "_lib", None)
    monkeypatch.setattr(mxq, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        mxq.load()


def test_product_path_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "block_scaled_precision_02_gb300")
    for path in glob.glob(os.path.join(pkg, "**", "*.*"), recursive=True):
        if path.endswith((".py", ".cu", ".cuh", ".h")):
            text = open(path).read()
            assert "import oracle" not in text and "from oracle" not in text, path


def test_group_argument_checks_need_no_gpu(so):
    """mxq_quantize_group: the group's own checks, then each job's, in job
    order, all before any launch (on a machine without a GPU the last step
    is the device check)."""
    from block_scaled_precision_02_gb300 import QuantJob
    g = so.mxq_quantize_group
    ok = QuantJob(0x10000, 64, 64, 64, 0, 0x10000, 0x10000, 0, 0)
    jobs = (QuantJob * 5)(ok, ok, ok, ok, ok)
    assert g(None, 1, 0, 1, 0, None) == -1                       # no jobs array
    assert g(jobs, 0, 0, 1, 0, None) == -1                       # empty group
    assert g(jobs, 5, 0, 1, 0, None) == -1                       # more than MXQ_QUANT_GROUP_MAX
    assert g(jobs, 2, 9, 1, 0, None) == -1                       # format
    assert g(jobs, 2, 0, 4, 0, None) == -1                       # orientation
    assert g(jobs, 2, 0, 1, 5, None) == -1                       # scale layout
    bad = (QuantJob * 2)(ok, QuantJob(0x10000, 48, 64, 64, 0, 0x10000, 0x10000, 0, 0))
    assert g(bad, 2, 0, 1, 0, None) == -2                        # the second job's shape
    bad = (QuantJob * 2)(ok, QuantJob(0x10000, 64, 64, 64, 2, 0x10000, 0x10000, 0, 0))
    assert g(bad, 2, 0, 1, 0, None) == -1                        # the second job's scale mode
    bad = (QuantJob * 2)(QuantJob(0x10008, 64, 64, 64, 0, 0x10000, 0x10000, 0, 0), ok)
    assert g(bad, 2, 0, 1, 0, None) == -3                        # the first job's input alignment
    bad = (QuantJob * 1)(QuantJob(0x10000, 64, 64, 64, 0, 0x10000, 0x10000, 0, 0))
    assert g(bad, 1, 0, 3, 0, None) == -1                        # DUAL without column outputs
    assert g(jobs, 4, 0, 1, 0, None) == -4                       # valid: no device here


def test_header_is_plain_c(tmp_path):
    """include/mxq.h is a C header: a C99 translation unit that uses its
    types and constants compiles (no C++ or torch types leak into it)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_header.c"
    src.write_text('#include "mxq.h"\n'
                   "int main(void) {\n"
                   "  mxq_quant_job j = {0};\n"
                   "  (void)j;\n"
                   "  return MXQ_QUANT_GROUP_MAX + MXQ_E2M1 + MXQ_SF_MMA;\n"
                   "}\n")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-I", os.path.join(ROOT, "include"),
                        str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
