"""The Python binding refuses, before any library call, arguments that would
send a kernel a host pointer or fewer bytes than it reads: operands that
disagree on K, scale tensors of the wrong size, wide element types, and
tensors that are not on the GPU.  CPU only: every call here raises."""

import pytest
import torch

import block_scaled_precision_02_gb300 as mxq


def u8(*shape):
    return torch.zeros(*shape, dtype=torch.uint8)


def test_gemm_operands_must_agree_on_k():
    with pytest.raises(ValueError, match="K differs"):
        mxq.mx_gemm(u8(256, 512), u8(256 * 16), u8(256, 256), u8(256 * 8), "e4m3")
    # packed E2M1 beside E4M3: 256 bytes of E2M1 codes are 512 elements
    with pytest.raises(ValueError, match="K differs"):
        mxq.mx_gemm(u8(256, 512), u8(256 * 16), u8(256, 512), u8(256 * 32), "e4m3", b_fmt="e2m1")
    with pytest.raises(ValueError, match="K differs"):
        mxq.mx_gemm(u8(256, 512), u8(256 * 16), u8(256, 512), u8(256 * 16), "e4m3", K=1024)
    with pytest.raises(ValueError, match="K differs"):
        mxq.mx_gemm_mx_out(u8(256, 512), u8(256 * 16), u8(256, 256), u8(256 * 8), "e4m3")


def test_gemm_scales_must_cover_every_block():
    with pytest.raises(ValueError, match="a_s holds"):
        mxq.mx_gemm(u8(256, 512), u8(256 * 15), u8(256, 512), u8(256 * 16), "e4m3")
    with pytest.raises(ValueError, match="b_s holds"):
        mxq.mx_gemm(u8(256, 512), u8(256 * 16), u8(128, 512), u8(256 * 16), "e4m3")
    with pytest.raises(ValueError, match="b_s holds"):
        mxq.mx_gemm(u8(256, 512), u8(256 * 16), u8(256, 256), u8(256 * 8), "e4m3", b_fmt="e2m1")


def test_gemm_operands_must_be_byte_codes_on_the_gpu():
    with pytest.raises(ValueError, match="1-byte elements"):
        mxq.mx_gemm(torch.zeros(256, 512, dtype=torch.bfloat16), u8(256 * 16), u8(256, 512), u8(256 * 16))
    with pytest.raises(ValueError, match="1-byte elements"):
        mxq.mx_gemm(u8(256, 512), u8(256 * 16), u8(256, 512).t().contiguous().t(), u8(256 * 16))
    with pytest.raises(ValueError, match="CUDA tensor"):
        mxq.mx_gemm(u8(256, 512), u8(256 * 16), u8(256, 512), u8(256 * 16), "e4m3")
    with pytest.raises(ValueError, match="out_dtype"):
        mxq.mx_gemm(u8(256, 512), u8(256 * 16), u8(256, 512), u8(256 * 16), out_dtype=torch.float16)


def test_dequantize_checks_scales_and_device():
    with pytest.raises(ValueError, match="s holds"):
        mxq.mx_dequantize(u8(64, 64), u8(64, 1), "e4m3")
    with pytest.raises(ValueError, match="CUDA tensor"):
        mxq.mx_dequantize(u8(64, 64), u8(64, 2), "e4m3")
    with pytest.raises(ValueError, match="out_dtype"):
        mxq.mx_dequantize(u8(64, 64), u8(64, 2), "e4m3", torch.int32)


def test_quantize_group_checks_before_any_call():
    x = torch.zeros(64, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="between 1 and"):
        mxq.mx_quantize_group([], "e4m3")
    with pytest.raises(ValueError, match="between 1 and"):
        mxq.mx_quantize_group([x] * 5, "e4m3")
    with pytest.raises(ValueError, match="one scale mode"):
        mxq.mx_quantize_group([x, x], "e4m3", "row", ["floor"])
    with pytest.raises(ValueError, match="CUDA tensor"):
        mxq.mx_quantize_group([x], "e4m3")
    with pytest.raises(ValueError, match="unknown format 'e3m4'"):
        mxq.mx_quantize_group([x], "e3m4")
    with pytest.raises(ValueError, match="unknown scale mode"):
        mxq.mx_quantize_group([x], "e4m3", "row", "round")


def test_mm_fp8_needs_byte_codes():
    a = torch.zeros(128, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="1-byte FP8 codes"):
        mxq.mm_fp8(a, a.t(), torch.ones(1))


def test_sf_to_mma_needs_a_gpu_tensor():
    with pytest.raises(ValueError, match="CUDA tensor"):
        mxq.sf_to_mma(u8(128, 4))
    with pytest.raises(ValueError, match="2-D"):
        mxq.sf_to_mma(u8(512))


def test_every_library_call_runs_with_the_tensors_device_current(monkeypatch):
    """The library launches on the current device and takes the stream of
    that device: each entry point of the binding calls the library through
    _call, which makes the tensors' device current around the call."""
    import ast
    import inspect
    src = inspect.getsource(mxq)
    tree = ast.parse(src)
    direct = []
    for fn in ast.walk(tree):
        # these guard the device themselves (with torch.cuda.device)
        if isinstance(fn, ast.FunctionDef) and fn.name not in ("_call", "load", "lib", "last_device_status",
                                                               "gemm_workspace"):
            for node in ast.walk(fn):
                if (isinstance(node, ast.Call) and isinstance(node.func, ast.Attribute)
                        and isinstance(node.func.value, ast.Call) and getattr(node.func.value.func, "id", "") == "load"):
                    direct.append(fn.name)
    assert direct == [], f"library called without the device guard in {direct}"

    events = []

    class FakeDevice:
        def __init__(self, d):
            self.d = d

        def __enter__(self):
            events.append(("enter", str(self.d)))

        def __exit__(self, *a):
            events.append(("exit", str(self.d)))

    class FakeLib:
        def mxq_sf_to_mma(self, *args):
            events.append(("call", args[-1]))
            return 0

    monkeypatch.setattr(mxq.torch.cuda, "device", FakeDevice)
    monkeypatch.setattr(mxq, "_stream", lambda d: f"stream of {d}")
    monkeypatch.setattr(mxq, "load", lambda: FakeLib())
    mxq._call("mxq_sf_to_mma", torch.device("cuda", 1), 1, 2)
    assert events == [("enter", "cuda:1"), ("call", "stream of cuda:1"), ("exit", "cuda:1")]
