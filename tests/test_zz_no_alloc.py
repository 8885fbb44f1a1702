"""mxq_gemm_noalloc, the GEMM entry point for callers that cannot allocate
device memory when they call (for example inside another framework's
executor that owns the device's memory): it runs the stream-K product of
mxq_gemm_ws with the library's own static scratch array instead of a caller
workspace.  Checked through the C ABI against mxq_gemm_ws with a caller
workspace, on two calls in a row (the second finds the first call's leftovers
in the shared array), on a shape whose sparse last wave makes the stream-K
schedule -- and so the scratch -- take part.  Collected last on purpose."""

import ctypes

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import gemm as og
from oracle import mx as omx

pytestmark = pytest.mark.gpu


def test_no_alloc_gemm_matches_the_workspace_gemm_twice(lib):
    dev = torch.device("cuda", torch.cuda.current_device())
    pairs = torch.cuda.get_device_properties(dev).multi_processor_count // 2
    nt_n = 8
    nt_m = -(-(pairs + 8) // nt_n)                 # one full wave of pairs and a sparse last one
    M, N, K = 256 * nt_m, 256 * nt_n, 2048
    rng = np.random.default_rng(11)
    a = omx.quantize(rng.standard_normal((M, K)), F.E4M3, omx.ROW)
    b = omx.quantize(rng.standard_normal((N, K)) * 0.02, F.E4M3, omx.ROW)
    t = lambda v: torch.from_numpy(np.ascontiguousarray(v)).to(dev)
    A, As, B, Bs = t(a["q_row"]), t(omx.sf_to_mma(a["s_row"])), t(b["q_row"]), t(omx.sf_to_mma(b["s_row"]))
    L = lib.load()
    p = lambda x: ctypes.c_void_p(x.data_ptr())
    st = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)

    n = ctypes.c_size_t(0)
    assert L.mxq_gemm_workspace_size(ctypes.byref(n)) == 0
    ws = torch.zeros(n.value, dtype=torch.uint8, device=dev)
    want = torch.empty(M, N, dtype=torch.float32, device=dev)
    assert L.mxq_gemm_ws(p(A), p(As), 0, p(B), p(Bs), 0, M, N, K, 1, p(want), 1, p(ws), n.value, st) == 0
    ref = og.reference(a["q_row"], a["s_row"], b["q_row"], b["s_row"], F.E4M3)
    w = want.cpu().numpy().astype(np.float64)
    assert og.gate_error(w, ref, out_is_bf16=False) <= 1e-5

    for call in range(2):
        got = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
        assert L.mxq_gemm_noalloc(p(A), p(As), 0, p(B), p(Bs), 0, M, N, K, 1, p(got), 1, st) == 0
        g = got.cpu().numpy().astype(np.float64)
        scale = np.maximum(np.abs(w), np.sqrt(np.mean(w ** 2)))
        assert np.max(np.abs(g - w) / scale) <= 1e-5, f"call {call}"
        assert og.gate_error(g, ref, out_is_bf16=False) <= 1e-5, f"call {call}"
    assert lib.last_device_status(dev) == 0
