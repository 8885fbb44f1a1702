"""Python binding of the ``libmxq`` C ABI (include/mxq.h).

Argument marshalling only: every step of the quantizers and the GEMM runs in
the library's sm_103a kernels.  PyTorch supplies device memory and the
current stream.  There is no fallback: if ``libmxq.so`` is missing or fails
to load, every call raises.

Entry points (same names as the C ABI):
  mx_quantize, mx_dequantize, fp8_quantize_pertensor, ring_fold, mx_gemm,
  mx_gemm_mx_out, mm_fp8, sf_to_mma, last_device_status; plus ``quantize`` / ``quantize_dual`` with the
  argument order of AstrAI's fp8 adapter (astrai/extension/ops/fp8.py).
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmxq.so")

E4M3, E5M2, E2M1 = 0, 1, 2
ROW, COL, DUAL = 1, 2, 3
FLOOR_OCP, CEIL = 0, 1
RNE, SR, SR4 = 0, 1, 2
SF_CANONICAL, SF_MMA = 0, 1

class _Choices(dict):
    """Name (or code) -> library code; an unknown name is a ValueError."""

    def __init__(self, what: str, items: dict):
        super().__init__(items)
        self.what = what

    def __missing__(self, key):
        names = sorted(k for k in self if isinstance(k, str))
        raise ValueError(f"unknown {self.what} {key!r} (one of {', '.join(names)})")


_FMT = _Choices("format", {"e4m3": E4M3, "e5m2": E5M2, "e2m1": E2M1, E4M3: E4M3, E5M2: E5M2, E2M1: E2M1})
_ORIENT = _Choices("orientation", {"row": ROW, "col": COL, "dual": DUAL, ROW: ROW, COL: COL, DUAL: DUAL})
_SCALE = _Choices("scale mode", {"floor": FLOOR_OCP, "floor_ocp": FLOOR_OCP, "ceil": CEIL, FLOOR_OCP: FLOOR_OCP,
                                 CEIL: CEIL})
_ROUND = _Choices("rounding", {"rne": RNE, "sr": SR, "stochastic": SR, "sr4": SR4, RNE: RNE, SR: SR, SR4: SR4})
_SF = _Choices("scale layout", {"canonical": SF_CANONICAL, "mma": SF_MMA, SF_CANONICAL: SF_CANONICAL,
                                SF_MMA: SF_MMA})

_lib = None


QUANT_GROUP_MAX = 4   # MXQ_QUANT_GROUP_MAX


class QuantJob(ctypes.Structure):
    """One job of mxq_quantize_group (the C struct mxq_quant_job)."""
    _fields_ = [("x", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("ld", ctypes.c_int64), ("scale_mode", ctypes.c_int), ("q_row", ctypes.c_void_p),
                ("s_row", ctypes.c_void_p), ("q_col", ctypes.c_void_p), ("s_col", ctypes.c_void_p)]


class MXQError(RuntimeError):
    def __init__(self, status: int, what: str):
        msg = _lib.mxq_strerror(status).decode() if _lib is not None else str(status)
        super().__init__(f"{what}: {msg} (status {status})")
        self.status = status


def load() -> ctypes.CDLL:
    """Load libmxq.so (built in-tree by ``build()``).  Raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                           "(there is no CPU or PyTorch fallback)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, u64, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64, ctypes.c_float
    L.mxq_quantize.argtypes = [vp, i64, i64, i64, i32, i32, i32, i32, i32, u64, u64, i32, vp, vp, vp, vp, vp]
    L.mxq_quantize_group.argtypes = [ctypes.POINTER(QuantJob), i32, i32, i32, i32, vp]
    L.mxq_dequantize.argtypes = [vp, vp, i64, i64, i32, i32, vp, vp]
    L.fp8_quantize_pertensor.argtypes = [vp, i64, i64, vp, i32, i32, vp, i32, i32, f32, f32, vp, vp, vp, vp]
    L.fp8_ring_fold.argtypes = [vp, vp, i32, i32, f32, f32, vp]
    L.mxq_gemm.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, i32, vp, i32, vp]
    L.mxq_gemm_mixed.argtypes = [vp, vp, i32, vp, vp, i32, i64, i64, i64, i32, vp, i32, vp]
    L.mxq_gemm_workspace_size.argtypes = [vp]
    L.mxq_gemm_ws.argtypes = [vp, vp, i32, vp, vp, i32, i64, i64, i64, i32, vp, i32, vp, ctypes.c_size_t, vp]
    L.mxq_gemm_noalloc.argtypes = [vp, vp, i32, vp, vp, i32, i64, i64, i64, i32, vp, i32, vp]
    L.mxq_gemm_mx_out.argtypes = [vp, vp, i32, vp, vp, i32, i64, i64, i64, i32, i32, i32, i32, vp, vp, vp, vp, vp]
    L.mxq_mm_fp8.argtypes = [vp, vp, i64, i64, i64, i64, i32, i32, i32, i32, i32, vp, vp, vp, vp]
    L.mxq_sf_to_mma.argtypes = [vp, i64, i64, vp, vp]
    L.mxq_last_device_status.argtypes = [vp]
    L.mxq_strerror.argtypes = [i32]
    L.mxq_strerror.restype = ctypes.c_char_p
    L.mxq_version.argtypes = []
    L.mxq_test_stall_next_launch.argtypes = [i32]
    for name in ("mxq_quantize", "mxq_quantize_group", "mxq_dequantize", "fp8_quantize_pertensor", "fp8_ring_fold", "mxq_gemm",
                 "mxq_gemm_mixed", "mxq_gemm_workspace_size", "mxq_gemm_ws", "mxq_gemm_noalloc",
                 "mxq_gemm_mx_out", "mxq_mm_fp8", "mxq_sf_to_mma",
                 "mxq_last_device_status", "mxq_version", "mxq_test_stall_next_launch"):
        getattr(L, name).restype = i32
    _lib = L
    return L


def lib() -> ctypes.CDLL:
    return load()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(rc: int, what: str):
    if rc != 0:
        raise MXQError(rc, what)


def _call(name: str, device: torch.device, *args) -> None:
    """Run library entry point ``name`` with ``device`` current and torch's
    current stream of that device appended as the last argument; raise on a
    non-zero status.  The library launches on the current device and keys
    its per-device state (status word, SM count, occupancy) on it, and the
    stream handle must belong to that device, so every call makes the
    tensors' device current first (restoring the previous one after)."""
    with torch.cuda.device(device):
        rc = getattr(load(), name)(*args, _stream(device))
    _check(rc, name)


def _cuda_2d(x: torch.Tensor, name: str):
    if not x.is_cuda or x.dim() != 2:
        raise ValueError(f"{name} must be a 2-D CUDA tensor")


# Argument checks that keep a wrong call from reaching a kernel: every device
# pointer the library dereferences must be a CUDA tensor on the call's device
# holding at least the bytes the call reads.  Structural checks come first.
def _on_device(ts, device: torch.device):
    for t, name in ts:
        if t is None:
            continue
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.device != device:
            raise ValueError(f"{name} is on {t.device}, the call's other tensors on {device}")


def _byte_tensor(t: torch.Tensor, name: str, numel: Optional[int] = None):
    """Codes or scales: contiguous, one byte per element (uint8 or a float8
    dtype), and exactly ``numel`` elements when given."""
    if not isinstance(t, torch.Tensor) or t.element_size() != 1 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous tensor of 1-byte elements")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} holds {t.numel()} bytes, expected {numel}")


def _mx_operands(a_q, a_s, f, b_q, b_s, fb, K):
    """(M, N, K) of a block-scaled product, after checking that A [M][K] and
    B [N][K] agree on K (E2M1 codes packed two per byte) and that each scale
    tensor holds one byte per row per 32 elements of K."""
    for t, name in ((a_q, "a_q"), (b_q, "b_q")):
        if not isinstance(t, torch.Tensor) or t.dim() != 2:
            raise ValueError(f"{name} must be a 2-D tensor of codes")
    M, N = a_q.shape[0], b_q.shape[0]
    ka = a_q.shape[1] * (2 if f == E2M1 else 1)
    kb = b_q.shape[1] * (2 if fb == E2M1 else 1)
    if K is None:
        K = ka
    if ka != K or kb != K:
        raise ValueError(f"K differs: a_q holds {ka}, b_q {kb}, K = {K}")
    _byte_tensor(a_q, "a_q")
    _byte_tensor(b_q, "b_q")
    if K % 32 == 0:
        _byte_tensor(a_s, "a_s", M * (K // 32))
        _byte_tensor(b_s, "b_s", N * (K // 32))
    else:
        _byte_tensor(a_s, "a_s")
        _byte_tensor(b_s, "b_s")
    _on_device(((a_q, "a_q"), (a_s, "a_s"), (b_q, "b_q"), (b_s, "b_s")), a_q.device)
    return M, N, K


# --------------------------------------------------------------------------- MX quantize
def mx_quantize(x: torch.Tensor, fmt="e4m3", orientation="row", scale_mode="floor", rounding="rne",
                hadamard32: bool = False, sr_key: int = 0, hadamard_seed: int = 7, sf_layout="canonical"):
    """MX-quantize bf16 ``x`` [rows][cols] (row stride may exceed cols).

    Returns (q_row, s_row, q_col, s_col); entries for an orientation not
    requested are None.  q_col / s_col are the transposed column copy."""
    _cuda_2d(x, "x")
    if x.dtype != torch.bfloat16 or x.stride(1) != 1:
        raise ValueError("x must be bf16 with a contiguous last dimension")
    f, o = _FMT[fmt], _ORIENT[orientation]
    rows, cols = x.shape
    dev = x.device
    qb = 2 if f == E2M1 else 1
    q_row = s_row = q_col = s_col = None
    if o & ROW:
        q_row = torch.empty(rows, cols // qb, dtype=torch.uint8, device=dev)
        s_row = torch.empty(rows, cols // 32, dtype=torch.uint8, device=dev)
    if o & COL:
        q_col = torch.empty(cols, rows // qb, dtype=torch.uint8, device=dev)
        s_col = torch.empty(cols, rows // 32, dtype=torch.uint8, device=dev)
    _call("mxq_quantize", dev, _ptr(x), rows, cols, x.stride(0), f, o, _SCALE[scale_mode], _ROUND[rounding],
          int(bool(hadamard32)), sr_key & (2**64 - 1), hadamard_seed & (2**64 - 1), _SF[sf_layout], _ptr(q_row),
          _ptr(s_row), _ptr(q_col), _ptr(s_col))
    return q_row, s_row, q_col, s_col


def mx_quantize_group(xs, fmt="e4m3", orientation="row", scale_modes="floor", sf_layout="canonical"):
    """MX-quantize up to QUANT_GROUP_MAX bf16 tensors of one format and
    orientation (RNE, no Hadamard) in one launch: the persistent grid runs
    through all of them, so the fill and drain of a launch are paid once.
    ``scale_modes`` is one mode for all tensors or a sequence, one per tensor.
    Returns one (q_row, s_row, q_col, s_col) tuple per tensor, each exactly
    what mx_quantize returns for it."""
    xs = list(xs)
    if not 1 <= len(xs) <= QUANT_GROUP_MAX:
        raise ValueError(f"between 1 and {QUANT_GROUP_MAX} tensors per group")
    modes = [scale_modes] * len(xs) if isinstance(scale_modes, str) else list(scale_modes)
    if len(modes) != len(xs):
        raise ValueError("one scale mode, or one per tensor")
    f, o, sf = _FMT[fmt], _ORIENT[orientation], _SF[sf_layout]
    codes = [_SCALE[m] for m in modes]
    qb = 2 if f == E2M1 else 1
    dev = None
    outs, jobs = [], (QuantJob * len(xs))()
    for k, (x, mode) in enumerate(zip(xs, codes)):
        _cuda_2d(x, f"xs[{k}]")
        if x.dtype != torch.bfloat16 or x.stride(1) != 1:
            raise ValueError("every tensor must be bf16 with a contiguous last dimension")
        dev = x.device if dev is None else dev
        _on_device(((x, f"xs[{k}]"),), dev)
        rows, cols = x.shape
        q_row = s_row = q_col = s_col = None
        if o & ROW:
            q_row = torch.empty(rows, cols // qb, dtype=torch.uint8, device=dev)
            s_row = torch.empty(rows, cols // 32, dtype=torch.uint8, device=dev)
        if o & COL:
            q_col = torch.empty(cols, rows // qb, dtype=torch.uint8, device=dev)
            s_col = torch.empty(cols, rows // 32, dtype=torch.uint8, device=dev)
        jobs[k] = QuantJob(x.data_ptr(), rows, cols, x.stride(0), mode,
                           *[0 if t is None else t.data_ptr() for t in (q_row, s_row, q_col, s_col)])
        outs.append((q_row, s_row, q_col, s_col))
    _call("mxq_quantize_group", dev, jobs, len(xs), f, o, sf)
    return outs


def mx_dequantize(q: torch.Tensor, s: torch.Tensor, fmt="e4m3", out_dtype=torch.float32) -> torch.Tensor:
    """Dequantize codes ``q`` with canonical scales ``s`` -> float32 or bf16."""
    f = _FMT[fmt]
    if not isinstance(q, torch.Tensor) or q.dim() != 2:
        raise ValueError("q must be a 2-D tensor of codes")
    if out_dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("out_dtype must be torch.float32 or torch.bfloat16")
    rows = q.shape[0]
    cols = q.shape[1] * (2 if f == E2M1 else 1)
    _byte_tensor(q, "q")
    _byte_tensor(s, "s", rows * (cols // 32) if cols % 32 == 0 else None)
    _on_device(((q, "q"), (s, "s")), q.device)
    out = torch.empty(rows, cols, dtype=out_dtype, device=q.device)
    _call("mxq_dequantize", q.device, _ptr(q), _ptr(s), rows, cols, f, int(out_dtype == torch.float32), _ptr(out))
    return out


# --------------------------------------------------------------------------- per-tensor FP8
def fp8_quantize_pertensor(x: torch.Tensor, scale: torch.Tensor, fmt="e4m3", orientation="row",
                           ring_state: Optional[torch.Tensor] = None, hist_idx: int = 0,
                           fp8_max: float = 448.0, pow2_margin: float = 1.0):
    """Per-tensor FP8 quantize with fused amax (and the delayed-scaling fold
    when ``ring_state`` is given).  Returns (x8, x8T, amax); ``amax`` is a
    fresh 1-element float32 tensor, or, with a ring, a view of the ring's
    amax slot (which the fold leaves at zero)."""
    _cuda_2d(x, "x")
    if x.dtype != torch.bfloat16 or not x.is_contiguous():
        raise ValueError("x must be contiguous bf16")
    f, o = _FMT[fmt], _ORIENT[orientation]
    if f not in (E4M3, E5M2):
        raise ValueError(f"unsupported fp8 format {fmt!r} (expected 'e4m3' or 'e5m2')")
    if not isinstance(scale, torch.Tensor) or scale.dtype != torch.float32 or scale.numel() < 1:
        raise ValueError("scale must be a float32 device tensor (its first element is the multiplier)")
    if ring_state is not None and (ring_state.dtype != torch.float32 or not ring_state.is_contiguous()
                                   or ring_state.numel() < 5):
        raise ValueError("ring_state must be a contiguous float32 tensor of hist_len + 4 >= 5 elements")
    _on_device(((scale, "scale"), (ring_state, "ring_state")), x.device)
    rows, cols = x.shape
    dev = x.device
    x8 = torch.empty(rows, cols, dtype=torch.uint8, device=dev) if o & ROW else None
    x8T = torch.empty(cols, rows, dtype=torch.uint8, device=dev) if o & COL else None
    n = 0
    if ring_state is not None:
        n = ring_state.numel() - 4
        amax = ring_state[n + 2:n + 3]
        amax_out = None
    else:
        amax = torch.empty(1, dtype=torch.float32, device=dev)
        amax_out = amax
    _call("fp8_quantize_pertensor", dev, _ptr(x), rows, cols, _ptr(scale), f, o, _ptr(ring_state), n, hist_idx,
          float(fp8_max), float(pow2_margin), _ptr(x8), _ptr(x8T), _ptr(amax_out))
    return x8, x8T, amax


def quantize(x, scale, fmt="e4m3", transposed=False, ring_state=None, hist_idx=0, fp8_max=448.0,
             pow2_margin=1.0):
    """(x8 | x8T, amax), argument order of AstrAI's ``quantize``."""
    x8, x8T, amax = fp8_quantize_pertensor(x, scale, fmt, "col" if transposed else "row", ring_state, hist_idx,
                                           fp8_max, pow2_margin)
    return (x8T if transposed else x8), amax


def quantize_dual(x, scale, fmt="e4m3", ring_state=None, hist_idx=0, fp8_max=448.0, pow2_margin=1.0):
    """(x8, x8T, amax) from one read, argument order of AstrAI's ``quantize_dual``."""
    return fp8_quantize_pertensor(x, scale, fmt, "dual", ring_state, hist_idx, fp8_max, pow2_margin)


def ring_fold(amax: torch.Tensor, ring_state: torch.Tensor, hist_idx: int = 0, fp8_max: float = 448.0,
              pow2_margin: float = 1.0) -> None:
    """Fold a given tensor amax (a 1-element float32 device tensor) into the
    ring and publish the next scale -- the fold fp8_quantize_pertensor runs
    in its last block, for a tensor quantized in row shards whose amaxes were
    MAX-reduced first (see ``shard.pertensor_step``)."""
    if not isinstance(amax, torch.Tensor) or amax.dtype != torch.float32 or amax.numel() < 1:
        raise ValueError("amax must be a float32 device tensor")
    if (not isinstance(ring_state, torch.Tensor) or ring_state.dtype != torch.float32
            or not ring_state.is_contiguous() or ring_state.numel() < 5):
        raise ValueError("ring_state must be a contiguous float32 tensor of hist_len + 4 >= 5 elements")
    _on_device(((amax, "amax"), (ring_state, "ring_state")), ring_state.device)
    n = ring_state.numel() - 4
    _call("fp8_ring_fold", ring_state.device, _ptr(amax), _ptr(ring_state), n, hist_idx, float(fp8_max),
          float(pow2_margin))


def ring_state_new(hist_len: int = 16, device="cuda") -> torch.Tensor:
    """Fresh ring [hist | scale | legacy | amax | done]: hist 0, scale 1, legacy 1, amax 0, done 0."""
    r = torch.zeros(hist_len + 4, dtype=torch.float32, device=device)
    r[hist_len] = 1.0
    r[hist_len + 1] = 1.0
    return r


# --------------------------------------------------------------------------- GEMM
_WS = {}


def gemm_workspace(device: torch.device) -> torch.Tensor:
    """The stream-K workspace the binding passes to mxq_gemm_ws for torch's
    current stream on ``device``: allocated (and zero-filled) by torch on
    first use, then kept; one per stream, because calls that share a
    workspace must not overlap on the GPU."""
    device = torch.device(device)
    key = (device.index, torch.cuda.current_stream(device).cuda_stream)
    w = _WS.get(key)
    if w is None:
        n = ctypes.c_size_t(0)
        with torch.cuda.device(device):
            _check(load().mxq_gemm_workspace_size(ctypes.byref(n)), "mxq_gemm_workspace_size")
        w = torch.zeros(n.value, dtype=torch.uint8, device=device)
        _WS[key] = w
    return w


def mx_gemm(a_q: torch.Tensor, a_s: torch.Tensor, b_q: torch.Tensor, b_s: torch.Tensor, fmt="e4m3",
            out_dtype=torch.bfloat16, sf_layout="mma", K: Optional[int] = None, b_fmt=None,
            stream_k: bool = True) -> torch.Tensor:
    """C = A * B^T from MX operands (A [M][K], B [N][K] codes, scales in the
    MMA layout).  ``fmt`` is A's element format and B's unless ``b_fmt`` is
    given (any two of E4M3, E5M2 and E2M1: an E2M1 operand beside an 8-bit
    one runs at the 8-bit rate).  Returns bf16 (or float32) [M][N].  Runs
    the stream-K schedule of mxq_gemm_ws with this stream's workspace, unless
    ``stream_k`` is False (mxq_gemm / mxq_gemm_mixed)."""
    f = _FMT[fmt]
    fb = f if b_fmt is None else _FMT[b_fmt]
    if out_dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("out_dtype must be torch.bfloat16 or torch.float32")
    M, N, K = _mx_operands(a_q, a_s, f, b_q, b_s, fb, K)
    c = torch.empty(M, N, dtype=out_dtype, device=a_q.device)
    if stream_k:
        ws = gemm_workspace(a_q.device)
        _call("mxq_gemm_ws", a_q.device, _ptr(a_q), _ptr(a_s), f, _ptr(b_q), _ptr(b_s), fb, M, N, K,
              _SF[sf_layout], _ptr(c), int(out_dtype == torch.float32), _ptr(ws), ws.numel())
    elif fb == f:
        _call("mxq_gemm", a_q.device, _ptr(a_q), _ptr(a_s), _ptr(b_q), _ptr(b_s), M, N, K, f, _SF[sf_layout],
              _ptr(c), int(out_dtype == torch.float32))
    else:
        _call("mxq_gemm_mixed", a_q.device, _ptr(a_q), _ptr(a_s), f, _ptr(b_q), _ptr(b_s), fb, M, N, K,
              _SF[sf_layout], _ptr(c), int(out_dtype == torch.float32))
    return c


def mx_gemm_mx_out(a_q: torch.Tensor, a_s: torch.Tensor, b_q: torch.Tensor, b_s: torch.Tensor, fmt="e4m3",
                   b_fmt=None, out_fmt="e4m3", out_scale_mode="floor", out_sf_layout="canonical",
                   orientation="row", K: Optional[int] = None):
    """A * B^T as mx_gemm, written as MX codes and scales straight from the
    accumulator: row blocks (1x32 along N) and/or column blocks (32x1 along
    M, stored transposed), per ``orientation`` ("row", "col", "dual").
    Returns (codes [M][N], scales [M][N/32], codesT [N][M], scalesT [N][M/32])
    with None for an orientation not requested (``out_fmt`` "e2m1": codes
    packed two per byte, [M][N/2] and [N][M/2]); MMA-layout scales hold the
    same number of bytes."""
    f = _FMT[fmt]
    fb = f if b_fmt is None else _FMT[b_fmt]
    o = _ORIENT[orientation]
    M, N, K = _mx_operands(a_q, a_s, f, b_q, b_s, fb, K)
    dev = a_q.device
    ob = 2 if _FMT[out_fmt] == E2M1 else 1          # E2M1 codes: two per byte
    cq = cs = cqT = csT = None
    if o & ROW:
        cq = torch.empty(M, N // ob, dtype=torch.uint8, device=dev)
        cs = torch.empty(M, N // 32, dtype=torch.uint8, device=dev)
    if o & COL:
        cqT = torch.empty(N, M // ob, dtype=torch.uint8, device=dev)
        csT = torch.empty(N, M // 32, dtype=torch.uint8, device=dev)
    _call("mxq_gemm_mx_out", dev, _ptr(a_q), _ptr(a_s), f, _ptr(b_q), _ptr(b_s), fb, M, N, K, SF_MMA,
          _FMT[out_fmt], _SCALE[out_scale_mode], _SF[out_sf_layout], _ptr(cq), _ptr(cs), _ptr(cqT), _ptr(csT))
    return cq, cs, cqT, csT


def mm_fp8(a: torch.Tensor, b: torch.Tensor, scale: torch.Tensor, trans_a: bool = False, trans_b: bool = False,
           bias: Optional[torch.Tensor] = None, fmt: Optional[str] = None) -> torch.Tensor:
    """Per-tensor FP8 GEMM ``op(a) @ op(b) * scale (+ bias)`` (AstrAI fp8.py
    mm_fp8), bf16 result.  ``a``/``b`` hold FP8 codes (uint8 or a torch
    float8 dtype, which also gives the format), 2-D or 3-D (a batch axis
    broadcasts); op transposes the last two axes when the flag is set.
    Transposed views are read in place, with no copy: op(a) may have
    K-contiguous rows (a row-major [M][K]) or M-contiguous columns (the
    transpose of a row-major [K][M]), op(b) K-contiguous columns (the
    transpose of a row-major [N][K] weight) or N-contiguous rows (a
    row-major [K][N]); any other layout raises ValueError.  ``scale`` is a
    1-element device float32 tensor, ``bias`` a bf16 [N] vector."""
    if fmt is None:
        names = {getattr(torch, "float8_e4m3fn", None): "e4m3", getattr(torch, "float8_e5m2", None): "e5m2"}
        fmt = names.get(a.dtype, "e4m3")
    f = _FMT[fmt]
    A = a.transpose(-1, -2) if trans_a else a
    B = b.transpose(-1, -2) if trans_b else b
    if A.dim() not in (2, 3) or B.dim() not in (2, 3):
        raise ValueError("mm_fp8 takes 2-D or 3-D operands")
    M, K = A.shape[-2], A.shape[-1]
    if B.shape[-2] != K:
        raise ValueError(f"inner dimensions differ: {K} vs {B.shape[-2]}")
    N = B.shape[-1]
    # storage of each operand: op(a) K-contiguous -> a row-major [M][K]
    # (library trans_a 0), M-contiguous -> [K][M] (1); op(b) K-contiguous ->
    # b row-major [N][K] (library trans_b 1), N-contiguous -> [K][N] (0)
    if A.stride(-1) == 1 and A.stride(-2) == K:
        ta = 0
    elif A.stride(-2) == 1 and A.stride(-1) == M:
        ta = 1
    else:
        raise ValueError("op(a) must be a row-major [M][K] matrix or the transpose of a row-major [K][M] one")
    if B.stride(-2) == 1 and B.stride(-1) == K:
        tb = 1
    elif B.stride(-1) == 1 and B.stride(-2) == N:
        tb = 0
    else:
        raise ValueError("op(b) must be a row-major [K][N] matrix or the transpose of a row-major [N][K] one")
    ba = A.shape[0] if A.dim() == 3 else 1
    bb = B.shape[0] if B.dim() == 3 else 1
    if ba > 1 and bb > 1 and ba != bb:
        raise ValueError(f"batch sizes differ: {ba} vs {bb}")
    batch = max(ba, bb)
    if A.dim() == 3 and ba > 1 and A.stride(0) != M * K:
        raise ValueError("a's batch entries must be contiguous")
    if B.dim() == 3 and bb > 1 and B.stride(0) != N * K:
        raise ValueError("b's batch entries must be contiguous")
    if a.element_size() != 1 or b.element_size() != 1:
        raise ValueError("a and b must hold 1-byte FP8 codes (uint8 or a torch float8 dtype)")
    if scale.dtype != torch.float32 or scale.numel() != 1 or not scale.is_cuda:
        raise ValueError("scale must be a 1-element float32 CUDA tensor")
    if bias is not None and (bias.dtype != torch.bfloat16 or bias.numel() != N or not bias.is_contiguous()):
        raise ValueError("bias must be a contiguous bf16 vector of length n")
    _on_device(((a, "a"), (b, "b"), (scale, "scale"), (bias, "bias")), a.device)
    shape = (batch, M, N) if (A.dim() == 3 or B.dim() == 3) else (M, N)
    c = torch.empty(shape, dtype=torch.bfloat16, device=a.device)
    _call("mxq_mm_fp8", a.device, _ptr(A), _ptr(B), batch, M, N, K, int(ba > 1), int(bb > 1), ta, tb, f,
          _ptr(scale), _ptr(bias), _ptr(c))
    return c


def sf_to_mma(s: torch.Tensor) -> torch.Tensor:
    """Canonical scales [rows][kb] -> the GEMM's 512-byte-chunk layout (flat)."""
    if not isinstance(s, torch.Tensor) or s.dim() != 2:
        raise ValueError("s must be a 2-D tensor of scales [rows][kb]")
    _byte_tensor(s, "s")
    _on_device(((s, "s"),), s.device)
    out = torch.empty(s.numel(), dtype=torch.uint8, device=s.device)
    _call("mxq_sf_to_mma", s.device, _ptr(s), s.shape[0], s.shape[1], _ptr(out))
    return out


def last_device_status(device=None) -> int:
    """Synchronize the device's current stream and return (then clear) the
    library's device status word of that device (0, or MXQ_ERR_TIMEOUT)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return load().mxq_last_device_status(_stream(dev))
