"""Benchmark of the block-scaled quantization hot path on one GB300 (or N
replicas under torchrun).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = the dual-orientation MXFP8 quantize workload: 8192 x 4096 bf16
activations (N(0,1), 0.1 % outlier columns x100) to E4M3 and a same-shape
gradient (N(0,1e-3)) to E5M2, each with the floor (OCP) and the ceil scale
rule -- four quantizations, every one writing the row copy, the transposed
column copy and both scale arrays (in the GEMM's tensor-core layout), run as
two grouped launches (one per format; the same four as single-tensor calls
are reported beside them).  Each quantization reads its own input copy
(inputs larger than L2: 520 MiB touched per step); one CUDA-event pair times
each step.  ``value`` is
MX quantize GB/s (algorithmic bytes / kernel time); the same JSON line also
reports the MXFP8 and MXFP4 GEMMs (TFLOP/s), the per-tensor FP8 step with the
delayed-scaling fold, the MXFP4 Hadamard + stochastic-rounding quantizer and
the small row-wise quantize + dequantize, each against its roofline.

The other rows flush L2 (129 MB) before every timed launch by writing a
256 MiB buffer and reading it back (so its dirty lines drain before the timed
kernel); flushes are outside the timed event pairs.  Inputs are resident in
HBM when timing starts (``e2e`` repeats the step through the public Python
API with host buffers and the copies inside the timed region).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

GIB = 1 << 30
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# dense tensor-core peaks relative to bf16 (nominal 2.25 / 4.5 / 13.5 PFLOP/s)
RATIO = {"e4m3": 2.0, "e5m2": 2.0, "e2m1": 6.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "of measured"
    return dict(FALLBACK), "of fallback"


# ---------------------------------------------------------------- algorithmic bytes / flops
def mx_quant_bytes(rows, cols, fmt="e4m3", orient="dual"):
    """Bytes a quantize launch must move: read x once (bf16), write codes and
    UE8M0 scales for each requested orientation."""
    n = rows * cols
    per = (n // 2 if fmt == "e2m1" else n) + n // 32
    k = 2 if orient == "dual" else 1
    return 2 * n + k * per


def pertensor_bytes(rows, cols, orient="dual"):
    n = rows * cols
    return 2 * n + (2 if orient == "dual" else 1) * n


def gemm_flops(M, N, K):
    return 2 * M * N * K


# ---------------------------------------------------------------- multi-rank aggregation
def max_over_ranks(ms: float, world: int, device=None) -> float:
    """Slowest rank's step time (the job finishes when the last rank does)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(bytes_per_rank_step: int, world: int, ms_step_max: float) -> float:
    """Whole-job GB/s: every rank quantizes its own same-size shard (no
    data-path collective), so the job moves world x the per-rank bytes in
    the slowest rank's time."""
    return world * bytes_per_rank_step / (ms_step_max * 1e-3) / 1e9


# ---------------------------------------------------------------- timing helpers
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while the
    timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.tmp = tempfile.NamedTemporaryFile(prefix="clocks_", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.tmp, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.close()
        rows = []
        with open(self.tmp.name) as fh:
            for line in fh:
                f = [x.strip() for x in line.split(",")]
                if len(f) >= 9:
                    rows.append(f)
        os.unlink(self.tmp.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# A GPU-side spin enqueued before each timed loop, long enough for the host
# to queue every launch of the loop behind it: the event pairs then time the
# kernels, not gaps while the GPU waits for Python to submit the next launch.
HOST_LEAD_CYCLES = 60_000_000


def make_timer(torch, flush):
    """Run fn() K times, each after an L2 flush, and return the mean device
    time (ms) of fn measured with CUDA events on the current stream."""
    def run(fn, k):
        st = torch.cuda.current_stream()
        evs = []
        torch.cuda._sleep(HOST_LEAD_CYCLES)
        for _ in range(k):
            flush()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(st)
            fn()
            b.record(st)
            evs.append((a, b))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in evs)
    return run


def source_sha(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "block_scaled_precision_02_gb300", "csrc", n), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_for(kernel: str, sha: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary, or None when the kernel source changed since the counters were
    taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        d = json.load(fh)
    e = d.get(f"{kernel} {workload}")
    if not e or e.get("source_sha") != sha:
        return None
    return e.get("bytes_per_launch")


# ---------------------------------------------------------------- CPU oracle baseline
SLAB = 512          # rows of one oracle sample slab (of the 8192 x 4096 headline tensors)


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the ISA)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for ln in fh:
                if ln.lower().startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def _oracle_slab_runs():
    """The headline's four runs (E4M3 activations / E5M2 gradients, floor and
    ceil scales) on one 512-row slab of each input, as oracle arguments."""
    from block_scaled_precision_02_gb300 import inputs
    from oracle import formats as F
    from oracle import mx as omx
    a = F.bf16_bits_to_f64(inputs.bf16_bits(inputs.activations(SLAB, 4096, seed=0)))
    g = F.bf16_bits_to_f64(inputs.bf16_bits(inputs.gradients(SLAB, 4096, seed=1)))
    return [(a, F.E4M3, omx.FLOOR), (a, F.E4M3, omx.CEIL), (g, F.E5M2, omx.FLOOR), (g, F.E5M2, omx.CEIL)]


def _oracle_slab_loop(runs, t_end: float):
    """Dual-quantize the slab runs in turn until wall time t_end (at least
    one full round of four); returns (bytes, runs done, seconds)."""
    from oracle import mx as omx
    t0 = time.perf_counter()
    done = nbytes = 0
    while True:
        x, f, m = runs[done % 4]
        omx.quantize(x, f, omx.DUAL, m)
        nbytes += mx_quant_bytes(SLAB, 4096)
        done += 1
        if done % 4 == 0 and time.time() >= t_end:
            break
    return nbytes, done, time.perf_counter() - t0


def _oracle_worker(barrier, budget_s: float):
    """One process of the all-core baseline: build its inputs, start with the
    others (barrier), run its slab loop for budget_s."""
    os.environ["OMP_NUM_THREADS"] = "1"
    runs = _oracle_slab_runs()
    barrier.wait()
    return _oracle_slab_loop(runs, time.time() + budget_s)


def oracle_quant_baseline(budget_s: float = 12.0, procs: int = 1):
    """The oracle (numpy, float64, as it stands) on a bounded sample of the
    same workload: dual quantize of 512-row slabs of the activation (E4M3)
    and gradient (E5M2) tensors, floor and ceil, for about budget_s.  With
    procs > 1 that many spawned processes run it side by side over the same
    window (each numpy process is single-threaded here), and the value is
    their summed bytes over the window."""
    if procs <= 1:
        runs = _oracle_slab_runs()
        nbytes, done, dt = _oracle_slab_loop(runs, time.time() + budget_s)
        return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                "sample": f"{done} dual quantize runs of {SLAB}x4096 row slabs (E4M3/E5M2 x floor/ceil), "
                          f"{dt:.1f} s, one process"}
    import multiprocessing as mp
    ctx = mp.get_context("spawn")            # never fork a process that holds a CUDA context
    with ctx.Manager() as mgr, ctx.Pool(procs) as pool:
        barrier = mgr.Barrier(procs)
        res = pool.starmap(_oracle_worker, [(barrier, budget_s)] * procs)
    nbytes = sum(r[0] for r in res)
    done = sum(r[1] for r in res)
    dt = max(r[2] for r in res)
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": procs, "kind": "oracle",
            "sample": f"{done} dual quantize runs of {SLAB}x4096 row slabs (E4M3/E5M2 x floor/ceil) in {procs} "
                      f"processes over {dt:.1f} s"}


def cpu_baselines(budget_s: float = 10.0):
    """The oracle timed on one core and on every core of the host, with the
    core count and CPU model."""
    n = os.cpu_count() or 1
    one = oracle_quant_baseline(budget_s, 1)
    allc = oracle_quant_baseline(budget_s, n) if n > 1 else dict(one)
    return {**one, "all_cores": allc, "nproc": n, "cpu_model": cpu_model()}


def oracle_gemm_baseline(budget_s: float = 6.0):
    """Oracle float64 dequantized product on 128 x 128 output tiles of the
    8192 x 4096 x 4096 MXFP8 GEMM (numpy matmul, threads as numpy uses)."""
    import numpy as np
    from block_scaled_precision_02_gb300 import inputs
    from oracle import formats as F
    from oracle import gemm as og
    from oracle import mx as omx
    a = omx.quantize(F.bf16_bits_to_f64(inputs.bf16_bits(inputs.activations(128, 4096, seed=0))), F.E4M3)
    b = omx.quantize(F.bf16_bits_to_f64(inputs.bf16_bits(inputs.weights(128, 4096, seed=4))), F.E4M3)
    t0 = time.perf_counter()
    tiles = 0
    while time.perf_counter() - t0 < budget_s or tiles == 0:
        og.reference(a["q_row"], a["s_row"], b["q_row"], b["s_row"], F.E4M3)
        tiles += 1
    dt = time.perf_counter() - t0
    return {"value": tiles * gemm_flops(128, 128, 4096) / dt / 1e12, "unit": "TFLOP/s",
            "cores": os.cpu_count(), "kind": "oracle", "cpu_model": cpu_model(),
            "threads": "the float64 matmul runs in numpy's BLAS, which threads over the host cores; "
                       "the dequantize is single-threaded numpy",
            "sample": f"{tiles} output tiles of 128x128 (K=4096, dequantize + float64 matmul), {dt:.1f} s"}


# ---------------------------------------------------------------- measured rows besides the headline
def gemm_part(args, mxq, X, q, outs, timed, bf16, peak_src, gemm_rows):
    """MXFP8 GEMMs 8192x4096x4096 and 8192x14336x4096 on operands from our
    quantizer (A = the activation quantized by the headline step), the
    mixed-format products of the headline's E5M2 gradient with the E4M3
    weights and of the activation with E2M1 weights, the MX-output and
    per-tensor products."""
    aq, as_, _, _ = outs[0]
    M, K = 8192, 4096
    W, W2 = X["W"], X["W2"]
    wq, ws, _, _ = q(W, "e4m3", "floor", "row")
    w2q, w2s, _, _ = q(W2, "e4m3", "floor", "row")
    gq, gs, _, _ = outs[2]                 # the E5M2 gradient of the headline step (row copy)
    n = 0
    for name, (a2, a2s, fa, bq, bs, N) in {
            "mxfp8_8192x4096x4096": (aq, as_, "e4m3", wq, ws, 4096),
            "mxfp8_8192x14336x4096": (aq, as_, "e4m3", w2q, w2s, 14336),
            "mxfp8_mixed_e5m2_x_e4m3_8192x4096x4096": (gq, gs, "e5m2", wq, ws, 4096)}.items():
        fn = lambda a2=a2, a2s=a2s, fa=fa, bq=bq, bs=bs: mxq.mx_gemm(a2, a2s, bq, bs, fa, b_fmt="e4m3")
        for _ in range(max(3, args.warmup)):
            fn()
        ms = timed(fn, args.steps)
        n += args.steps
        tf = gemm_flops(M, N, K) / (ms * 1e-3) / 1e12
        pk = bf16 * RATIO["e4m3"]
        gemm_rows.append({"workload": name, "ms": round(ms, 4), "tflops": round(tf, 1),
                          "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": round(pk, 1),
                                       "unit": "TFLOP/s", "frac": round(tf / pk, 4),
                                       "peak_source": f"bf16 burst x {RATIO['e4m3']} ({peak_src})",
                                       "traffic": traffic_for("mx_gemm_pair_kernel", source_sha("gemm.cu"), name)}})
    # MXFP8 activations times MXFP4 weights (the weights quantized to E2M1 by
    # our quantizer; the E2M1 codes are widened on their way into shared memory)
    w4q, w4s, _, _ = q(W, "e2m1", "floor", "row")
    fn = lambda: mxq.mx_gemm(aq, as_, w4q, w4s, "e4m3", b_fmt="e2m1")
    n += extra_gemm_row(args, fn, timed, "mxfp8_x_mxfp4_e4m3_x_e2m1_8192x4096x4096", M, 4096, K, bf16, peak_src,
                        gemm_rows)
    # the same MXFP8 product written as MX E4M3 codes + scales (MMA layout:
    # the next GEMM's A operand) straight from the accumulator
    fn = lambda: mxq.mx_gemm_mx_out(aq, as_, wq, ws, "e4m3", out_fmt="e4m3", out_sf_layout="mma")
    n += extra_gemm_row(args, fn, timed, "mxfp8_gemm_mx_e4m3_out_8192x4096x4096", M, 4096, K, bf16, peak_src,
                        gemm_rows)
    # row and transposed column blocks together (the copies a backward pass reads)
    fn = lambda: mxq.mx_gemm_mx_out(aq, as_, wq, ws, "e4m3", out_fmt="e4m3", out_sf_layout="mma",
                                    orientation="dual")
    n += extra_gemm_row(args, fn, timed, "mxfp8_gemm_mx_e4m3_dual_out_8192x4096x4096", M, 4096, K, bf16, peak_src,
                        gemm_rows)
    # per-tensor FP8 product with scale and bias (mm_fp8): the per-tensor
    # quantizer's E4M3 activations times E4M3 weights
    x8 = mxq.fp8_quantize_pertensor(X["A"], X["one"], "e4m3", "row")[0]
    w8 = mxq.fp8_quantize_pertensor(W, X["one"], "e4m3", "row")[0]
    fn = lambda: mxq.mm_fp8(x8, w8, X["one"], trans_b=True, bias=X["bias"], fmt="e4m3")
    n += extra_gemm_row(args, fn, timed, "fp8_pertensor_gemm_bias_8192x4096x4096", M, 4096, K, bf16, peak_src,
                        gemm_rows)
    # a product whose last wave of 256 x 256 tiles is sparse (80 tiles on the
    # GPU's 76 CTA pairs): the stream-K schedule (default) against the plain one
    Ms, Ns, Ks = 2560, 2048, 16384
    xs = q(inputs_tail(X, "a", Ms, Ks), "e4m3", "floor", "row")
    ws_ = q(inputs_tail(X, "b", Ns, Ks), "e4m3", "floor", "row")
    fn = lambda: mxq.mx_gemm(xs[0], xs[1], ws_[0], ws_[1], "e4m3")
    n += extra_gemm_row(args, fn, timed, "mxfp8_sparse_tail_stream_k_2560x2048x16384", Ms, Ns, Ks, bf16, peak_src,
                        gemm_rows)
    fn = lambda: mxq.mx_gemm(xs[0], xs[1], ws_[0], ws_[1], "e4m3", stream_k=False)
    n += extra_gemm_row(args, fn, timed, "mxfp8_sparse_tail_plain_2560x2048x16384", Ms, Ns, Ks, bf16, peak_src,
                        gemm_rows)
    # the default layout of mm_fp8: b stored row-major [K][N] (the per-tensor
    # quantizer's transposed copy of the [N][K] weight), read N-contiguous
    w8kn = mxq.fp8_quantize_pertensor(W, X["one"], "e4m3", "col")[1]
    fn = lambda: mxq.mm_fp8(x8, w8kn, X["one"], bias=X["bias"], fmt="e4m3")
    n += extra_gemm_row(args, fn, timed, "fp8_pertensor_gemm_bias_kn_weight_8192x4096x4096", M, 4096, K, bf16,
                        peak_src, gemm_rows)
    return n


def inputs_tail(X, which, rows, K):
    """Operands of the sparse-tail product: N(0,1) activations with outlier
    columns (seed 0) and N(0,0.02^2) weights (seed 4), on the device."""
    from block_scaled_precision_02_gb300 import inputs
    dev = X["A"].device
    if which == "a":
        return inputs.activations(rows, K, seed=0).to(dev)
    return inputs.weights(rows, K, seed=4).to(dev)


def extra_gemm_row(args, fn, timed, name, M, N, K, bf16, peak_src, gemm_rows):
    for _ in range(max(3, args.warmup)):
        fn()
    ms = timed(fn, args.steps)
    tf = gemm_flops(M, N, K) / (ms * 1e-3) / 1e12
    pk = bf16 * RATIO["e4m3"]
    gemm_rows.append({"workload": name, "ms": round(ms, 4), "tflops": round(tf, 1),
                      "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": round(pk, 1),
                                   "unit": "TFLOP/s", "frac": round(tf / pk, 4),
                                   "peak_source": f"bf16 burst x {RATIO['e4m3']} ({peak_src})",
                                   "traffic": traffic_for("mx_gemm_pair_kernel", source_sha("gemm.cu"), name)}})
    return args.steps


def fp4_part(args, mxq, X, q, timed, bf16, peak_src, gemm_rows):
    """MXFP4 path: Hadamard + stochastic-rounding quantize of the 4096 x 14336
    gradient (key 0, signs from seed 7), Hadamard + RNE of the operand, and the
    MXFP4 GEMM 4096 x 4096 x 14336."""
    G5, B5 = X["G5"], X["B5"]
    fp4q = lambda: q(G5, "e2m1", "floor", "row", rounding="sr", hadamard32=True, sr_key=0, hadamard_seed=7)
    for _ in range(3):
        g5 = fp4q()
    ms_q5 = timed(fp4q, args.steps)
    # the same quantize with the four-draws-per-call option
    fp4q4 = lambda: q(G5, "e2m1", "floor", "row", rounding="sr4", hadamard32=True, sr_key=0, hadamard_seed=7)
    for _ in range(3):
        fp4q4()
    ms_q5b = timed(fp4q4, args.steps)
    # ceil scales (the recipe runs both scale rules)
    fp4qc = lambda: q(G5, "e2m1", "ceil", "row", rounding="sr", hadamard32=True, sr_key=0, hadamard_seed=7)
    for _ in range(3):
        fp4qc()
    ms_q5c = timed(fp4qc, args.steps)
    b5 = q(B5, "e2m1", "floor", "row", hadamard32=True, hadamard_seed=7)
    fn5 = lambda: mxq.mx_gemm(g5[0], g5[1], b5[0], b5[1], "e2m1")
    for _ in range(3):
        fn5()
    ms5 = timed(fn5, args.steps)
    tf5 = gemm_flops(4096, 4096, 14336) / (ms5 * 1e-3) / 1e12
    pk5 = bf16 * RATIO["e2m1"]
    gemm_rows.append({"workload": "mxfp4_4096x4096x14336", "ms": round(ms5, 4), "tflops": round(tf5, 1),
                      "roofline": {"bound": "tensor", "achieved": round(tf5, 1), "peak": round(pk5, 1),
                                   "unit": "TFLOP/s", "frac": round(tf5 / pk5, 4),
                                   "peak_source": f"bf16 burst x {RATIO['e2m1']} ({peak_src})",
                                   "traffic": traffic_for("mx_gemm_pair_kernel", source_sha("gemm.cu"),
                                                          "mxfp4_4096x4096x14336")}})
    # the same product written as MX E2M1 codes + scales (MMA layout: the
    # next MXFP4 product's A operand) straight from the accumulator
    fn6 = lambda: mxq.mx_gemm_mx_out(g5[0], g5[1], b5[0], b5[1], "e2m1", out_fmt="e2m1", out_sf_layout="mma")
    for _ in range(3):
        fn6()
    ms6 = timed(fn6, args.steps)
    tf6 = gemm_flops(4096, 4096, 14336) / (ms6 * 1e-3) / 1e12
    gemm_rows.append({"workload": "mxfp4_gemm_mx_e2m1_out_4096x4096x14336", "ms": round(ms6, 4),
                      "tflops": round(tf6, 1),
                      "roofline": {"bound": "tensor", "achieved": round(tf6, 1), "peak": round(pk5, 1),
                                   "unit": "TFLOP/s", "frac": round(tf6 / pk5, 4),
                                   "peak_source": f"bf16 burst x {RATIO['e2m1']} ({peak_src})",
                                   "traffic": None}})
    return (ms_q5, ms_q5b, ms_q5c), 5 * args.steps


def pertensor_part(args, mxq, X, timed):
    """Per-tensor FP8 E4M3 dual quantize of 4096 x 14336 with the in-kernel
    fold into a 16-entry history, steps taken in sequence: step t quantizes
    base * 2^v_t (v_t from the seeded step law, the 16 step inputs resident
    on the device) with the multiplier the previous fold published."""
    from block_scaled_precision_02_gb300 import inputs
    X3 = X["X3"]
    xs = [inputs.pertensor_step(X3, v) for v in inputs.pertensor_step_exponents(16, seed=3)]
    ring = mxq.ring_state_new(16, X3.device)
    t3 = {"k": 0}

    def pt():
        t = t3["k"] % 16
        mxq.quantize_dual(xs[t], ring[17:18], "e4m3", ring, t)
        t3["k"] += 1
    for _ in range(3):
        pt()
    k = max(16, args.steps)
    ms_dual = timed(pt, k)

    def ptt():                              # transposed output only (x8T), same ring
        t = t3["k"] % 16
        mxq.quantize(xs[t], ring[17:18], "e4m3", True, ring, t)
        t3["k"] += 1
    for _ in range(3):
        ptt()
    return (ms_dual, timed(ptt, k)), 2 * k


def small_part(args, mxq, X, timed):
    """256 x 512 row-wise E4M3 quantize (floor, RNE) and its dequantize."""
    X1 = X["X1"]
    q1 = lambda: mxq.mx_quantize(X1, "e4m3", "row", "floor")
    r1 = q1()
    ms1q = timed(q1, args.steps)
    d1 = lambda: mxq.mx_dequantize(r1[0], r1[1], "e4m3")
    ms1d = timed(d1, args.steps)
    return ms1q, ms1d, 2 * args.steps


def alu_roofline(key: str, elems: int, ms: float, sm_mhz: float):
    """Integer-issue roofline of an ALU-bound quantizer path: the thread
    instructions it executes per element (profiles/alu.json, from one ncu
    capture of the same kernel source) times the elements per second, against
    the issue peak of the SMs (4 schedulers x 32 lanes, one instruction per
    clock each, at the maximum SM clock), with the per-pipe busy fractions of
    the capture beside it.  None once the kernel source differs from the
    captured one."""
    p = os.path.join(ROOT, "profiles", "alu.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        e = json.load(fh).get(f"quant_tiles_kernel {key}")
    if not e or e.get("source_sha") != source_sha("quantize.cu"):
        return None
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    achieved = e["inst_per_element"] * elems / (ms * 1e-3)
    peak = sms * 128 * sm_mhz * 1e6
    r = {"bound": "alu", "achieved": round(achieved / 1e12, 2), "peak": round(peak / 1e12, 2),
         "unit": "T thread-instructions/s", "frac": round(achieved / peak, 4),
         "inst_per_element": e["inst_per_element"], "peak_source": f"{sms} SMs x 128 lanes x {sm_mhz:.0f} MHz"}
    if "pipe_busy_pct" in e:
        r["pipe_busy_pct_ncu"] = e["pipe_busy_pct"]
    return r


def hbm_row(nbytes, ms, hbm, note=None):
    gbs = nbytes / (ms * 1e-3) / 1e9
    r = {"ms": round(ms, 4), "gbs": round(gbs, 1),
         "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                      "frac": round(gbs / hbm, 4), "algorithmic_bytes_per_launch": nbytes}}
    if note:
        r["roofline"]["note"] = note
    return r


# ---------------------------------------------------------------- reference arm
def run_reference(args, rank, world):
    """The oracle as the reference arm: each step is the headline's four runs
    (E4M3 / E5M2 x floor / ceil dual quantize) on one 512-row slab of each
    8192 x 4096 input -- a bounded sample of the headline step -- timed on the
    host, one process.  ms_per_step is the measured time of that sampled
    step; the time a whole 8192-row step would take at the same rate is
    reported separately as a projection."""
    if rank != 0:
        return 0
    runs = _oracle_slab_runs()
    from oracle import mx as omx

    def step():
        for x, f, m in runs:
            omx.quantize(x, f, omx.DUAL, m)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    per = []
    for _ in range(args.steps):
        a = time.perf_counter()
        step()
        per.append(time.perf_counter() - a)
    el = time.perf_counter() - t0
    sample_bytes = 4 * mx_quant_bytes(SLAB, 4096)
    ms = statistics.mean(per) * 1e3
    v = sample_bytes / (ms * 1e-3) / 1e9
    full_bytes = 4 * mx_quant_bytes(8192, 4096)
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded numpy, rounded to bf16)",
            "config": {"workload": WORKLOAD, "sampled": True,
                       "sample": (f"each step: the four headline runs on one {SLAB}-row slab of each 8192x4096 "
                                  f"input ({sample_bytes} algorithmic bytes, {SLAB / 8192:.4f} of a full step)"),
                       "bytes_per_step": sample_bytes},
            "projected_full_step_ms": round(full_bytes / (v * 1e9) * 1e3, 1),
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"{args.steps} sampled steps of {SLAB}-row slabs, one process",
                             "cpu_model": cpu_model(), "nproc": os.cpu_count()},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s_timed_steps": round(el, 2)}
    print(json.dumps(line), flush=True)
    return 0


METRIC = "MX quantize GB/s (% of HBM peak); MX GEMM TFLOP/s (% of tensor peak)"
WORKLOAD = ("mx_dual_quantize 8192x4096 bf16: activations->E4M3 and gradients->E5M2, "
            "floor-OCP and ceil scales, row + transposed column copies, MMA scale layout")


# ---------------------------------------------------------------- our arm
def run_ours(args, rank, world):
    import torch
    import block_scaled_precision_02_gb300 as mxq
    from block_scaled_precision_02_gb300 import inputs

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    mxq.load()
    peaks, peak_src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    bf16 = float(peaks["bf16_tflops"])
    sm_max = float(peaks.get("sm_max_mhz", 2070.0))

    # L2 flush: write a 256 MiB buffer (twice the 129 MB L2), then read it
    # back so the dirty lines are written out here, outside the timed pair,
    # and the timed kernel starts on a cold, clean L2
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_sink = torch.empty(1, dtype=torch.int64, device=dev)

    def flush():
        flush_buf.fill_(1)
        torch.sum(flush_buf.view(torch.int64), dim=0, out=flush_sink[0])
    timed = make_timer(torch, flush)
    launches = 0

    # ---------------- inputs resident in HBM
    A_h = inputs.activations(8192, 4096, seed=0)
    G_h = inputs.gradients(8192, 4096, seed=1)
    A, G = A_h.to(dev), G_h.to(dev)
    M, K = A.shape
    X = {}
    if args.case in ("all", "gemm"):
        X["W"] = inputs.weights(4096, 4096, seed=4).to(dev)
        X["W2"] = inputs.weights(14336, 4096, seed=5).to(dev)
        X["A"] = A
        X["one"] = torch.ones(1, dtype=torch.float32, device=dev)
        X["bias"] = inputs.weights(1, 4096, seed=9).reshape(4096).to(dev)
    if args.case in ("all", "fp4"):
        X["G5"] = inputs.heavy_gradient().to(dev)
        X["B5"] = inputs.fp4_operand().to(dev)
    if args.case in ("all", "pertensor"):
        X["X3"] = inputs.pertensor_base().to(dev)
    if args.case in ("all", "small"):
        X["X1"] = inputs.small_rowwise().to(dev)

    def q(x, fmt, mode, orient="dual", **kw):
        return mxq.mx_quantize(x, fmt, orient, mode, sf_layout="mma", **kw)

    # each launch of a step reads its own copy of its input and writes its own
    # outputs: a step touches 4 x (64 MiB in + 66 MiB out) = 520 MiB, four
    # times the L2, so every launch starts with its input out of L2
    A2, G2 = A.clone(), G.clone()
    runs = [(A, "e4m3", "floor"), (A2, "e4m3", "ceil"), (G, "e5m2", "floor"), (G2, "e5m2", "ceil")]
    # pre-allocate outputs so the timed step is the kernels only
    outs = []
    for x, fmt, mode in runs:
        outs.append(q(x, fmt, mode))
    L = mxq.load()
    stream = lambda: __import__("ctypes").c_void_p(torch.cuda.current_stream(dev).cuda_stream)

    def launch_quant(i):
        x, fmt, mode = runs[i]
        qr, sr, qc, sc = outs[i]
        rc = L.mxq_quantize(mxq._ptr(x), M, K, K, mxq._FMT[fmt], mxq.DUAL, mxq._SCALE[mode], mxq.RNE, 0, 0, 7,
                            mxq.SF_MMA, mxq._ptr(qr), mxq._ptr(sr), mxq._ptr(qc), mxq._ptr(sc), stream())
        assert rc == 0, rc

    # the step as the headline runs it: two grouped launches (one per format),
    # each quantizing its tensor's two copies with floor and ceil scales
    def group_jobs(idx):
        jobs = (mxq.QuantJob * len(idx))()
        for k, i in enumerate(idx):
            x, fmt, mode = runs[i]
            qr, sr, qc, sc = outs[i]
            jobs[k] = mxq.QuantJob(x.data_ptr(), M, K, K, mxq._SCALE[mode], qr.data_ptr(), sr.data_ptr(),
                                   qc.data_ptr(), sc.data_ptr())
        return jobs
    groups = [(group_jobs([0, 1]), "e4m3"), (group_jobs([2, 3]), "e5m2")]

    def launch_group(g):
        jobs, fmt = groups[g]
        rc = L.mxq_quantize_group(jobs, len(jobs), mxq._FMT[fmt], mxq.DUAL, mxq.SF_MMA, stream())
        assert rc == 0, rc

    # clocks are sampled from the warm-up through the last timed launch
    sampler = ClockSampler(local)
    sampler.start()
    # ---------------- warmup
    for _ in range(args.warmup):
        for g in range(2):
            launch_group(g)
        for i in range(4):
            launch_quant(i)
    torch.cuda.synchronize()

    # ---------------- timed region: K steps of 2 grouped quantize launches
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    st = torch.cuda.current_stream(dev)
    evs = []
    torch.cuda._sleep(HOST_LEAD_CYCLES)
    for _ in range(args.steps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(st)
        for g in range(2):
            launch_group(g)
            launches += 1
        b.record(st)
        evs.append((a, b))
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - t_wall
    per_step = [a.elapsed_time(b) for a, b in evs]
    ms_step = statistics.mean(per_step)
    per_launch = [t / 2 for t in per_step]
    # the same step as four single-tensor calls (mxq_quantize), timed the same way
    evs1 = []
    torch.cuda._sleep(HOST_LEAD_CYCLES)
    for _ in range(args.steps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(st)
        for i in range(4):
            launch_quant(i)
        b.record(st)
        evs1.append((a, b))
    torch.cuda.synchronize()
    ms_step_single = statistics.mean(a.elapsed_time(b) for a, b in evs1)
    # for reference: one single-tensor launch alone after an L2 flush (write + read-back)
    iso_ms = timed(lambda: launch_quant(0), 20)
    launch_detail = {"headline_steps": launches, "single_call_steps": 4 * args.steps, "headline_isolated": 20}
    launches += 4 * args.steps + 20
    ms_step = max_over_ranks(ms_step, world, dev)
    step_bytes = 4 * mx_quant_bytes(M, K)
    value = weak_scaling_value(step_bytes, world, ms_step)
    launch_ms = statistics.mean(per_launch)
    ach = 2 * mx_quant_bytes(M, K) / (launch_ms * 1e-3) / 1e9          # a launch quantizes two tensors

    gemm_rows, ms3, ms_q5, ms1q, ms1d = [], None, None, None, None
    b3 = pertensor_bytes(4096, 14336)
    b_q5 = mx_quant_bytes(4096, 14336, "e2m1", "row")
    rows_before = launches
    if args.case in ("all", "gemm"):
        launches += gemm_part(args, mxq, X, q, outs, timed, bf16, peak_src, gemm_rows)
    if args.case in ("all", "fp4"):
        ms_q5, n = fp4_part(args, mxq, X, q, timed, bf16, peak_src, gemm_rows)
        launches += n
    if args.case in ("all", "pertensor"):
        ms3, n = pertensor_part(args, mxq, X, timed)
        launches += n
    if args.case in ("all", "small"):
        ms1q, ms1d, n = small_part(args, mxq, X, timed)
        launches += n
    clocks = sampler.stop()
    if args.case != "all":
        if rank == 0:
            print(json.dumps({"case": args.case, "quant_ms_per_step": ms_step,
                              "quant_ms_per_step_single_calls": ms_step_single, "gemm": gemm_rows, "pertensor_ms": ms3,
                              "fp4_quant_ms": ms_q5, "small_us": [ms1q, ms1d], "clocks": clocks}), flush=True)
        return 0
    # ---------------- e2e through the public API: host buffers, copies inside
    A_pin, G_pin = A_h.pin_memory(), G_h.pin_memory()
    out_pin = [tuple(torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in o) for o in outs]
    # two device copies of the inputs, used by alternate steps, so the next
    # step's input copy overlaps this step's kernels
    A_d = [torch.empty_like(A) for _ in range(2)]
    G_d = [torch.empty_like(G) for _ in range(2)]

    # Three streams: inputs in, quantize, results out.  The host link is
    # full duplex, so the next input copy, the kernels and the previous
    # result copies overlap; every byte still crosses inside the timed loop.
    s_cmp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    kernels_done = [None, None]                 # per input set: the last step's kernels on it
    step_no = {"k": 0}

    def e2e_step():
        b = step_no["k"] % 2
        step_no["k"] += 1
        if kernels_done[b] is not None:
            s_in.wait_event(kernels_done[b])    # the step before last is done with this input set
        with torch.cuda.stream(s_in):
            A_d[b].copy_(A_pin, non_blocking=True)
            ev_a = s_in.record_event()
            G_d[b].copy_(G_pin, non_blocking=True)
            ev_g = s_in.record_event()
        for i, (x, fmt, mode) in enumerate(((A_d[b], "e4m3", "floor"), (A_d[b], "e4m3", "ceil"),
                                             (G_d[b], "e5m2", "floor"), (G_d[b], "e5m2", "ceil"))):
            s_cmp.wait_event(ev_a if i < 2 else ev_g)
            res = q(x, fmt, mode)
            done = s_cmp.record_event()
            s_out.wait_event(done)
            with torch.cuda.stream(s_out):
                for h, d in zip(out_pin[i], res):
                    d.record_stream(s_out)      # not reused before its copy has finished
                    h.copy_(d, non_blocking=True)
        kernels_done[b] = s_cmp.record_event()
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - t0) / args.steps
    launch_detail["rows"] = launches - rows_before
    launch_detail["e2e"] = 4 * args.steps
    launches += 4 * args.steps
    h2d = A.numel() * 2 + G.numel() * 2
    d2h = sum(t.numel() for o in outs for t in o)

    if rank != 0:
        return 0
    cpu = cpu_baselines()
    gcpu = oracle_gemm_baseline()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "ms_per_step_median": round(statistics.median(per_step), 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u8", "data": "synthetic (seeded numpy, rounded to bf16)",
        "config": {"workload": WORKLOAD, "rows": M, "cols": K, "launches_per_step": 2,
                   "grouping": ("two mxq_quantize_group launches per step, E4M3 [floor, ceil] on the activations' "
                                "two copies and E5M2 [floor, ceil] on the gradients' two copies; the same bytes as "
                                "four mxq_quantize calls (reported under rows.dual_quantize_step_four_single_calls)"),
                   "l2": ("inputs larger than L2: each quantize of a step reads its own 64 MiB input copy and "
                          "writes its own outputs (520 MiB per step, 4x the 129 MB L2); one event pair per step"),
                   "bytes_per_step": step_bytes,
                   "isolated_launch_us": round(iso_ms * 1e3, 2),
                   "isolated_launch_note": "one launch after an L2 flush (256 MiB written then read back), event-timed"},
        "roofline": {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(ach / hbm, 4), "peak_source": f"hbm_gbs ({peak_src})",
                     "traffic": traffic_for("quant_tiles_kernel", source_sha("quantize.cu"),
                                            "group_dual_e4m3_floor_ceil_8192x4096"),
                     "algorithmic_bytes_per_launch": 2 * mx_quant_bytes(M, K)},
        "clocks": clocks,
        "e2e": {"value": round(step_bytes / e2e_s / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_s * 1e3, 3),
                "api": "block_scaled_precision_02_gb300.mx_quantize (pinned host in, pinned host out)",
                "streams": ("inputs in, quantize and results out on three streams (copies overlap the kernels and "
                            "each other); two device input buffers used by alternate steps")},
        "gpu_launches": launches,
        "gpu_launches_detail": launch_detail,
        "gemm": {"metric": "MX GEMM TFLOP/s", "rows": gemm_rows, "cpu_baseline": gcpu},
        "rows": {
            "dual_quantize_step_four_single_calls": dict(
                hbm_row(step_bytes, ms_step_single, hbm, "the headline step as four mxq_quantize launches"),
                ms_per_launch=round(ms_step_single / 4, 4)),
            "pertensor_fp8_ring_4096x14336_dual": hbm_row(b3, ms3[0], hbm),
            "pertensor_fp8_ring_4096x14336_transposed": hbm_row(pertensor_bytes(4096, 14336, "col"), ms3[1], hbm),
            "mxfp4_hadamard_sr_quantize_4096x14336": dict(hbm_row(
                b_q5, ms_q5[0], hbm, "one Philox-4x32-10 draw per element: integer-ALU bound"),
                alu_roofline=alu_roofline("sr_hadamard_e2m1_4096x14336", 4096 * 14336, ms_q5[0], sm_max)),
            "mxfp4_hadamard_sr_ceil_quantize_4096x14336": hbm_row(
                b_q5, ms_q5[2], hbm, "ceil scales; one Philox-4x32-10 draw per element"),
            "mxfp4_hadamard_sr4_quantize_4096x14336": dict(hbm_row(
                b_q5, ms_q5[1], hbm, "option SR4: four draws per Philox-4x32-10 call"),
                alu_roofline=alu_roofline("sr4_hadamard_e2m1_4096x14336", 4096 * 14336, ms_q5[1], sm_max)),
            "small_rowwise_256x512": {"quantize_us": round(ms1q * 1e3, 2), "dequantize_us": round(ms1d * 1e3, 2)},
        },
        "cpu_baseline": cpu,
        "wall_s_timed_region": round(wall, 3),
    }
    # a compact copy of every row's time and roofline fraction, last on the
    # line so that a reader who keeps only its tail still has all of them
    line["summary"] = {
        "headline": {"us_per_launch": round(launch_ms * 1e3, 2), "launches_per_step": 2,
                     "frac": line["roofline"]["frac"]},
        "gemm": {r["workload"]: [r["ms"], r["roofline"]["frac"]] for r in gemm_rows},
        "quant": {k: [v["ms"], v["roofline"]["frac"]] for k, v in line["rows"].items() if "ms" in v},
        "cpu_gbs": {"one_core": round(cpu["value"], 4), "all_cores": round(cpu["all_cores"]["value"], 4),
                    "nproc": cpu["nproc"]},
        "clocks_sm_mhz": clocks.get("sm_mhz"),
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--case", choices=["all", "quant", "gemm", "fp4", "pertensor", "small"], default="all",
                    help="run only one part (for profiling); the contract line needs 'all'")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if world > 1:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        torch.distributed.init_process_group("nccl")
    try:
        return run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
