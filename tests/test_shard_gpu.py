"""The row-shard plan on one GPU: a tensor quantized as row shards gives the
bytes of the whole-tensor call.  Per-tensor FP8: shard calls without a ring
(each returns its shard amax), the MAX of those amaxes (what the all-reduce
computes across GPUs), then fp8_ring_fold -- equal, step after step, to the
whole-tensor call with its in-kernel fold, and to the oracle's host fold.
MX quantize: 32-row-aligned shards need no exchange at all."""

import numpy as np
import pytest
import torch

from block_scaled_precision_02_gb300 import inputs, shard
from oracle import formats as F
from oracle import pertensor as opt
from tests.helpers import assert_bytes_equal, f64, np_

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("orient", ["dual", "row", "col"])
def test_pertensor_row_shards_fold_like_the_whole_tensor(lib, orient):
    dev = torch.device("cuda")
    R, C, n = 512, 768, 16
    base = inputs.pertensor_base(R, C, seed=2).to(dev)
    exps = inputs.pertensor_step_exponents(16, seed=3)
    ring_whole = lib.ring_state_new(n, dev)
    ring_shard = lib.ring_state_new(n, dev)
    ring_ref = opt.ring_new(n)
    cuts = [shard.row_shard(R, r, 3, multiple=16) for r in range(3)]     # uneven: 160, 176, 176 rows
    for t, v in enumerate(exps):
        x = inputs.pertensor_step(base, v)
        x[(t * 97) % R, t] = 2.0 ** (v + 4)         # the tensor amax moves between shards
        w8, w8T, _ = lib.fp8_quantize_pertensor(x, ring_whole[n + 1:n + 2], "e4m3", orient, ring_whole, t % n)
        parts = [lib.fp8_quantize_pertensor(x[c].contiguous(), ring_shard[n + 1:n + 2], "e4m3", orient)
                 for c in cuts]
        amax = parts[0][2].clone()
        for p in parts[1:]:
            torch.maximum(amax, p[2], out=amax)      # the MAX all-reduce of the shard amaxes
        lib.ring_fold(amax, ring_shard, t % n)
        for c, (s8, s8T, _) in zip(cuts, parts):
            if w8 is not None:
                assert torch.equal(s8, w8[c]), f"x8 rows, step {t}"
            if w8T is not None:
                assert torch.equal(s8T, w8T[:, c]), f"x8T columns, step {t}"
        assert torch.equal(ring_shard.view(torch.int32), ring_whole.view(torch.int32)), f"ring step {t}"
        ring_ref = opt.ring_fold(ring_ref, float(np.max(np.abs(f64(x.cpu())))), t % n)
        assert_bytes_equal(np_(ring_shard).view(np.uint32), ring_ref.view(np.uint32), f"oracle ring step {t}")


def test_shard_helper_on_one_gpu(lib):
    """shard.pertensor_step without a process group (one rank): quantize,
    no exchange, fold -- the whole-tensor step."""
    dev = torch.device("cuda")
    x = inputs.pertensor_base(256, 512, seed=5).to(dev)
    ring_a = lib.ring_state_new(4, dev)
    ring_b = lib.ring_state_new(4, dev)
    for t in range(5):
        xt = inputs.pertensor_step(x, t - 2)
        a8, a8T, _ = shard.pertensor_step(xt, ring_a, t % 4)
        b8, b8T, _ = lib.quantize_dual(xt, ring_b[5:6], "e4m3", ring_b, t % 4)
        assert torch.equal(a8, b8) and torch.equal(a8T, b8T)
        assert torch.equal(ring_a.view(torch.int32), ring_b.view(torch.int32))


def test_fold_publishes_nothing_for_a_zero_history(lib):
    dev = torch.device("cuda")
    ring = lib.ring_state_new(4, dev)
    lib.ring_fold(torch.zeros(1, device=dev), ring, 2)
    assert np_(ring).tolist() == [0.0, 0.0, 0.0, 0.0, 1.0, 1.0, 0.0, 0.0]
    lib.ring_fold(torch.tensor([896.0], device=dev), ring, 3, 448.0, 2.0)
    assert np_(ring).tolist() == [0.0, 0.0, 0.0, 896.0, 1.0, 1.0, 0.0, 0.0]


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
@pytest.mark.parametrize("sf", ["canonical", "mma"])
def test_mx_row_shards_need_no_exchange(lib, fmt, sf):
    """MX dual quantize of 32-row-aligned row shards (128-row for the MMA
    scale layout) equals the whole-tensor call: rows of the row copy,
    columns of the transposed copy, and their scales."""
    from oracle import mx as omx
    dev = torch.device("cuda")
    R, C = 768, 512
    x = inputs.activations(R, C, seed=0).to(dev)
    mult = 128 if sf == "mma" else 32
    cuts = [shard.row_shard(R, r, 3, multiple=mult) for r in range(3)]
    qr, sr, qc, sc = lib.mx_quantize(x, fmt, "dual", "floor", sf_layout=sf)
    per = 2 if fmt == "e2m1" else 1
    if sf == "mma":
        sr = torch.from_numpy(omx.sf_from_mma(np_(sr), R, C // 32))
        sc = torch.from_numpy(omx.sf_from_mma(np_(sc), C, R // 32))
    for c in cuts:
        pr, ps, pc, pcs = lib.mx_quantize(x[c].contiguous(), fmt, "dual", "floor", sf_layout=sf)
        rows = c.stop - c.start
        if sf == "mma":
            ps = torch.from_numpy(omx.sf_from_mma(np_(ps), rows, C // 32))
            pcs = torch.from_numpy(omx.sf_from_mma(np_(pcs), C, rows // 32))
        assert torch.equal(pr, qr[c])
        assert torch.equal(ps.cpu(), sr.cpu()[c])
        assert torch.equal(pc, qc[:, c.start // per:c.stop // per])
        assert torch.equal(pcs.cpu(), sc.cpu()[:, c.start // 32:c.stop // 32])
