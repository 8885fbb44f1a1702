"""The row-sharded per-tensor FP8 step on CPU ranks (gloo, world size 2):
each rank quantizes its row shard, the shard amaxes meet in one MAX
all-reduce, and every rank folds the tensor amax into its own replica of the
ring.  The quantize and the fold are the oracle's here (CPU tensors), so the
test checks the exchange wiring: the shards' outputs put together, and every
rank's ring, equal one whole-tensor step of the oracle, step after step."""

import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from block_scaled_precision_02_gb300 import inputs, shard
from oracle import formats as F
from oracle import pertensor as opt

ROWS, COLS, STEPS, HIST = 96, 64, 5, 4


class OracleOps:
    """fp8_quantize_pertensor / ring_fold with the binding's signatures,
    computed by the oracle on CPU tensors."""

    @staticmethod
    def fp8_quantize_pertensor(x, scale, fmt, orientation, ring_state):
        assert ring_state is None
        xv = F.bf16_bits_to_f64(inputs.bf16_bits(x))
        x8, x8T, amax = opt.quantize_pertensor(xv, float(scale[0]), F.fmt(fmt))
        return torch.from_numpy(x8), torch.from_numpy(x8T), torch.tensor([amax], dtype=torch.float32)

    @staticmethod
    def ring_fold(amax, ring_state, hist_idx, fp8_max, pow2_margin):
        r = opt.ring_fold(ring_state.numpy(), float(amax[0]), hist_idx, fp8_max, pow2_margin)
        ring_state.copy_(torch.from_numpy(r))


def _step_input(t):
    base = inputs.pertensor_base(ROWS, COLS, seed=2)
    v = inputs.pertensor_step_exponents(STEPS, seed=3)[t]
    x = inputs.pertensor_step(base, v)
    # make a different rank hold the tensor amax on different steps
    hot = (t * 37) % ROWS
    x[hot, t % COLS] = torch.tensor(3.0 * (t + 1), dtype=torch.bfloat16)
    return x


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sl = shard.row_shard(ROWS, rank, world)
        ring = torch.zeros(HIST + 4, dtype=torch.float32)
        ring[HIST] = ring[HIST + 1] = 1.0
        out = []
        for t in range(STEPS):
            x8, x8T, amax = shard.pertensor_step(_step_input(t)[sl], ring, t % HIST, "e4m3", "dual", 448.0, 1.0,
                                                 ops=OracleOps)
            out.append((x8.numpy().copy(), x8T.numpy().copy(), float(amax[0]), ring.numpy().copy()))
        q.put((rank, sl.start, sl.stop, out))
    finally:
        dist.destroy_process_group()


def test_row_shards_with_max_exchange_equal_the_whole_tensor_step():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    ring_ref = opt.ring_new(HIST)
    holders = set()
    for t in range(STEPS):
        xv = F.bf16_bits_to_f64(inputs.bf16_bits(_step_input(t)))
        m = float(ring_ref[HIST + 1])
        r8, r8T, ramax = opt.quantize_pertensor(xv, m, F.E4M3)
        ring_ref = opt.ring_fold(ring_ref, ramax, t % HIST)
        for rank, lo, hi, out in res:
            x8, x8T, amax, ring = out[t]
            assert np.array_equal(x8, r8[lo:hi]), (t, rank)
            assert np.array_equal(x8T, r8T[:, lo:hi]), (t, rank)
            assert amax == ramax, (t, rank)
            assert np.array_equal(ring.view(np.uint32), ring_ref.view(np.uint32)), (t, rank)
            if np.max(np.abs(xv[lo:hi])) == ramax:
                holders.add(rank)
    assert holders == {0, 1}          # the exchange mattered on both sides


def test_row_shards_are_32_row_aligned_and_cover_the_tensor():
    for rows, world in ((96, 2), (4096, 3), (8192, 8), (32, 4)):
        cuts = [shard.row_shard(rows, r, world) for r in range(world)]
        assert cuts[0].start == 0 and cuts[-1].stop == rows
        for a, b in zip(cuts, cuts[1:]):
            assert a.stop == b.start
        assert all(c.start % 32 == 0 and c.stop % 32 == 0 for c in cuts)
