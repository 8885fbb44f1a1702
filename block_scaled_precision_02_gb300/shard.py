"""Row-sharded per-tensor FP8 step across ranks (one GPU per rank).

The per-tensor quantize with the delayed-scaling fold (AstrAI fp8.py: the
fold takes the tensor's amax into the history and publishes the next scale)
shards by rows.  Each rank quantizes its own row shard against the same
multiplier; the one exchange is a MAX all-reduce of the 4-byte shard amax;
then every rank folds that tensor amax into its own replica of the ring, so
all replicas stay identical to what one whole-tensor call leaves.  The MX
quantizers and the GEMM shard with no exchange at all (rows in multiples of
32, so no 32 x 1 block straddles two shards; the GEMM by M with the other
operand replicated).

Plumbing only: the quantize and the fold run in the library's kernels; the
exchange is ``torch.distributed.all_reduce`` (NCCL on GPUs).
"""

from __future__ import annotations

import sys

import torch
import torch.distributed as dist


def pertensor_step(x_shard: torch.Tensor, ring_state: torch.Tensor, hist_idx: int, fmt="e4m3",
                   orientation="dual", fp8_max: float = 448.0, pow2_margin: float = 1.0, group=None, ops=None):
    """One delayed-scaling step of a row-sharded tensor.

    ``x_shard`` is this rank's rows, ``ring_state`` this rank's replica of
    the ring [hist | scale | legacy | amax | done]; the multiplier is the
    ring's legacy slot, as in a whole-tensor step.  Returns (x8, x8T, amax)
    for the shard: x8 its rows of the tensor's x8, x8T its columns of the
    tensor's x8T, amax the tensor amax that was folded.  ``ops`` is the
    module that provides ``fp8_quantize_pertensor`` and ``ring_fold`` (the
    library's binding by default)."""
    if ops is None:
        ops = sys.modules[__package__]
    n = ring_state.numel() - 4
    x8, x8T, amax = ops.fp8_quantize_pertensor(x_shard, ring_state[n + 1:n + 2], fmt, orientation, None)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(amax, op=dist.ReduceOp.MAX, group=group)
    ops.ring_fold(amax, ring_state, hist_idx, fp8_max, pow2_margin)
    return x8, x8T, amax


def row_shard(rows: int, rank: int, world: int, multiple: int = 32) -> slice:
    """This rank's rows: consecutive, equal where possible, every boundary a
    multiple of ``multiple`` (32 keeps MX column blocks inside one shard)."""
    units = rows // multiple
    if units * multiple != rows:
        raise ValueError(f"rows ({rows}) must be a multiple of {multiple}")
    lo = (units * rank) // world
    hi = (units * (rank + 1)) // world
    return slice(lo * multiple, hi * multiple)
