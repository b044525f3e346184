"""Cross-rank reductions around the cast kernels.

amax_allreduce -- the amax reduction for delayed scaling.

"[PyTorch] cuda graph support" (feature list): the forward and backward
amaxes of a step are reduced across the ranks of a distributed group within
the current iteration, before the scale update, so that every rank derives
the same scale for a tensor that is sharded or replicated across the group.
The reduction is an element-wise MAX over the contiguous amax buffer (the
current row of the amax history, n fp32 values): a collective of the
communication library (NCCL for CUDA tensors, gloo for CPU tensors), called
through torch.distributed, between the cast kernels and
fp8_amax_and_scale_update.  The max of IEEE magnitudes is order-free, so
every rank ends with identical bits.

dbias_allreduce -- the bias gradient of a row-sharded dy ("[PyTorch] cuda
graph support", the DbiasCastTranspose example: db = dy.sum(dim=0)): each
rank's kernel sums its own rows, and an element-wise SUM over the ranks gives
the sum over all rows.  It reduces the fp32 db (CT_DBIAS_FP32), so the only
extra rounding is the fp32 addition of the per-rank sums; every rank ends
with identical bits.

Nothing here runs on the data path of one GPU: with world size 1 the calls
return at once.
"""
from __future__ import annotations

import torch


def amax_allreduce(amax: torch.Tensor, group=None) -> torch.Tensor:
    """In-place MAX all-reduce of an amax buffer (e.g. amax_history[0]) over
    `group` (default: the world).  Returns the tensor.  A no-op when
    torch.distributed is not initialised or the group has one rank."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return amax
    if dist.get_world_size(group) == 1:
        return amax
    if not amax.is_contiguous():
        raise ValueError("amax buffer must be contiguous")
    dist.all_reduce(amax, op=dist.ReduceOp.MAX, group=group)
    return amax


def dbias_allreduce(db: torch.Tensor, group=None) -> torch.Tensor:
    """In-place SUM all-reduce of an fp32 db buffer over `group` (default:
    the world).  Returns the tensor.  A no-op when torch.distributed is not
    initialised or the group has one rank."""
    import torch.distributed as dist
    if db.dtype != torch.float32:
        raise TypeError("dbias_allreduce reduces the fp32 db (CT_DBIAS_FP32)")
    if not (dist.is_available() and dist.is_initialized()):
        return db
    if dist.get_world_size(group) == 1:
        return db
    if not db.is_contiguous():
        raise ValueError("db buffer must be contiguous")
    dist.all_reduce(db, op=dist.ReduceOp.SUM, group=group)
    return db
