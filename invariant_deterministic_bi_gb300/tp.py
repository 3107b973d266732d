"""Tensor-parallel glue for the deterministic all-reduce + RMSNorm.

The pages' fix for non-determinism under tensor parallelism is a reduction
whose order does not vary (vLLM PR #51292, root-cause discussion: a
fixed-order reduction is bitwise-stable). Here every rank gathers all ranks'
partial rows, indexed by rank, and reduces them with bi_rank_sum_rmsnorm in
rank order 0..R-1, so every rank computes the same bits no matter in which
order the partials arrive.

Only data movement happens here (torch.distributed all_gather); all arithmetic
runs in libbi's kernel.
"""
from __future__ import annotations


def gather_rank_ordered(x, group=None):
    """All ranks' copies of `x`, as a list indexed by rank in `group`.

    Tensors travel as raw bytes (uint8 views), so every backend (gloo, NCCL)
    carries bf16 bit patterns unchanged."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    xs = x.contiguous()
    wire = xs.view(torch.uint8)
    out = [torch.empty_like(wire) for _ in range(world)]
    dist.all_gather(out, wire, group=group)
    return [o.view(xs.dtype) for o in out]


def allreduce_rmsnorm(x_partial, w, eps: float, residual=None, group=None, sum_out=None, out=None):
    """Deterministic all-reduce of the ranks' partial rows, then RMSNorm (with
    optional in-place residual add). CUDA tensors only: the reduction and the
    norm run in libbi."""
    from . import rank_sum_rmsnorm
    parts = gather_rank_ordered(x_partial, group)
    return rank_sum_rmsnorm(parts, w, eps, residual=residual, sum_out=sum_out, out=out)
