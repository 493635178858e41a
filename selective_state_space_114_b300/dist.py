"""Multi-GPU host logic for the selective scan.

Every (batch, channel) row of the scan is independent, so data-parallel
replicas need no collective in the forward, the backward's per-row outputs
or the decode step.  The one exchange step is the sum over replicas of the
parameter gradients dA, dD and ddelta_bias (each replica holds its own
batch), done as a single all-reduce of one packed buffer.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

PARAM_GRADS = ("dA", "dD", "ddelta_bias")


def rank_seed(base: int, rank: int) -> int:
    """Seed of a replica's synthetic batch: distinct per rank, fixed per run."""
    return base + 7919 * rank


def allreduce_param_grads(g: dict, group=None) -> dict:
    """Sum dA, dD and ddelta_bias over the ranks of ``group`` in place (one
    all-reduce on a packed buffer); absent (None) gradients are skipped."""
    present = [k for k in PARAM_GRADS if g.get(k) is not None]
    if not present or not dist.is_initialized() or dist.get_world_size(group) == 1:
        return g
    flat = torch.cat([g[k].reshape(-1) for k in present])
    dist.all_reduce(flat, op=dist.ReduceOp.SUM, group=group)
    off = 0
    for k in present:
        n = g[k].numel()
        g[k].copy_(flat[off : off + n].view_as(g[k]))
        off += n
    return g


def max_over_ranks(x: float, device=None) -> float:
    """Largest value of a host float over all ranks (the job's step time)."""
    if not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
