"""Data-parallel replicas of the layer (one process per GPU).

Every rank holds all experts and runs the layer on its own token shard.  The one
exchange is the per-expert load: counts are summed across ranks before the bias
update, and the update uses the global token count, so every replica applies the
same b_i += gamma * sign(T_global*k/E - count_i) ("DeepSeek-V3 技术报告要点" 4.2:
the bias follows the load observed over the batch).
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def shard_rows(T_global: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous token shard [lo, hi) of rank; shards differ in size by at most one."""
    base, rem = divmod(T_global, world)
    lo = rank * base + min(rank, rem)
    return lo, lo + base + (1 if rank < rem else 0)


def global_counts(counts: torch.Tensor, group=None) -> torch.Tensor:
    """Sums the per-expert counts of every rank in place (the global load)."""
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(counts, op=dist.ReduceOp.SUM, group=group)
    return counts


def global_token_count(T_local: int, group=None, device="cpu") -> int:
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        t = torch.tensor([T_local], dtype=torch.int64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
        return int(t.item())
    return T_local


def bias_update_global(counts: torch.Tensor, bias: torch.Tensor, T_global: int, gamma: float, update_fn,
                       group=None):
    """All-reduces counts, then calls update_fn(counts, bias, T_global, gamma) on every rank.

    update_fn is the library's moe_bias_update (wrapped with a shape whose T is
    T_global) on GPUs; any function with the same meaning elsewhere."""
    global_counts(counts, group)
    update_fn(counts, bias, T_global, gamma)
    return bias
