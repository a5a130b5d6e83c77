"""Multi-GPU layout of the attention path: independent heads, no collective on the data path.

Every (batch, head) pair is an independent attention problem ("flash-attention-v2-
sram-tiling" §7: the work splits by rows and heads), so N ranks take disjoint ranges
of the B*H heads and never exchange activations. The only cross-rank traffic is the
benchmark's timing reduction (max over ranks).
"""
from __future__ import annotations


def head_shard(total_heads: int, rank: int, world: int) -> tuple[int, int]:
    """[start, stop) of the heads rank `rank` owns; sizes differ by at most one."""
    if world < 1 or not 0 <= rank < world or total_heads < 0:
        raise ValueError("bad shard request")
    base, extra = divmod(total_heads, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def max_over_ranks(values, device=None):
    """Element-wise max of a list of floats over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()
