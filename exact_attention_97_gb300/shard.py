"""Splitting the attention work over ranks (one process per GPU).

Every (batch, head) pair of the forward and of the backward is an independent
problem, so the work shards by heads with no exchange step: rank r of W takes
a contiguous block of the B*H heads and runs the library's kernels on it.
Nothing is reduced across ranks for attention itself. The one collective in a
multi-rank run is the timing's maximum over ranks (``max_over_ranks``).

Host logic only (plain Python and torch.distributed); no arithmetic of the
method lives here.
"""
from __future__ import annotations


def head_range(n_heads: int, rank: int, world: int) -> tuple[int, int]:
    """[lo, hi) of the heads rank `rank` of `world` owns: contiguous blocks
    whose sizes differ by at most one, covering 0..n_heads-1 once."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("need 0 <= rank < world")
    if n_heads < 0:
        raise ValueError("n_heads must be >= 0")
    base, extra = divmod(n_heads, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def local_heads(t, rank: int, world: int):
    """This rank's heads of a [B, H, rows, d] (or [B, H, rows]) tensor, as a
    contiguous [1, h, ...] view of the flattened B*H heads (the library takes
    B = 1, H = h for it)."""
    B, H = t.shape[0], t.shape[1]
    lo, hi = head_range(B * H, rank, world)
    return t.reshape(B * H, *t.shape[2:])[lo:hi].unsqueeze(0)


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of `value` over all ranks of the default process group (the
    value itself without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
