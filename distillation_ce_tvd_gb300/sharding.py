"""Row sharding across ranks (data parallel, no collective on the data path).

Rows of the loss are independent, so a global batch splits into contiguous
row blocks, one per rank, and each rank calls the library on its block.
The only collectives here are for bookkeeping around that: the max of a
timing over ranks and gathering per-row results (for checks).
"""
from __future__ import annotations

import torch


def row_block(BT: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous, balanced [lo, hi) row range of `rank` among `world` ranks."""
    if world < 1 or not 0 <= rank < world or BT < 0:
        raise ValueError("bad shard request")
    base, rem = divmod(BT, world)
    lo = rank * base + min(rank, rem)
    return lo, lo + base + (1 if rank < rem else 0)


def max_over_ranks(x: float, world: int, device="cpu") -> float:
    if world == 1:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def gather_rows(x: torch.Tensor, BT: int, world: int) -> torch.Tensor:
    """All-gather the row blocks of a per-rank tensor into the global (BT, ...) tensor."""
    if world == 1:
        return x
    import torch.distributed as dist
    sizes = [row_block(BT, r, world) for r in range(world)]
    width = max(hi - lo for lo, hi in sizes)
    pad = torch.zeros((width,) + tuple(x.shape[1:]), dtype=x.dtype, device=x.device)
    pad[: x.shape[0]] = x
    parts = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(parts, pad)
    return torch.cat([p[: hi - lo] for p, (lo, hi) in zip(parts, sizes)])
