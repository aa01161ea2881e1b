"""Row sharding across ranks for multi-GPU runs.

Rows are independent problems, so a batch is split into contiguous row ranges, one per
rank, with no data-path collective; the only collective is the max-over-ranks of the
timed region.  Host logic only (no CUDA)."""
from __future__ import annotations


def row_range(total_rows: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous [lo, hi) rows of `rank` when `total_rows` rows are split as evenly as
    possible over `world` ranks (the first total_rows % world ranks get one more)."""
    if world < 1 or not 0 <= rank < world or total_rows < 0:
        raise ValueError("bad world/rank/rows")
    base, extra = divmod(total_rows, world)
    lo = rank * base + min(rank, extra)
    hi = lo + base + (1 if rank < extra else 0)
    return lo, hi


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of `value` over the ranks of the default process group (the value itself
    when torch.distributed is not initialised)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
