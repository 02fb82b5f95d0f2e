"""Replica aggregation for multi-GPU runs (one process per GPU).

The decode step has no exchange between GPUs: each rank serves its own slots
on its own GPU.  A multi-GPU run is therefore N independent replicas; the
whole-job throughput is the rows all ranks processed divided by the slowest
rank's time.  Only host-side bookkeeping crosses ranks (a barrier and one
max/sum reduction of two scalars), never the data path.
"""
from __future__ import annotations

from typing import Optional


def world() -> tuple:
    """(rank, world_size, local_rank) from the launcher's environment."""
    import os
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def aggregate(elapsed_ms: float, rows: int, device: Optional[str] = None) -> dict:
    """Whole-job figures from this rank's timed region.

    elapsed_ms: this rank's time for its timed steps; rows: rows it processed.
    Returns max elapsed over ranks, total rows over ranks and rows/s.  Works
    without an initialised process group (a single replica).
    """
    import torch
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        t = torch.tensor([elapsed_ms], dtype=torch.float64, device=device)
        n = torch.tensor([rows], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(n, op=dist.ReduceOp.SUM)
        elapsed_ms, rows = float(t.item()), int(n.item())
        world_size = dist.get_world_size()
    else:
        world_size = 1
    return {"max_ms": elapsed_ms, "rows": rows, "rows_per_s": rows / (elapsed_ms / 1e3), "world": world_size}
