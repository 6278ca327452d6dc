"""Host-side sharding of decode-step work across ranks (one process per GPU).

The (b, kvh) units of a decode step are independent: the slot write, the
attention, LongFlowScore and the eviction never cross a unit. Ranks therefore
take disjoint sequences and run with no collective on the data path. Under
weak scaling every rank keeps the workload's own batch B and takes sequences
[rank * B, (rank + 1) * B) of one recipe of B * world sequences, so the union
of the shards is the unsharded run of that recipe, bit for bit.

The only collectives are for timing: a barrier around the timed region and a
max over ranks of the elapsed time.
"""
from __future__ import annotations

from dataclasses import dataclass

from .workloads import Workload


@dataclass(frozen=True)
class Shard:
    rank: int
    world: int
    workload: Workload       # this rank's per-step work (batch B)
    batch_offset: int        # first sequence of the recipe this rank owns
    full_batch: int          # sequences in the recipe (B * world)


def weak_shard(wl: Workload, rank: int, world: int) -> Shard:
    """Rank `rank` of `world` runs sequences [rank*B, (rank+1)*B) of B*world."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"bad rank {rank} of world {world}")
    return Shard(rank=rank, world=world, workload=wl, batch_offset=rank * wl.B,
                 full_batch=wl.B * world)


def max_over_ranks(value: float, device=None) -> float:
    """Max of a per-rank float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
