"""Batch replicas across ranks (one process per GPU).

Sequences are independent units: no sequence reads another's tokens or K/V,
so N GPUs run N full replicas of the weights, each decoding its own contiguous
slice of the global batch.  No collective touches the data path; the only
cross-rank operations are the timing reduction (max of the elapsed times, sum
of the committed tokens) and the barriers around the timed region.
"""
from __future__ import annotations

import dataclasses


@dataclasses.dataclass(frozen=True)
class Shard:
    rank: int
    world: int
    batch: int          # sequences decoded by this rank
    first_seq: int      # index of this rank's first sequence in the global batch

    @property
    def global_batch(self) -> int:
        return self.batch * self.world


def shard(rank: int, world: int, batch_per_rank: int) -> Shard:
    """Rank ``rank`` of ``world`` decodes sequences [rank*b, rank*b + b) of the
    global batch (weak scaling: the per-rank batch is fixed)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside world {world}")
    if batch_per_rank < 1:
        raise ValueError("batch_per_rank must be >= 1")
    return Shard(rank, world, batch_per_rank, rank * batch_per_rank)


def reduce_timing(elapsed_ms: float, tokens: int, device=None) -> tuple[float, int]:
    """(max elapsed over ranks, total committed tokens over ranks).

    Uses the default process group when one is initialised (any backend;
    ``device`` is where the reduction tensors live: a CUDA device under NCCL,
    None for gloo), else returns the inputs unchanged.
    """
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(elapsed_ms), int(tokens)
    t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
    n = torch.tensor([int(tokens)], dtype=torch.int64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), int(n.item())
