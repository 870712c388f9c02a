"""Host logic for running the draft-block head as independent replicas, one
process per GPU (sequences are independent, so the batch shards with no
collective on the data path).

Each rank draws its own shard of the synthetic workload (rank-dependent seeds);
timing takes the maximum elapsed time over the ranks, and the whole-job value
counts every rank's blocks.
"""


def rank_seed(base_seed: int, rank: int) -> int:
    """Seed of rank `rank`'s data shard (rank 0 keeps the base seed)."""
    return base_seed + 1_000_003 * rank


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The maximum of `value` over all ranks (the value itself without a process group)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, world: int, elapsed_s: float) -> float:
    """Units processed by all ranks divided by the (max-over-ranks) elapsed time."""
    return units_per_rank * world / elapsed_s
