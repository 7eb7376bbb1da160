"""Multi-GPU host logic for the mHC step: tokens are independent (one statistic per token,
Stream weights for the feed-forward, Code: hc_mixes), so ranks take contiguous token shards and
exchange nothing on the data path. Only the timing reduction crosses ranks."""
from __future__ import annotations

import torch


def token_shard(N: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous [start, end) of the N tokens for `rank` of `world`; sizes differ by at most 1
    and the shards cover 0..N exactly once."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    base, extra = divmod(N, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` over all ranks of the default process group (the slowest rank's time).
    Without an initialised group it returns `value`."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_throughput(tokens_per_rank: int, world: int, seconds_per_step_max: float) -> float:
    """All ranks' tokens over the slowest rank's step time."""
    return world * tokens_per_rank / seconds_per_step_max
