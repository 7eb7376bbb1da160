"""Multi-GPU path of the mHC step: tokens are independent (one statistic per token, Stream weights
for the feed-forward, Code: hc_mixes), so a batch splits into contiguous token shards, one per
GPU, with the parameters replicated on every GPU and nothing exchanged on the data path.

Two ways to run it:
  * one process, several devices: `fused_step_sharded` takes one batch of host tensors, cuts it
    with `token_shard` and runs each shard on its own device through the host-tensor step
    (copies in, fused kernel, copies out, on that device), writing every shard's outputs into
    its rows of one set of host output tensors. No peer access, no collective.
  * one process per device (torchrun): each rank takes `token_shard(N, rank, world)` of the
    batch; only the timing reduction (`max_over_ranks`) crosses ranks.

`run_sharded` is the dispatch both share: the shard plan and the per-shard call, with the call
passed in, so that host-side tests can drive the same code with a CPU stand-in for the launch.
"""
from __future__ import annotations

from typing import Callable

import torch

PER_TOKEN_INPUTS = ("X", "F", "pre", "post", "comb")
PER_TOKEN_OUTPUTS = ("Xp", "y", "pre", "post", "comb", "mixes")


def token_shard(N: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous [start, end) of the N tokens for `rank` of `world`; sizes differ by at most 1
    and the shards cover 0..N exactly once."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    base, extra = divmod(N, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def shard_plan(N: int, parts: int) -> list[tuple[int, int, int]]:
    """(part, start, end) of every non-empty shard of N tokens over `parts` parts, in order."""
    return [(i, *token_shard(N, i, parts)) for i in range(parts)
            if token_shard(N, i, parts)[1] > token_shard(N, i, parts)[0]]


def slice_tokens(tensors: dict, start: int, end: int) -> dict:
    """The per-token tensors of `tensors` restricted to rows [start, end) (views, no copy)."""
    return {k: v[start:end] for k, v in tensors.items() if k in PER_TOKEN_INPUTS + PER_TOKEN_OUTPUTS}


def run_sharded(N: int, parts: int, launch: Callable[[int, int, int], None]) -> list:
    """Cut N tokens into `parts` contiguous shards and call launch(part, start, end) for each
    non-empty one, in part order. Returns the plan."""
    plan = shard_plan(N, parts)
    for part, start, end in plan:
        launch(part, start, end)
    return plan


def replicate_params(W, scale, base, gain, devices, chunk_tokens: int, with_mixes: bool = False):
    """Per-device copies of the parameters (W_mix, scale, base, gain) and a staging buffer for
    the host-tensor step on each device: one dict per device, in the order given."""
    from stream_residual_fusion_gb300 import mhc
    d = gain.shape[0]
    reps = []
    for dev in devices:
        dev = torch.device(dev)
        reps.append({
            "device": dev,
            "W": W.to(dev), "scale": scale.to(dev), "base": base.to(dev), "gain": gain.to(dev),
            "staging": torch.empty(mhc.host_staging_bytes(d, chunk_tokens, with_mixes),
                                   dtype=torch.uint8, device=dev),
            "chunk_tokens": chunk_tokens,
        })
    return reps


def fused_step_sharded(X, F, pre_prev, post_prev, comb_prev, replicas, *, iters=20, hc_eps=1e-6,
                       norm_eps=1e-6, flags=0, with_mixes=False, out=None):
    """The fused step on one batch of HOST tensors (X [N,4,d] bf16, F [N,d] bf16, the previous
    tuple fp32; pinned for the copies to overlap), split into contiguous token shards over the
    devices of `replicas` (from replicate_params). Shard i runs on replicas[i]'s device through
    mhc_fused_step_host on that device's current stream and writes its rows of the host
    outputs (allocated here, pinned, unless passed in `out`). Every device is synchronised
    before the call returns."""
    from stream_residual_fusion_gb300 import mhc
    N = X.shape[0]
    o = mhc._step_outputs(X, out, with_mixes)
    inputs = {"X": X, "F": F, "pre": pre_prev, "post": post_prev, "comb": comb_prev}
    used = []

    def launch(part, start, end):
        rep = replicas[part]
        dev = rep["device"]
        ins = slice_tokens(inputs, start, end)
        outs = slice_tokens(o, start, end)
        with torch.cuda.device(dev):
            mhc.fused_step_host(ins["X"], ins["F"], ins["pre"], ins["post"], ins["comb"], rep["W"],
                                rep["scale"], rep["base"], rep["gain"], iters=iters,
                                hc_eps=hc_eps, norm_eps=norm_eps, flags=flags,
                                with_mixes=with_mixes, out=outs, staging=rep["staging"],
                                chunk_tokens=rep["chunk_tokens"],
                                stream=torch.cuda.current_stream(dev))
        used.append(dev)

    run_sharded(N, len(replicas), launch)
    for dev in used:
        torch.cuda.current_stream(dev).synchronize()
    return o


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


def strong_scaling_throughput(total_tokens: int, seconds_per_step_max: float) -> float:
    """One batch of `total_tokens` split over the ranks, over the slowest rank's step time."""
    return total_tokens / seconds_per_step_max
