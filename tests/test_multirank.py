"""The N>1 host path on CPU: two gloo ranks shard the tokens with no data-path collective, and
the step on the shards equals the step on the whole batch (the oracle stands in for the GPU).
The timing reduction takes the slowest rank."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from stream_residual_fusion_gb300.dist import max_over_ranks, token_shard, weak_scaling_throughput


def test_token_shard_covers_exactly_once():
    for N in (0, 1, 7, 256, 1001):
        for world in (1, 2, 3, 8):
            seen = []
            for r in range(world):
                a, b = token_shard(N, r, world)
                assert 0 <= a <= b <= N
                seen.extend(range(a, b))
            assert seen == list(range(N))
            sizes = [token_shard(N, r, world)[1] - token_shard(N, r, world)[0] for r in range(world)]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        token_shard(10, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle as O
        from stream_residual_fusion_gb300 import synth
        N, d = 13, 128
        inp = synth.make_inputs(N, 4, d, seed=77)            # every rank draws the same batch
        a, b = token_shard(N, rank, world)
        sub = synth.subset(inp, torch.arange(a, b))
        f = O.inputs_to_f64(sub)
        out = O.fused_step(f["X"], f["F"], f["pre"], f["post"], f["comb"], f["W"], f["scale"],
                           f["base"], f["gain"])
        # the only cross-rank step: the slowest rank's time
        t = max_over_ranks(1.0 + rank)
        q.put((rank, a, b, {k: out[k] for k in ("Xp", "y", "pre", "post", "comb")}, t))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_the_step():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=240) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    import oracle as O
    from stream_residual_fusion_gb300 import synth
    inp = synth.make_inputs(13, 4, 128, seed=77)
    f = O.inputs_to_f64(inp)
    whole = O.fused_step(f["X"], f["F"], f["pre"], f["post"], f["comb"], f["W"], f["scale"],
                         f["base"], f["gain"])
    results.sort()
    for k in ("Xp", "y", "pre", "post", "comb"):
        np.testing.assert_array_equal(np.concatenate([r[3][k] for r in results]), whole[k])
    assert all(r[4] == 2.0 for r in results)                  # max over ranks 1.0, 2.0
    assert weak_scaling_throughput(32768, 2, 0.5e-3) == pytest.approx(2 * 32768 / 0.5e-3)
