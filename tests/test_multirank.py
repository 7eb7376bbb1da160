"""The multi-GPU host path on CPU: the shard dispatch of the one-process, several-device call and
two gloo ranks that each take their token shard, with no data-path collective; the step on the
shards equals the step on the whole batch (the oracle stands in for the device call). The timing
reduction takes the slowest rank."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from stream_residual_fusion_gb300.dist import (max_over_ranks, strong_scaling_throughput, token_shard,
                                              weak_scaling_throughput)


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


def oracle_launch(inputs, outputs):
    """CPU stand-in for the library call on one shard: the oracle on the shard's inputs, written
    into the shard's output rows (views of the whole batch's outputs)."""
    import oracle as O
    f = O.inputs_to_f64(inputs)
    r = O.fused_step(f["X"], f["F"], f["pre"], f["post"], f["comb"], f["W"], f["scale"],
                     f["base"], f["gain"])
    for k, v in outputs.items():
        v.copy_(torch.from_numpy(r[k]).to(v.dtype))


def _outputs(N, d):
    return {"Xp": torch.empty(N, 4, d, dtype=torch.float64), "y": torch.empty(N, d, dtype=torch.float64),
            "pre": torch.empty(N, 4, dtype=torch.float64), "post": torch.empty(N, 4, dtype=torch.float64),
            "comb": torch.empty(N, 4, 4, dtype=torch.float64)}


def _params(inp):
    return {k: inp[k] for k in ("W", "scale", "base", "gain")}


def test_run_sharded_in_one_process_equals_the_whole_batch():
    """The dispatch of fused_step_sharded (shard plan, per-shard slices of inputs and outputs)
    with the oracle in place of the device call: 13 tokens over 3 and over 5 parts (uneven
    shards), and more parts than tokens."""
    from stream_residual_fusion_gb300 import synth
    from stream_residual_fusion_gb300.dist import run_sharded, slice_tokens
    N, d = 13, 128
    inp = synth.make_inputs(N, 4, d, seed=78)
    whole = _outputs(N, d)
    oracle_launch(inp, whole)
    for parts in (3, 5, 20):
        out = _outputs(N, d)
        for v in out.values():
            v.fill_(float("nan"))
        seen = []

        def launch(part, start, end):
            seen.append((part, start, end))
            oracle_launch(dict(slice_tokens(inp, start, end), **_params(inp)),
                          slice_tokens(out, start, end))
        plan = run_sharded(N, parts, launch)
        assert seen == plan and [p[0] for p in plan] == sorted(p[0] for p in plan)
        assert sum(e - s for _, s, e in plan) == N and len(plan) == min(parts, N)
        for k in ("Xp", "y"):
            assert torch.equal(out[k], whole[k]), (parts, k)
        for k in ("pre", "post", "comb"):     # float64 matmul blocking differs with the batch
            torch.testing.assert_close(out[k], whole[k], rtol=0, atol=1e-12)


def _rank_main(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from stream_residual_fusion_gb300 import synth
        from stream_residual_fusion_gb300.dist import slice_tokens
        N, d = 13, 128
        inp = synth.make_inputs(N, 4, d, seed=77)            # every rank draws the same batch
        a, b = token_shard(N, rank, world)                   # this rank's shard, as bench.py
        out = _outputs(N, d)
        oracle_launch(dict(slice_tokens(inp, a, b), **_params(inp)), slice_tokens(out, a, b))
        # the only cross-rank step: the slowest rank's time
        t = max_over_ranks(1.0 + rank)
        q.put((rank, a, b, {k: v[a:b].numpy() for k, v in out.items()}, t))
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
    for k in ("Xp", "y"):
        np.testing.assert_array_equal(np.concatenate([r[3][k] for r in results]), whole[k])
    for k in ("pre", "post", "comb"):          # float64 matmul blocking differs with the batch
        np.testing.assert_allclose(np.concatenate([r[3][k] for r in results]), whole[k],
                                   rtol=0, atol=1e-12)
    assert all(r[4] == 2.0 for r in results)                  # max over ranks 1.0, 2.0
    assert weak_scaling_throughput(32768, 2, 0.5e-3) == pytest.approx(2 * 32768 / 0.5e-3)
    assert strong_scaling_throughput(32768, 0.5e-3) == pytest.approx(32768 / 0.5e-3)
