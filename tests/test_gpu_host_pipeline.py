"""The fused step on host-resident tensors (mhc_fused_step_host): chunks through the staging
slots on three streams give, token for token, the device step's results and the oracle's, for
ragged last chunks, chunk sizes that are not a multiple of the token tile, one chunk larger than
the batch, an in-place host update, and a caller stream other than the default.

A chunk may run with another launch shape (CTAs per tile) than the whole batch, which changes
the order in which the projection's partial sums are added: X' is bit-exact whatever the shape,
y and the mix outputs agree within the parity tolerances."""
import numpy as np
import pytest
import torch

from tests.parity import (TOL_M_REL, TOL_PUC, assert_abs, assert_bf16_within, assert_exact,
                          assert_mixes, check_step, oracle_step, to64)

pytestmark = pytest.mark.gpu
DEV = "cuda"
HOST_KEYS = ("X", "F", "pre", "post", "comb")


@pytest.fixture(scope="module")
def M():
    from stream_residual_fusion_gb300 import build
    build.build()
    import stream_residual_fusion_gb300.mhc as m
    return m


@pytest.fixture(scope="module")
def synth():
    from stream_residual_fusion_gb300 import synth as s
    return s


def _host_inputs(inp):
    return {k: inp[k].cpu().pin_memory() for k in HOST_KEYS}


def _host_step(M, inp, h, stream=None, **kw):
    o = M.fused_step_host(h["X"], h["F"], h["pre"], h["post"], h["comb"], inp["W"], inp["scale"],
                          inp["base"], inp["gain"], stream=stream, **kw)
    (stream or torch.cuda.current_stream()).synchronize()
    return o


def _same_step(got, want):
    """X' bit-exact; y within 2 bf16 ulps; p, u, C and m within the parity tolerances."""
    assert set(got) == set(want)
    for k in want:
        assert got[k].device.type == "cpu"
    assert_exact(to64(got["Xp"]), to64(want["Xp"]), "X'")
    assert_bf16_within(to64(got["y"]), to64(want["y"]))
    for k in ("pre", "post", "comb"):
        assert_abs(to64(got[k]), to64(want[k]), TOL_PUC, k)
    if "mixes" in want:
        assert_mixes(to64(got["mixes"]), to64(want["mixes"]), TOL_M_REL)


def _device_step(M, inp, with_mixes):
    o = M.fused_step(inp["X"], inp["F"], inp["pre"], inp["post"], inp["comb"], inp["W"],
                     inp["scale"], inp["base"], inp["gain"], with_mixes=with_mixes)
    torch.cuda.synchronize()
    return {k: v.cpu() for k, v in o.items()}


@pytest.mark.parametrize("N,d,chunk,with_mixes", [
    (700, 5120, 256, True),      # 3 chunks, last one 188 tokens
    (1000, 512, 300, False),     # chunks that straddle token tiles
    (90, 1024, 4096, True),      # one chunk larger than the batch
    (1, 256, 1, True),           # one token
    (1500, 1024, 256, True),     # ramped: 32, 64, 128, 4 x 256 + 28, 128, 64, 32 tokens
    (704, 512, 256, False),      # the smallest batch that ramps: one full-size chunk
])
def test_host_pipeline_matches_device_step(M, synth, N, d, chunk, with_mixes):
    inp = synth.make_inputs(N, 4, d, seed=7100 + N, device=DEV)
    h = _host_inputs(inp)
    got = _host_step(M, inp, h, chunk_tokens=chunk, with_mixes=with_mixes)
    assert M.get_status() == M.MHC_OK
    want = _device_step(M, inp, with_mixes)
    _same_step(got, want)


def test_host_pipeline_oracle_parity_side_stream(M, synth):
    N, d = 530, 5120
    inp = synth.make_inputs(N, 4, d, seed=7200, device=DEV, scale_uniform=True, x_stream_std=True)
    h = _host_inputs(inp)
    side = torch.cuda.Stream()
    got = _host_step(M, inp, h, stream=side, chunk_tokens=128, with_mixes=True)
    check_step(got, oracle_step({k: v.cpu() for k, v in inp.items()}))


def test_host_pipeline_in_place(M, synth):
    N, d = 600, 2048
    inp = synth.make_inputs(N, 4, d, seed=7300, device=DEV)
    h = _host_inputs(inp)
    want = _device_step(M, inp, False)
    X_host = h["X"]
    got = _host_step(M, inp, h, chunk_tokens=200, out={"Xp": X_host})
    assert got["Xp"].data_ptr() == X_host.data_ptr()
    _same_step(got, want)


def test_host_pipeline_repeated_calls_reuse_staging(M, synth):
    N, d = 400, 1024
    stg = torch.empty(M.host_staging_bytes(d, 128), dtype=torch.uint8, device=DEV)
    for seed in (7400, 7401):
        inp = synth.make_inputs(N, 4, d, seed=seed, device=DEV)
        h = _host_inputs(inp)
        got = _host_step(M, inp, h, chunk_tokens=128, staging=stg)
        want = _device_step(M, inp, False)
        _same_step(got, want)
    with pytest.raises(M.MhcError):
        M.fused_step_host(h["X"], h["F"], h["pre"], h["post"], h["comb"], inp["W"], inp["scale"],
                          inp["base"], inp["gain"], chunk_tokens=256, staging=stg)
    np.testing.assert_equal(M.get_status(), M.MHC_OK)


def test_sharded_step_over_device_replicas(M, synth):
    """dist.fused_step_sharded: one host batch cut into contiguous token shards, each run by the
    host-tensor step on its replica's device and written into its rows of the host outputs. With
    one GPU every replica sits on cuda:0 (three shards, uneven), which runs the same dispatch;
    the result equals the unsharded host-tensor step bit for bit. (The launch shape is pinned:
    a token's sums are grouped by the CTAs of its tile, so an automatic shape that differs with
    the launch's token count may move the mix numbers in their last bits.)"""
    from stream_residual_fusion_gb300 import dist
    N, d = 1001, 5120
    inp = synth.make_inputs(N, 4, d, seed=4242, scale_uniform=True)
    host = {k: inp[k].pin_memory() for k in ("X", "F", "pre", "post", "comb")}
    par = {k: inp[k].to(DEV) for k in ("W", "scale", "base", "gain")}
    reps = dist.replicate_params(par["W"], par["scale"], par["base"], par["gain"],
                                 [DEV] * 3, chunk_tokens=256, with_mixes=True)
    flags = M.split_flag(8) | M.tile_flag(32)
    got = dist.fused_step_sharded(host["X"], host["F"], host["pre"], host["post"], host["comb"],
                                  reps, with_mixes=True, flags=flags)
    want = M.fused_step_host(host["X"], host["F"], host["pre"], host["post"], host["comb"],
                             par["W"], par["scale"], par["base"], par["gain"], with_mixes=True,
                             chunk_tokens=256, flags=flags)
    torch.cuda.synchronize()
    assert M.get_status() == M.MHC_OK
    for k in want:
        assert torch.equal(got[k], want[k]), k
