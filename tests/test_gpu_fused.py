"""Parity of the fused single-pass mHC step (mhc_fused_step / mhc_fused_step_packed) with the
CPU oracle: several tiles with a ragged tail, every width split, both readings of comb, in place,
edge cases, the bounded-wait status path, and the five benchmark workloads, every token of each
compared with the oracle (the two largest in chunks on a process pool)."""
import numpy as np
import pytest
import torch

import oracle as O
from tests.oracle_pool import full_parity
from tests.parity import (TOL_PUC, assert_abs, assert_bf16_within, assert_exact, check_step,
                          oracle_step, to64)

pytestmark = pytest.mark.gpu
DEV = "cuda"


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


def _run(M, inp, **kw):
    return M.fused_step(inp["X"], inp["F"], inp["pre"], inp["post"], inp["comb"], inp["W"],
                        inp["scale"], inp["base"], inp["gain"], with_mixes=True, **kw)


CASES = [
    # N, d, split (0 = automatic)
    (1, 256, 0),
    (128, 256, 1),
    (200, 256, 1),
    (300, 512, 2),
    (300, 1024, 4),
    (260, 2048, 8),
    (300, 5120, 0),
    (130, 640, 1),           # widest slice the TMEM stash ring holds (640 columns)
    (260, 128, 1),           # narrowest slice (4 stages)
    (300, 5120, 16),         # 16 CTAs per tile, 320 columns each
    (200, 8192, 16),
    (160, 4096, 32),         # 32 CTAs per tile, the narrowest slices
    (300, 5120, 32),         # 5 slots per CTA: the last accumulation group holds one slot
    (200, 704, 2),           # 11 slots per CTA
]


@pytest.mark.parametrize("N,d,split", CASES)
def test_fused_parity(M, synth, N, d, split):
    inp = synth.make_inputs(N, 4, d, seed=1000 + N + d, device=DEV, scale_uniform=True,
                            x_stream_std=True)
    out = _run(M, inp, flags=M.split_flag(split))
    assert M.get_status() == M.MHC_OK
    check_step(out, oracle_step(inp))


def test_fused_comb_row_dest(M, synth):
    inp = synth.make_inputs(150, 4, 1024, seed=5, device=DEV)
    comb = torch.rand(150, 4, 4, device=DEV)            # not symmetric: the readings differ
    inp["comb"] = comb
    out = _run(M, inp, flags=M.COMB_ROW_DEST)
    ref = oracle_step(inp, comb_row_dest=True)
    check_step(out, ref)
    other = oracle_step(inp, comb_row_dest=False)
    assert np.any(other["Xp"] != ref["Xp"])


def test_fused_packed_and_in_place(M, synth):
    inp = synth.make_inputs(257, 4, 5120, seed=9, device=DEV, scale_uniform=True)
    ref = oracle_step(inp)
    Wp = M.pack_weights(inp["W"])
    X = inp["X"].clone()
    out = M.fused_step(X, inp["F"], inp["pre"], inp["post"], inp["comb"], None, inp["scale"],
                       inp["base"], inp["gain"], with_mixes=True, W_packed=Wp,
                       out={"Xp": X})
    assert out["Xp"].data_ptr() == X.data_ptr()
    check_step(out, ref)


def test_fused_identity_tuple(M, synth):
    """u_prev = 0 and C_prev = I leave the streams bit-identical; one-hot p_prev makes y the
    RMSNorm of one stream."""
    N, d = 140, 512
    inp = synth.make_inputs(N, 4, d, seed=11, device=DEV)
    inp["post"] = torch.zeros(N, 4, device=DEV)
    inp["comb"] = torch.eye(4, device=DEV).expand(N, 4, 4).contiguous()
    inp["pre"] = torch.tensor([0.0, 0.0, 1.0, 0.0], device=DEV).expand(N, 4).contiguous()
    inp["gain"] = torch.rand(d, device=DEV) + 0.5
    out = _run(M, inp)
    assert torch.equal(out["Xp"], inp["X"])
    assert_bf16_within(to64(out["y"]), O.rmsnorm(to64(inp["X"][:, 2]), to64(inp["gain"]), 1e-6))


def test_fused_zero_tokens(M, synth):
    inp = synth.make_inputs(0, 4, 5120, seed=1, device=DEV)
    out = _run(M, inp)
    assert out["Xp"].numel() == 0 and M.get_status() == M.MHC_OK


def test_fused_tiny_eps_and_outliers(M, synth):
    """norm_eps = 1e-20 (the formula block's value) and tokens scaled by 100."""
    inp = synth.make_inputs(200, 4, 1024, seed=13, device=DEV, outlier_frac=0.05)
    out = _run(M, inp, norm_eps=1e-20, hc_eps=1e-6)
    check_step(out, oracle_step(inp, norm_eps=1e-20))


def test_fused_sinkhorn_iterations(M, synth):
    inp = synth.make_inputs(100, 4, 512, seed=17, device=DEV)
    for iters in (1, 2, 7):
        out = _run(M, inp, iters=iters)
        check_step(out, oracle_step(inp, iters=iters))


def test_bounded_wait_reports_timeout(M, synth):
    """A wait that nothing completes gives up after ~2 ms, the call still finishes with correct
    results, mhc_get_status reports the timeout once, and the next call is clean."""
    inp = synth.make_inputs(130, 4, 512, seed=19, device=DEV)
    out = _run(M, inp, flags=M.DEBUG_NEVER_ARRIVE)
    assert M.get_status() == M.MHC_ERR_TIMEOUT
    check_step(out, oracle_step(inp))
    assert M.get_status() == M.MHC_OK
    out = _run(M, inp)
    assert M.get_status() == M.MHC_OK
    check_step(out, oracle_step(inp))


def test_unfused_chain_matches(M, synth):
    """hc_post, hc_mixes, hc_pre and RMSNorm as four kernels give the fused step's results."""
    inp = synth.make_inputs(300, 4, 5120, seed=23, device=DEV, scale_uniform=True)
    fused = _run(M, inp)
    Xp = M.hc_post(inp["X"], inp["F"], inp["post"], inp["comb"])
    mx = M.mixes(Xp, inp["W"], inp["scale"], inp["base"])
    y = M.rmsnorm(M.hc_pre(Xp, inp["pre"]), inp["gain"], 1e-6)
    assert torch.equal(Xp, fused["Xp"])
    for k in ("pre", "post", "comb"):
        assert_abs(to64(mx[k]), to64(fused[k]), 1e-6, k)
    assert_bf16_within(to64(y), to64(fused["y"]), 1, "y")


# ---------------------------------------------------------------------------------------------
# the benchmark workloads


@pytest.mark.parametrize("name", ["tiny", "prefill4k", "decode256"])
def test_workload_full(M, synth, name):
    w = synth.WORKLOADS[name]
    inp = synth.make_workload(w, seed=1)
    inp = {k: v.to(DEV) for k, v in inp.items()}
    out = _run(M, inp)
    assert M.get_status() == M.MHC_OK
    check_step(out, oracle_step(inp))


@pytest.mark.parametrize("name", ["prefill32k", "prefill128k"])
def test_workload_full_chunked(M, synth, name):
    """The two large workloads at full size, in the bench's launch configuration: every token
    against the oracle (chunks on a spawned process pool, tests/oracle_pool.py), every outlier
    token of the B=8, T=16384 batch included, plus properties that hold for every token."""
    w = synth.WORKLOADS[name]
    inp = synth.make_workload(w, seed=1, device=DEV)
    inp.pop("outliers", None)
    out = _run(M, inp)
    assert M.get_status() == M.MHC_OK
    for k in ("Xp", "y", "pre", "post", "comb", "mixes"):
        assert torch.isfinite(out[k].float()).all(), k
    col = out["comb"].sum(dim=1)
    assert (col <= 1.0 + 1e-5).all() and (out["comb"] > 0).all()
    assert ((out["post"] >= 0) & (out["post"] <= 2)).all()   # 2*sigmoid saturates in fp32
    assert full_parity(inp, out) == w.N


@pytest.mark.parametrize("N,d,tile", [
    (300, 512, 8),           # 8-token tiles: 38 tiles, ragged last one
    (1000, 5120, 40),        # rows 40..127 of every tile idle
    (700, 2048, 96),
    (330, 1024, 120),
    (129, 256, 128),
])
def test_fused_tile_heights(M, synth, N, d, tile):
    """Tiles shorter than the 128 TMEM lanes: rows at and past the tile height compute on stale
    shared memory and are never stored; every token still matches the oracle."""
    inp = synth.make_inputs(N, 4, d, seed=4000 + N + tile, device=DEV, scale_uniform=True,
                            x_stream_std=True)
    flags = M.tile_flag(tile)
    assert M.step_config(N, d, flags)[1] == tile
    out = _run(M, inp, flags=flags)
    assert M.get_status() == M.MHC_OK
    check_step(out, oracle_step(inp))


def test_automatic_shape_choice(M):
    """The persistent kernel's automatic launch shape minimises the busiest group's rounds x slots
    x (height + fixed slot cost) over the splits that fit and the heights that are multiples of
    the split: the fewest CTAs per tile and 128-token tiles for the B=4, T=8192 batch, wider
    groups for decode (where the cluster kernel runs by default: test_gpu_cluster.py)."""
    P = M.PATH_PERSISTENT
    split, _, groups = M.step_config(32768, 5120, P)
    ctas = split * groups

    def cost(N, s, t):
        return -(-(-(-N // t)) // (ctas // s)) * (5120 // (32 * s)) * (t + 96)
    for N in (256, 4096, 32768, 131072, 1000):
        split, tile, groups = M.step_config(N, 5120, P)
        assert tile % 8 == 0 and 8 <= tile <= 128 and tile % split == 0
        options = [cost(N, s, t) for s in (8, 16, 32) for t in range(128, 7, -8) if t % s == 0]
        assert cost(N, split, tile) == min(options), N
    assert M.step_config(32768, 5120) == M.step_config(32768, 5120, P)
    if ctas == 152:
        assert M.step_config(32768, 5120, P)[:2] == (8, 128)
        assert M.step_config(4096, 5120, P)[:2] == (8, 112)
        assert M.step_config(256, 5120, P)[:2] == (32, 64)


def test_fused_step_in_cuda_graph(M, synth):
    """The packed step (counter reset + cooperative launch) captures into a CUDA graph; replays
    with new inputs copied into the captured buffers give the eager results."""
    N, d = 256, 5120
    inp = synth.make_inputs(N, 4, d, seed=8100, device=DEV)
    Wp = M.pack_weights(inp["W"])
    scratch = torch.empty(M.step_scratch_bytes(d), dtype=torch.uint8, device=DEV)
    out = {"Xp": torch.empty_like(inp["X"]), "y": torch.empty(N, d, dtype=torch.bfloat16, device=DEV),
           "pre": torch.empty(N, 4, device=DEV), "post": torch.empty(N, 4, device=DEV),
           "comb": torch.empty(N, 4, 4, device=DEV)}

    def step(stream=None):
        M.fused_step(inp["X"], inp["F"], inp["pre"], inp["post"], inp["comb"], None, inp["scale"],
                     inp["base"], inp["gain"], W_packed=Wp, scratch=scratch, out=out, stream=stream)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        step(side)
    for seed in (8101, 8102):
        fresh = synth.make_inputs(N, 4, d, seed=seed, device=DEV)
        for k in ("X", "F", "pre", "post", "comb"):
            inp[k].copy_(fresh[k])
        graph.replay()
        torch.cuda.synchronize()
        assert M.get_status() == M.MHC_OK
        got = {k: v.clone() for k, v in out.items()}
        # per-token inputs are new; the parameters are the captured ones
        want = M.fused_step(fresh["X"], fresh["F"], fresh["pre"], fresh["post"], fresh["comb"], None,
                            inp["scale"], inp["base"], inp["gain"], W_packed=Wp)
        torch.cuda.synchronize()
        for k in out:
            assert torch.equal(got[k], want[k]), (seed, k)
