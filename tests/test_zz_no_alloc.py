"""The allocation-free fused step, mhc_fused_step_noalloc, against the workspace entry point.

mhc_fused_step_noalloc serves callers that cannot allocate device memory when they run the
step (a serving loop with a fixed memory budget, or one whose caching allocator it may not enter;
a plain C host that links the library and has no device allocator of its own): it keeps its
scratch in one fixed array per GPU. This test calls it straight through the C ABI, twice in a
row on different inputs (the array keeps the previous call's contents), and checks each result
against mhc_fused_step with the tolerances every parity test uses; a width whose scratch does not
fit the array is refused before anything runs. The file is named to be collected last.
"""
import ctypes

import pytest
import torch

from tests.parity import TOL_PUC, assert_abs, assert_bf16_within, assert_exact, assert_mixes, to64

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


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _noalloc(M, inp):
    X = inp["X"]
    N, n, d = X.shape
    out = {"Xp": torch.empty_like(X), "y": torch.empty(N, d, dtype=torch.bfloat16, device=DEV),
           "pre": torch.empty(N, n, device=DEV), "post": torch.empty(N, n, device=DEV),
           "comb": torch.empty(N, n, n, device=DEV), "mixes": torch.empty(N, 24, device=DEV)}
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = M.lib.mhc_fused_step_noalloc(
        _p(X), _p(inp["F"]), _p(inp["pre"]), _p(inp["post"]), _p(inp["comb"]), _p(inp["W"]),
        _p(inp["scale"]), _p(inp["base"]), _p(inp["gain"]), _p(out["Xp"]), _p(out["y"]),
        _p(out["pre"]), _p(out["post"]), _p(out["comb"]), _p(out["mixes"]), N, n, d, 20,
        1e-6, 1e-6, 0, stream)
    assert rc == M.MHC_OK, M.lib.mhc_strerror(rc)
    return out


def test_noalloc_matches_workspace_entry_point_twice(M, synth):
    assert M.lib.mhc_noalloc_scratch_bytes() == 8 << 20
    assert M.lib.mhc_workspace_bytes(4, 5120) <= M.lib.mhc_noalloc_scratch_bytes()
    for seed in (41, 42):                          # two calls in a row, different inputs
        inp = synth.make_inputs(300, 4, 5120, seed=seed, device=DEV, scale_uniform=True,
                                x_stream_std=True)
        got = _noalloc(M, inp)
        ref = M.fused_step(inp["X"], inp["F"], inp["pre"], inp["post"], inp["comb"], inp["W"],
                           inp["scale"], inp["base"], inp["gain"], with_mixes=True)
        assert M.get_status() == M.MHC_OK
        assert_exact(to64(got["Xp"]), to64(ref["Xp"]), "X'")
        assert_bf16_within(to64(got["y"]), to64(ref["y"]))
        for k in ("pre", "post", "comb"):
            assert_abs(to64(got[k]), to64(ref[k]), TOL_PUC, k)
        assert_mixes(to64(got["mixes"]), to64(ref["mixes"]))


def test_noalloc_refuses_a_width_beyond_the_fixed_array(M):
    """d = 20480 is a valid width (32 CTAs of 640 columns) whose packed weights alone take
    13 MB: the call returns MHC_ERR_WORKSPACE and writes nothing. The buffers are real and of
    the full size, so the call would be safe even if it ran."""
    N, n, d = 1, 4, 20480
    assert M.lib.mhc_workspace_bytes(n, d) > M.lib.mhc_noalloc_scratch_bytes()
    X = torch.zeros(N, n, d, dtype=torch.bfloat16, device=DEV)
    F = torch.zeros(N, d, dtype=torch.bfloat16, device=DEV)
    small = {k: torch.zeros(N, *s, device=DEV) for k, s in
             (("pre", (n,)), ("post", (n,)), ("comb", (n, n)))}
    W = torch.zeros(24, n * d, device=DEV)
    par = (torch.ones(3, device=DEV), torch.zeros(24, device=DEV), torch.ones(d, device=DEV))
    out = {"Xp": torch.full((N, n, d), 7.0, dtype=torch.bfloat16, device=DEV),
           "y": torch.full((N, d), 7.0, dtype=torch.bfloat16, device=DEV),
           "pre": torch.full((N, n), 7.0, device=DEV), "post": torch.full((N, n), 7.0, device=DEV),
           "comb": torch.full((N, n, n), 7.0, device=DEV), "mixes": torch.full((N, 24), 7.0, device=DEV)}
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = M.lib.mhc_fused_step_noalloc(
        _p(X), _p(F), _p(small["pre"]), _p(small["post"]), _p(small["comb"]), _p(W), _p(par[0]),
        _p(par[1]), _p(par[2]), _p(out["Xp"]), _p(out["y"]), _p(out["pre"]), _p(out["post"]),
        _p(out["comb"]), _p(out["mixes"]), N, n, d, 20, 1e-6, 1e-6, 0, stream)
    assert rc == M.MHC_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert M.get_status() == M.MHC_OK
    for k, v in out.items():
        assert bool((v == 7.0).all()), k
