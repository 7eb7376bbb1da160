"""Parity of the backward of the fused step (mhc_fused_step_backward) with the float64 backward
oracle (oracle/backward.py): full width with a ragged tile, narrower widths, both comb readings,
1, 3 and 20 Sinkhorn rounds, one token and no token.

Tolerances (the pages give none for gradients; these follow from the arithmetic):
  * gX, gF (bf16): within 2 bf16 ulps of the oracle's float64 value plus a per-token floor of
    2^-13 times the token's largest |g_X'| (the projection term W^T (r g_m) is formed from two
    bf16 planes of each factor, error ~2^-16 of the largest product, and the sums over streams
    may cancel).
  * gpre_prev, gpost_prev, gcomb_prev (sums over the width): per token, max error <= 2e-4 times
    the token's largest value of that output.
  * gW, ggain, gbase, gscale (sums over the tokens): max error <= 2e-4 times the largest value.
"""
import numpy as np
import pytest
import torch

from oracle import backward as OB
from oracle import mhc as O
from tests.parity import bf16_ulp, to64

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


def _forward(M, inp, flags):
    return M.fused_step(inp["X"], inp["F"], inp["pre"], inp["post"], inp["comb"], inp["W"],
                        inp["scale"], inp["base"], inp["gain"], with_mixes=True, flags=flags)


def _oracle(inp, up, iters, row_dest):
    a = O.inputs_to_f64(inp)
    u = {k: to64(v) for k, v in up.items()}
    return OB.fused_step_backward(a["X"], a["F"], a["pre"], a["post"], a["comb"], a["W"],
                                  a["scale"], a["base"], a["gain"], u["gXp"], u["gy"],
                                  u["gpre"], u["gpost"], u["gcomb"], iters=iters,
                                  comb_row_dest=row_dest)


def _check(got, ref):
    N = ref["gX"].shape[0]
    floor = 2.0 ** -13 * np.abs(ref["gXp_total"]).reshape(N, -1).max(axis=1)
    for k, shape in (("gX", (N, 1, 1)), ("gF", (N, 1))):
        g = to64(got[k])
        lim = 2 * bf16_ulp(ref[k]) + floor.reshape(shape)
        bad = np.abs(g - ref[k]) > lim
        assert not bad.any(), (k, int(bad.sum()), np.argwhere(bad)[:3].tolist())
    for k in ("gpre_prev", "gpost_prev", "gcomb_prev"):
        g = to64(got[k]).reshape(N, -1)
        r = ref[k].reshape(N, -1)
        scale = np.abs(r).max(axis=1, keepdims=True) + 1e-30
        worst = float((np.abs(g - r) / scale).max())
        assert worst <= 2e-4, (k, worst)
    for k in ("gW", "ggain", "gbase", "gscale"):
        g, r = to64(got[k]), ref[k]
        worst = float(np.abs(g - r).max() / (np.abs(r).max() + 1e-30))
        assert worst <= 2e-4, (k, worst)


CASES = [
    # N, d, iters, row_dest
    (300, 5120, 20, False),
    (300, 5120, 20, True),
    (1000, 512, 20, False),
    (200, 256, 1, False),
    (129, 128, 3, True),
    (1, 5120, 20, False),
]


@pytest.mark.parametrize("N,d,iters,row_dest", CASES)
def test_backward_parity(M, synth, N, d, iters, row_dest):
    inp = synth.make_inputs(N, 4, d, seed=7000 + N + d, device=DEV, scale_uniform=True,
                            x_stream_std=True)
    up = synth.make_upstream(N, 4, d, seed=7100 + N + d, device=DEV)
    flags = M.COMB_ROW_DEST if row_dest else 0
    fw = M.fused_step(inp["X"], inp["F"], inp["pre"], inp["post"], inp["comb"], inp["W"],
                      inp["scale"], inp["base"], inp["gain"], with_mixes=True, flags=flags,
                      iters=iters)
    got = M.fused_step_backward(inp["X"], inp["F"], fw["Xp"], fw["mixes"], inp["pre"],
                                inp["post"], inp["comb"], inp["W"], inp["scale"], inp["base"],
                                inp["gain"], up["gXp"], up["gy"], up["gpre"], up["gpost"],
                                up["gcomb"], iters=iters, flags=flags)
    torch.cuda.synchronize()
    assert M.get_status() == M.MHC_OK
    _check(got, _oracle(inp, up, iters, row_dest))


def test_backward_no_tokens_zeroes_parameter_gradients(M, synth):
    inp = synth.make_inputs(4, 4, 256, seed=7300, device=DEV)
    up = synth.make_upstream(4, 4, 256, seed=7301, device=DEV)
    e = {k: v[:0] for k, v in inp.items() if k in ("X", "F", "pre", "post", "comb")}
    u = {k: v[:0] for k, v in up.items()}
    out = {"gW": torch.full_like(inp["W"], 7.0), "gbase": torch.full_like(inp["base"], 7.0),
           "gscale": torch.full((3,), 7.0, device=DEV), "ggain": torch.full_like(inp["gain"], 7.0)}
    mixes = torch.empty(0, 24, device=DEV)
    got = M.fused_step_backward(e["X"], e["F"], e["X"], mixes, e["pre"], e["post"], e["comb"],
                                inp["W"], inp["scale"], inp["base"], inp["gain"], u["gXp"], u["gy"],
                                u["gpre"], u["gpost"], u["gcomb"], out=out)
    torch.cuda.synchronize()
    for k in ("gW", "gbase", "gscale", "ggain"):
        assert torch.count_nonzero(got[k]).item() == 0, k


def test_backward_bench_workload_sampled(M, synth):
    """The B=4,T=8192 workload as the bench runs it: the parameter gradients (sums over all
    32,768 tokens) against the oracle's, and the per-token outputs of a spread sample of tokens
    (first and last tiles included)."""
    w = synth.WORKLOADS["prefill32k"]
    inp = synth.make_workload(w, seed=3000, device=DEV)
    up = synth.make_upstream(w.N, seed=3001, device=DEV)
    fw = M.fused_step(inp["X"], inp["F"], inp["pre"], inp["post"], inp["comb"], inp["W"],
                      inp["scale"], inp["base"], inp["gain"], with_mixes=True)
    got = M.fused_step_backward(inp["X"], inp["F"], fw["Xp"], fw["mixes"], inp["pre"],
                                inp["post"], inp["comb"], inp["W"], inp["scale"], inp["base"],
                                inp["gain"], up["gXp"], up["gy"], up["gpre"], up["gpost"],
                                up["gcomb"])
    torch.cuda.synchronize()
    assert M.get_status() == M.MHC_OK
    idx = torch.cat([torch.arange(0, 130), torch.arange(w.N - 130, w.N),
                     torch.randperm(w.N, generator=torch.Generator().manual_seed(5))[:240]]).unique()
    sub = {k: v[idx.to(v.device)] for k, v in inp.items() if k in ("X", "F", "pre", "post", "comb")}
    sub.update({k: inp[k] for k in ("W", "scale", "base", "gain")})
    usub = {k: v[idx.to(v.device)] for k, v in up.items()}
    ref = _oracle(sub, usub, 20, False)
    got_sub = {k: got[k][idx.to(got[k].device)] for k in ("gX", "gF", "gpre_prev", "gpost_prev", "gcomb_prev")}
    got_sub.update({k: torch.zeros(1) for k in ("gW", "ggain", "gbase", "gscale")})
    ref_sub = dict(ref)
    ref_sub.update({k: np.zeros(1) for k in ("gW", "ggain", "gbase", "gscale")})
    _check(got_sub, ref_sub)
    # parameter gradients over every token: the oracle's sums, in chunks
    acc = {k: 0.0 for k in ("gW", "ggain", "gbase", "gscale")}
    for c0 in range(0, w.N, 2048):
        sl = slice(c0, c0 + 2048)
        cin = {k: inp[k][sl] for k in ("X", "F", "pre", "post", "comb")}
        cin.update({k: inp[k] for k in ("W", "scale", "base", "gain")})
        cup = {k: v[sl] for k, v in up.items()}
        r = _oracle(cin, cup, 20, False)
        for k in acc:
            acc[k] = acc[k] + r[k]
    for k, r in acc.items():
        g = to64(got[k])
        worst = float(np.abs(g - r).max() / (np.abs(r).max() + 1e-30))
        assert worst <= 2e-4, (k, worst)


@pytest.mark.parametrize("N,d", [(1, 256), (129, 512), (300, 5120)])
def test_backward_outputs_stay_in_bounds(M, synth, N, d):
    """Every output of the backward sits at the start of a larger buffer filled with a sentinel:
    after the call nothing past the output's end has changed, ragged token counts included, and
    the inputs are unchanged."""
    inp = synth.make_inputs(N, 4, d, seed=7400 + N, device=DEV, scale_uniform=True)
    up = synth.make_upstream(N, 4, d, seed=7401 + N, device=DEV)
    fw = M.fused_step(inp["X"], inp["F"], inp["pre"], inp["post"], inp["comb"], inp["W"],
                      inp["scale"], inp["base"], inp["gain"], with_mixes=True)
    pad = 4096
    shapes = {"gX": ((N, 4, d), torch.bfloat16), "gF": ((N, d), torch.bfloat16),
              "gpre_prev": ((N, 4), torch.float32), "gpost_prev": ((N, 4), torch.float32),
              "gcomb_prev": ((N, 4, 4), torch.float32), "gW": (tuple(inp["W"].shape), torch.float32),
              "gbase": ((24,), torch.float32), "gscale": ((3,), torch.float32),
              "ggain": ((d,), torch.float32)}
    big, out = {}, {}
    for k, (shape, dt) in shapes.items():
        n = 1
        for v in shape:
            n *= v
        big[k] = torch.full((n + pad,), -7.0, dtype=dt, device=DEV)
        out[k] = big[k][:n].view(shape)
    before = {k: v.clone() for k, v in list(inp.items()) + list(up.items()) if torch.is_tensor(v)}
    M.fused_step_backward(inp["X"], inp["F"], fw["Xp"], fw["mixes"], inp["pre"], inp["post"],
                          inp["comb"], inp["W"], inp["scale"], inp["base"], inp["gain"],
                          up["gXp"], up["gy"], up["gpre"], up["gpost"], up["gcomb"], out=out)
    torch.cuda.synchronize()
    assert M.get_status() == M.MHC_OK
    for k, b in big.items():
        n = b.numel() - pad
        assert bool((b[n:] == -7.0).all()), k
        assert bool(torch.isfinite(b[:n].float()).all()), k
    for k, v in before.items():
        src = inp.get(k, up.get(k))
        assert torch.equal(src, v), k
    _check(out, _oracle(inp, up, 20, False))
