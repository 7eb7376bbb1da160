"""Pins of the backward oracle (oracle/backward.py) against what does not depend on its own
derivation (no GPU).

* Central finite differences of the continuous float64 forward, in a random direction, for
  every input and parameter (Sinkhorn's rounds included, both comb readings, 1, 3 and 20
  rounds).
* Reverse-mode differentiation by torch's autograd of the same forward written out here with
  torch float64 ops: a second, independent derivative of the step.
* Exact identities the mathematics fixes: the softmax's shift invariance (each row of the logit
  gradient sums to zero), the scale invariance of the mix numbers and of the RMSNorm up to eps
  (x . g_x = eps r^2 (g_m . m), y_hat . g_y_hat = eps r_y^3 T), the split's derivative at zero,
  and the rounded form equal to the continuous one where the forward's roundings are exact.
"""
import numpy as np
import pytest
import torch

from oracle import backward as B
from oracle import mhc as O

N_, n_, d_ = 3, 4, 8


def _inputs(seed, N=N_, n=n_, d=d_, w_std=0.3):
    rng = np.random.default_rng(seed)
    mix = (2 + n) * n
    comb = rng.uniform(0.05, 1.0, (N, n, n))
    comb /= comb.sum(axis=1, keepdims=True)
    return {
        "X": rng.standard_normal((N, n, d)),
        "F": rng.standard_normal((N, d)),
        "pre_prev": rng.uniform(0.0, 1.0, (N, n)),
        "post_prev": rng.uniform(0.0, 2.0, (N, n)),
        "comb_prev": comb,
        "W": rng.standard_normal((mix, n * d)) * w_std,
        "scale": rng.uniform(0.5, 2.0, 3),
        "base": rng.standard_normal(mix),
        "gain": rng.uniform(0.5, 1.5, d),
    }


def _upstream(seed, N=N_, n=n_, d=d_):
    rng = np.random.default_rng(seed + 1000)
    return {
        "gXp": rng.standard_normal((N, n, d)),
        "gy": rng.standard_normal((N, d)),
        "gpre": rng.standard_normal((N, n)),
        "gpost": rng.standard_normal((N, n)),
        "gcomb": rng.standard_normal((N, n, n)),
    }


OUT_OF = {"gXp": "Xp", "gy": "y", "gpre": "pre", "gpost": "post", "gcomb": "comb"}
GRAD_OF = {"X": "gX", "F": "gF", "pre_prev": "gpre_prev", "post_prev": "gpost_prev",
           "comb_prev": "gcomb_prev", "W": "gW", "scale": "gscale", "base": "gbase",
           "gain": "ggain"}


def _loss(inp, up, **kw):
    out = B.forward_continuous(**inp, **kw)
    return sum(float((up[g] * out[o]).sum()) for g, o in OUT_OF.items())


@pytest.mark.parametrize("iters,row_dest", [(20, False), (20, True), (1, False), (3, False)])
def test_finite_differences_every_input(iters, row_dest):
    inp, up = _inputs(7 + iters), _upstream(7 + iters)
    kw = dict(iters=iters, hc_eps=1e-6, norm_eps=1e-6, comb_row_dest=row_dest)
    g = B.fused_step_backward(**inp, **up, rounded=False, **kw)
    rng = np.random.default_rng(99)
    for name, gname in GRAD_OF.items():
        v = rng.standard_normal(np.shape(inp[name]))
        h = 1e-5 * max(1.0, float(np.abs(inp[name]).max()))
        plus = dict(inp, **{name: inp[name] + h * v})
        minus = dict(inp, **{name: inp[name] - h * v})
        fd = (_loss(plus, up, **kw) - _loss(minus, up, **kw)) / (2 * h)
        an = float((g[gname] * v).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def _torch_forward(t, iters, hc_eps, norm_eps):
    """The step written with torch float64 ops (no rounding), for autograd."""
    X, F, C = t["X"], t["F"], t["comb_prev"]
    N, n, d = X.shape
    Xp = t["post_prev"][:, :, None] * F[:, None, :] + torch.einsum("njk,njd->nkd", C, X)
    x = Xp.reshape(N, n * d)
    r = torch.rsqrt((x * x).mean(dim=1) + norm_eps)
    m = (x @ t["W"].T) * r[:, None]
    s, b = t["scale"], t["base"]
    p = torch.sigmoid(s[0] * m[:, :n] + b[:n]) + hc_eps
    u = 2 * torch.sigmoid(s[1] * m[:, n:2 * n] + b[n:2 * n])
    c = torch.softmax((s[2] * m[:, 2 * n:] + b[2 * n:]).reshape(N, n, n), dim=2) + hc_eps
    c = c / (c.sum(dim=1, keepdim=True) + hc_eps)
    for _ in range(iters - 1):
        c = c / (c.sum(dim=2, keepdim=True) + hc_eps)
        c = c / (c.sum(dim=1, keepdim=True) + hc_eps)
    yh = torch.einsum("nj,njd->nd", t["pre_prev"], Xp)
    y = t["gain"] * yh * torch.rsqrt((yh * yh).mean(dim=1, keepdim=True) + norm_eps)
    return {"Xp": Xp, "y": y, "pre": p, "post": u, "comb": c}


def test_matches_torch_autograd():
    N, n, d = 5, 4, 64
    inp, up = _inputs(3, N, n, d, w_std=0.05), _upstream(3, N, n, d)
    t = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in inp.items()}
    out = _torch_forward(t, 20, 1e-6, 1e-6)
    loss = sum((torch.tensor(up[g]) * out[o]).sum() for g, o in OUT_OF.items())
    loss.backward()
    g = B.fused_step_backward(**inp, **up, rounded=False, iters=20, hc_eps=1e-6, norm_eps=1e-6)
    for name, gname in GRAD_OF.items():
        ref = t[name].grad.numpy()
        np.testing.assert_allclose(g[gname], ref, rtol=1e-9, atol=1e-11 * max(1.0, np.abs(ref).max()),
                                   err_msg=name)


def test_softmax_shift_invariance_rows_of_logit_gradient_sum_to_zero():
    rng = np.random.default_rng(5)
    L = rng.standard_normal((50, 4, 4)) * 3.0
    gC = rng.standard_normal((50, 4, 4))
    for iters in (1, 2, 20):
        _, tape = B.sinkhorn_taped(L, iters, 1e-6)
        gL = B.sinkhorn_backward(gC, tape)
        assert np.abs(gL.sum(axis=2)).max() < 1e-12 * np.abs(gL).max() * 16


def test_sinkhorn_taped_is_the_oracle_sinkhorn():
    rng = np.random.default_rng(6)
    L = rng.standard_normal((20, 4, 4)) * 2.0
    C, _ = B.sinkhorn_taped(L, 20, 1e-6)
    np.testing.assert_array_equal(C, O.sinkhorn(L, 20, 1e-6))


def test_scale_invariance_of_mix_numbers_up_to_eps():
    """m(a x) = m(x) when eps = 0, so the gradient through m is orthogonal to x up to the eps
    term: x . g_x = eps r^2 (g_m . m) exactly."""
    rng = np.random.default_rng(8)
    N, n, d = 6, 4, 16
    Xp = rng.standard_normal((N, n, d)) * 0.01       # small |x| makes the eps term visible
    W = rng.standard_normal((24, n * d))
    gm = rng.standard_normal((N, 24))
    eps = 1e-6
    gx, _, r = B.mixes_backward(Xp, W, gm, eps)
    x = Xp.reshape(N, -1)
    m = (x @ W.T) * r[:, None]
    lhs = (x * gx.reshape(N, -1)).sum(axis=1)
    rhs = eps * r ** 2 * (gm * m).sum(axis=1)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-7, atol=1e-12 * np.abs(gx).max())
    assert np.abs(rhs).max() > 1e-3 * np.abs(gx).max() * np.abs(x).max()   # the term is there


def test_rmsnorm_scale_invariance_up_to_eps():
    rng = np.random.default_rng(9)
    yh = rng.standard_normal((7, 32)) * 0.003
    gain = rng.uniform(0.5, 1.5, 32)
    gy = rng.standard_normal((7, 32))
    eps = 1e-6
    gyh, _, ry, T = B.rmsnorm_backward(yh, gain, gy, eps)
    np.testing.assert_allclose((yh * gyh).sum(axis=1), eps * ry ** 3 * T, rtol=1e-7,
                               atol=1e-14 * np.abs(gyh).max())


def test_split_derivative_at_zero():
    """sigma'(0) = 1/4: at m = 0, b = 0, g_m = s0 g_p / 4 for p and s1 g_u / 2 for u."""
    n = 4
    gp, gu = np.arange(1.0, 5.0)[None], np.arange(5.0, 9.0)[None]
    s = np.array([0.5, 1.5, 2.0])
    gm, gb, gs = B.split_backward(np.zeros((1, 24)), s, np.zeros(24), gp, gu, np.ones((1, n, n)), n)
    np.testing.assert_array_equal(gm[0, :4], s[0] * gp[0] / 4)
    np.testing.assert_array_equal(gm[0, 4:8], s[1] * gu[0] / 2)
    np.testing.assert_array_equal(gm[0, 8:], np.full(16, s[2]))
    np.testing.assert_array_equal(gs, [0.0, 0.0, 0.0])        # m = 0: no scale gradient
    np.testing.assert_array_equal(gb[:8], np.concatenate([gp[0] / 4, gu[0] / 2]))


def test_rounded_equals_continuous_where_the_forward_is_exact():
    """With C_prev = a permutation, u_prev = 0 and one-hot p_prev, X' is a permutation of the
    bf16 streams and y_hat one of them: every rounding of the forward is exact, so both forms
    of the backward must agree to the last bit of float64 arithmetic order."""
    inp, up = _inputs(11), _upstream(11)
    inp["X"] = O.bf16_round(inp["X"])
    inp["F"] = O.bf16_round(inp["F"])
    perm = np.eye(4)[[2, 0, 3, 1]]
    inp["comb_prev"] = np.repeat(perm[None], N_, axis=0)
    inp["post_prev"] = np.zeros((N_, 4))
    inp["pre_prev"] = np.eye(4)[[1, 3, 0]]
    a = B.fused_step_backward(**inp, **up, rounded=True)
    b = B.fused_step_backward(**inp, **up, rounded=False)
    for k in ("gX", "gF", "gpre_prev", "gpost_prev", "gcomb_prev", "gW", "gbase", "gscale", "ggain"):
        np.testing.assert_allclose(a[k], b[k], rtol=1e-13, atol=1e-13, err_msg=k)
