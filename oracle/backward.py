"""Gradients of the single-pass mHC step (oracle; test infrastructure only).

The pages define the forward step only (Stream weights for the feed-forward, Code: hc_post,
hc_mixes, hc_pre and the hc_split_sinkhorn kernel; MoE RMSNorm, Code: RMSNorm and
Block.forward). They say nothing of a backward pass. The reading taken here is the plainest one:
the gradient that reverse-mode differentiation of that forward code yields, in float64, with the
step's casts to bf16 passed straight through (a dtype cast's derivative is the identity, as
autograd treats it) and every derivative evaluated at the values the forward actually computed
(the bf16 X' and the bf16 y_hat of oracle.mhc, which is what a differentiated forward saves).
`rounded=False` evaluates the same formulas at the continuous float64 forward instead; that is
the form the finite-difference pins check.

Upstream gradients come in for every output of the step: gXp [N,n,d] (of X'), gy [N,d] (of y),
gpre, gpost [N,n] and gcomb [N,n,n] (of the new p, u, C). The mix numbers m are internal (they
are an optional output of the forward, not a differentiated one). Returned gradients: gX, gF,
gpre_prev, gpost_prev, gcomb_prev per token; gW [(2+n)n, n d], gbase, gscale, ggain summed over
tokens.

Derivatives, per token (K = n d, x = the flattened X'):
  Sinkhorn: each normalisation c' = c / (s + eps), s the row or column sum of c, has
      g_c = g_c' / (s + eps) - sum_line(g_c' * c) / (s + eps)^2;
    the row softmax before it has g_L = sm * (g - sum_row(g * sm)) (the +eps and the max
    subtraction have no derivative).
  split: p = sigma(z_p) + eps, u = 2 sigma(z_u), L = s2 m_L + b_L with z = s m + b:
      g_z = g * sigma'(z) (times 2 for u); g_m = s g_z; g_b = g_z; g_s = sum g_z m.
  projection and its RMS scale: m = (W x) r, r = (|x|^2 / K + eps)^(-1/2):
      g_W += (r g_m) x^T; g_x = W^T (r g_m) - (r^3 / K)(g_m . W x) x.
  RMSNorm: y = gain * y_hat * r_y, r_y = (|y_hat|^2 / d + eps)^(-1/2), T = sum gain gy y_hat:
      g_gain += gy y_hat r_y; g_y_hat = r_y gain gy - (r_y^3 / d) T y_hat.
  hc_pre: y_hat = sum_j p_j X'_j: g_X'_j += p_j g_y_hat; g_p_j = g_y_hat . X'_j.
  hc_post (the code's reading X'_k = u_k F + sum_j C_jk X_j):
      g_X_j = sum_k C_jk g_X'_k; g_F = sum_k u_k g_X'_k; g_u_k = g_X'_k . F;
      g_C_jk = g_X'_k . X_j.
  (The other comb reading transposes C and g_C.)
"""
from __future__ import annotations

import numpy as np

from .mhc import hc_post, hc_pre

__all__ = [
    "forward_continuous", "sinkhorn_taped", "sinkhorn_backward", "split_backward",
    "mixes_backward", "rmsnorm_backward", "fused_step_backward",
]


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def _sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


# ----------------------------------------------------------------------------------------------
# forward pieces in float64 that the backward differentiates


def sinkhorn_taped(L, iters: int, eps: float):
    """The hc_split_sinkhorn normalisation of each token's n x n logits (Stream weights for the
    feed-forward, Code: hc_split_sinkhorn kernel): row softmax + eps, a column step, then
    iters - 1 (row step, column step) rounds, eps in every denominator. Returns C and the tape
    of every step's input and denominator, which sinkhorn_backward walks in reverse."""
    if iters < 1:
        raise ValueError("iters must be >= 1")
    L = _f64(L)
    e = np.exp(L - L.max(axis=2, keepdims=True))
    sm = e / e.sum(axis=2, keepdims=True)
    tape = [("softmax", sm, None)]
    c = sm + eps

    def step(c, axis, kind):
        s = c.sum(axis=axis, keepdims=True) + eps
        tape.append((kind, c, s))
        return c / s

    c = step(c, 1, "col")
    for _ in range(iters - 1):
        c = step(c, 2, "row")
        c = step(c, 1, "col")
    return c, tape


def sinkhorn_backward(gC, tape) -> np.ndarray:
    """Gradient with respect to the logits L of the taped Sinkhorn, given the gradient gC of its
    result (module docstring)."""
    g = _f64(gC)
    for kind, c, s in reversed(tape):
        if kind == "softmax":
            g = c * (g - (g * c).sum(axis=2, keepdims=True))
        else:
            axis = 2 if kind == "row" else 1
            g = g / s - (g * c).sum(axis=axis, keepdims=True) / (s * s)
    return g


def forward_continuous(X, F, pre_prev, post_prev, comb_prev, W, scale, base, gain, *,
                       iters: int = 20, hc_eps: float = 1e-6, norm_eps: float = 1e-6,
                       comb_row_dest: bool = False) -> dict:
    """The step with no rounding anywhere: every quantity in float64. Same formulas as
    oracle.mhc.fused_step (hc_post, hc_mixes, hc_pre, RMSNorm), minus its bf16 and float32
    roundings; the finite-difference pins differentiate this."""
    X, F = _f64(X), _f64(F)
    C = _f64(comb_prev)
    if comb_row_dest:
        C = np.swapaxes(C, 1, 2)
    N, n, d = X.shape
    Xp = _f64(post_prev)[:, :, None] * F[:, None, :] + np.einsum("njk,njd->nkd", C, X)
    x = Xp.reshape(N, n * d)
    r = 1.0 / np.sqrt((x * x).sum(axis=1) / (n * d) + norm_eps)
    m = (x @ _f64(W).T) * r[:, None]
    s, b = _f64(scale), _f64(base)
    p = _sigmoid(s[0] * m[:, :n] + b[:n]) + hc_eps
    u = 2.0 * _sigmoid(s[1] * m[:, n:2 * n] + b[n:2 * n])
    Cn, _ = sinkhorn_taped((s[2] * m[:, 2 * n:] + b[2 * n:]).reshape(N, n, n), iters, hc_eps)
    y_hat = np.einsum("nj,njd->nd", _f64(pre_prev), Xp)
    ry = 1.0 / np.sqrt((y_hat * y_hat).sum(axis=1) / d + norm_eps)
    y = _f64(gain)[None, :] * y_hat * ry[:, None]
    return {"Xp": Xp, "y": y, "pre": p, "post": u, "comb": Cn, "mixes": m, "y_hat": y_hat}


# ----------------------------------------------------------------------------------------------
# backward pieces


def split_backward(m, scale, base, gpre, gpost, gL, n: int):
    """Gradients of the split (module docstring) -> (gm [N,(2+n)n], gbase [(2+n)n], gscale [3])."""
    m, s, b = _f64(m), _f64(scale), _f64(base)
    N = m.shape[0]
    sp = _sigmoid(s[0] * m[:, :n] + b[:n])
    su = _sigmoid(s[1] * m[:, n:2 * n] + b[n:2 * n])
    gzp = _f64(gpre) * sp * (1.0 - sp)
    gzu = 2.0 * _f64(gpost) * su * (1.0 - su)
    gzl = _f64(gL).reshape(N, n * n)
    gz = np.concatenate([gzp, gzu, gzl], axis=1)
    gm = np.concatenate([s[0] * gzp, s[1] * gzu, s[2] * gzl], axis=1)
    gscale = np.array([(gzp * m[:, :n]).sum(), (gzu * m[:, n:2 * n]).sum(),
                       (gzl * m[:, 2 * n:]).sum()])
    return gm, gz.sum(axis=0), gscale


def mixes_backward(Xp, W, gm, norm_eps: float):
    """Gradients of m = (W x) r, r = (|x|^2/K + eps)^(-1/2), at the given X' -> (gx [N,n,d],
    gW [(2+n)n, n d], r [N])."""
    Xp, W, gm = _f64(Xp), _f64(W), _f64(gm)
    N = Xp.shape[0]
    x = Xp.reshape(N, -1)
    K = x.shape[1]
    r = 1.0 / np.sqrt((x * x).sum(axis=1) / K + norm_eps)
    a = x @ W.T
    ga = gm * r[:, None]
    gW = ga.T @ x
    coef = (r ** 3 / K) * (gm * a).sum(axis=1)
    gx = ga @ W - coef[:, None] * x
    return gx.reshape(Xp.shape), gW, r


def rmsnorm_backward(y_hat, gain, gy, norm_eps: float):
    """Gradients of y = gain * y_hat * r_y -> (g_y_hat [N,d], ggain [d], r_y [N], T [N])."""
    y_hat, gain, gy = _f64(y_hat), _f64(gain), _f64(gy)
    d = y_hat.shape[1]
    ry = 1.0 / np.sqrt((y_hat * y_hat).sum(axis=1) / d + norm_eps)
    ggain = (gy * y_hat * ry[:, None]).sum(axis=0)
    T = (gain[None, :] * gy * y_hat).sum(axis=1)
    gyh = ry[:, None] * gain[None, :] * gy - (ry ** 3 * T / d)[:, None] * y_hat
    return gyh, ggain, ry, T


def fused_step_backward(X, F, pre_prev, post_prev, comb_prev, W, scale, base, gain,
                        gXp, gy, gpre, gpost, gcomb, *, iters: int = 20, hc_eps: float = 1e-6,
                        norm_eps: float = 1e-6, comb_row_dest: bool = False,
                        rounded: bool = True) -> dict:
    """Gradients of the fused step's inputs and parameters (module docstring). Also returns the
    per-token intermediates a fused backward kernel produces on the way: gm [N,(2+n)n] (the
    gradient of the mix numbers), r, r_y and T [N], and g_y_hat [N,d]."""
    X, F = _f64(X), _f64(F)
    N, n, d = X.shape
    if rounded:
        Xp = hc_post(X, F, post_prev, comb_prev, comb_row_dest)
        y_hat = hc_pre(Xp, pre_prev)
    else:
        fw = forward_continuous(X, F, pre_prev, post_prev, comb_prev, W, scale, base, gain,
                                iters=iters, hc_eps=hc_eps, norm_eps=norm_eps,
                                comb_row_dest=comb_row_dest)
        Xp, y_hat = fw["Xp"], fw["y_hat"]
    x = Xp.reshape(N, n * d)
    r = 1.0 / np.sqrt((x * x).sum(axis=1) / (n * d) + norm_eps)
    m = (x @ _f64(W).T) * r[:, None]
    s, b = _f64(scale), _f64(base)
    _, tape = sinkhorn_taped((s[2] * m[:, 2 * n:] + b[2 * n:]).reshape(N, n, n), iters, hc_eps)
    gL = sinkhorn_backward(gcomb, tape)
    gm, gbase, gscale = split_backward(m, scale, base, gpre, gpost, gL, n)
    gx, gW, _ = mixes_backward(Xp, W, gm, norm_eps)
    gyh, ggain, ry, T = rmsnorm_backward(y_hat, gain, gy, norm_eps)
    pre_prev = _f64(pre_prev)
    gX_total = _f64(gXp) + gx + pre_prev[:, :, None] * gyh[:, None, :]
    gpre_prev = np.einsum("nd,njd->nj", gyh, Xp)
    C = _f64(comb_prev)
    if comb_row_dest:
        C = np.swapaxes(C, 1, 2)
    gX = np.einsum("njk,nkd->njd", C, gX_total)
    gF = np.einsum("nk,nkd->nd", _f64(post_prev), gX_total)
    gpost_prev = np.einsum("nkd,nd->nk", gX_total, F)
    gcomb_prev = np.einsum("nkd,njd->njk", gX_total, X)
    if comb_row_dest:
        gcomb_prev = np.swapaxes(gcomb_prev, 1, 2)
    return {"gX": gX, "gF": gF, "gpre_prev": gpre_prev, "gpost_prev": gpost_prev,
            "gcomb_prev": gcomb_prev, "gW": gW, "gbase": gbase, "gscale": gscale,
            "ggain": ggain, "gm": gm, "r": r, "ry": ry, "T": T, "gy_hat": gyh,
            "gXp_total": gX_total}
