"""Plain CPU definition of the single-pass mHC step (oracle; test infrastructure only).

Precision. The pages' code runs every step in float32 torch ops on bf16 streams. The oracle
computes the continuous results (the mix projection and its RMS scale, the split, Sinkhorn, the
RMSNorm) in float64: they are compared against the GPU with tolerances. Two steps end in a bf16
rounding whose result feeds later steps -- hc_post's X' (fed to the projection and to hc_pre) and
hc_pre's y_hat (fed to the RMSNorm). There the oracle evaluates the float32 arithmetic the pages'
code spells out (Stream weights for the feed-forward, Code: hc_pre and hc_post): every product of
a float32 weight and a stream element is its own float32 tensor, so each product is rounded to
float32; the products are then summed over the stream index in float32, in index order
(j = 0, 1, 2, 3, each addition rounded); hc_post adds its rounded sublayer product u_k * F to that
sum; the float32 result is cast to bf16. numpy's float32 multiply and add are single IEEE
operations (no fused multiply-add), so the code below is that evaluation as written.

All arrays are numpy; bf16 values are carried as float64 holding exactly representable values.
"""
from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------------------------------------
# rounding helpers


def fl32(x) -> np.ndarray:
    """Round to the nearest float32 (numpy's cast is IEEE round-to-nearest-even)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32)


_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def bf16_round(x) -> np.ndarray:
    """Round float64 values directly to the nearest bfloat16 (ties to even), as float64.

    bfloat16 keeps 8 significant bits and float32's exponent range; below 2^-126 the spacing is
    fixed at 2^-133 (subnormals). Overflow past the largest finite value rounds to +-inf. The
    rounding is done once from the float64 value, never through float32, so there is no double
    rounding.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, dtype=np.float64, copy=True)
    finite = np.isfinite(x) & (x != 0.0)
    xf = x[finite]
    _, e = np.frexp(xf)                        # |x| in [2^(e-1), 2^e)
    q = np.ldexp(1.0, np.maximum(e - 8, -133))  # spacing of bf16 numbers around x
    r = np.rint(xf / q) * q                    # np.rint rounds halves to even
    r = np.where(np.abs(r) > _BF16_MAX, np.copysign(np.inf, r), r)
    out[finite] = r
    return out


def inputs_to_f64(inputs: dict) -> dict:
    """Widen a dict of torch tensors (any device) exactly to float64 numpy arrays."""
    out = {}
    for k, v in inputs.items():
        if k == "outliers":
            continue
        out[k] = v.detach().to("cpu").double().numpy()
    return out


# ----------------------------------------------------------------------------------------------
# the steps


def hc_post(X, F, post, comb, comb_row_dest: bool = False) -> np.ndarray:
    """Expand the sublayer output back to the streams and mix the residual in through comb.

    Stream weights for the feed-forward, Code: hc_post. The excerpt forms post[k]*x plus the sum
    over comb's first stream index of comb[j,k]*residual[j], i.e.
    X'_k = u_k F + sum_j C_jk X_j, in float32, then casts to the stream dtype. Float32 order
    (module docstring): P_j = fl(C_jk X_j); S = ((P_0 + P_1) + P_2) + P_3; X'_k = fl(u_k F) + S,
    each operation rounded to float32. `comb_row_dest=True` takes the other reading,
    X'_j = u_j F + sum_k C_jk X_k (element (i,j) of comb as "from stream j into stream i",
    section 3 of "2A · Single-Pass mHC").

    X [N,n,d], F [N,d], post [N,n], comb [N,n,n] -> X' [N,n,d] (bf16 values).
    """
    X = fl32(X)
    F = fl32(F)
    post = fl32(post)
    comb = fl32(comb)
    if comb_row_dest:
        comb = np.swapaxes(comb, 1, 2)
    N, n, d = X.shape
    out = np.empty((N, n, d), dtype=np.float64)
    for k in range(n):
        mixed = comb[:, 0, k, None] * X[:, 0, :]               # float32 product, rounded
        for j in range(1, n):                                  # sum over j in index order
            mixed = mixed + comb[:, j, k, None] * X[:, j, :]   # rounded product, rounded sum
        Xk = post[:, k, None] * F + mixed                      # rounded product, rounded sum
        assert Xk.dtype == np.float32
        out[:, k, :] = bf16_round(Xk.astype(np.float64))
    return out


def hc_pre(Xp, pre) -> np.ndarray:
    """Collapse the streams into one sublayer input: y_hat = sum_j pre_j X'_j.

    Stream weights for the feed-forward, Code: hc_pre (float32 products, sum over the stream
    index, cast to the stream dtype). Float32 order (module docstring):
    Q_j = fl(p_j X'_j); y_hat = bf16(((Q_0 + Q_1) + Q_2) + Q_3), each operation rounded.
    X' [N,n,d], pre [N,n] -> y_hat [N,d] (bf16 values).
    """
    Xp = fl32(Xp)
    pre = fl32(pre)
    n = Xp.shape[1]
    acc = pre[:, 0, None] * Xp[:, 0, :]
    for j in range(1, n):
        acc = acc + pre[:, j, None] * Xp[:, j, :]
    assert acc.dtype == np.float32
    return bf16_round(acc.astype(np.float64))


def hc_mixes_scores(Xp, W, norm_eps: float) -> np.ndarray:
    """The 24 mix numbers of each token: m = (x^f W^T) / sqrt(mean((x^f)^2) + eps).

    Stream weights for the feed-forward, "All 5 steps" (x^f = reshape(X'), formula for m) and
    Code: hc_mixes (flatten over streams then width, one statistic per token, eps = norm_eps).
    X' [N,n,d], W [(2+n)n, n*d] -> m [N,(2+n)n].
    """
    N = Xp.shape[0]
    x = np.asarray(Xp, dtype=np.float64).reshape(N, -1)       # index k*d + i
    r = 1.0 / np.sqrt(np.mean(x * x, axis=1) + norm_eps)
    return (x @ np.asarray(W, dtype=np.float64).T) * r[:, None]


def _sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def hc_split(m, scale, base, n: int, hc_eps: float):
    """Split the mix numbers into reading weights, writing weights and comb logits.

    Stream weights for the feed-forward, "All 5 steps" and Code: hc_split_sinkhorn kernel:
      p_j  = sigmoid(s_0 m_j + b_j) + eps
      u_j  = 2 sigmoid(s_1 m_{n+j} + b_{n+j})
      L_jk = s_2 m_{2n + j n + k} + b_{2n + j n + k}
    m [N,(2+n)n] -> p [N,n], u [N,n], L [N,n,n].
    """
    m = np.asarray(m, dtype=np.float64)
    s = np.asarray(scale, dtype=np.float64)
    b = np.asarray(base, dtype=np.float64)
    N = m.shape[0]
    p = _sigmoid(m[:, 0:n] * s[0] + b[0:n]) + hc_eps
    u = 2.0 * _sigmoid(m[:, n:2 * n] * s[1] + b[n:2 * n])
    L = (m[:, 2 * n:] * s[2] + b[2 * n:]).reshape(N, n, n)
    return p, u, L


def sinkhorn(L, iters: int, eps: float) -> np.ndarray:
    """Make comb (nearly) doubly stochastic, in the form of the hc_split_sinkhorn kernel.

    Stream weights for the feed-forward, Code: hc_split_sinkhorn kernel. Steps, on each token's
    n x n logits:
      1. softmax along each row (max subtracted), then + eps;
      2. divide every column by (its sum + eps);
      3. iters - 1 times: divide every row by (row sum + eps), then every column by
         (column sum + eps).
    L [N,n,n] -> C [N,n,n].
    """
    if iters < 1:
        raise ValueError("iters must be >= 1")
    c = np.asarray(L, dtype=np.float64)
    c = np.exp(c - c.max(axis=2, keepdims=True))
    c = c / c.sum(axis=2, keepdims=True) + eps
    c = c / (c.sum(axis=1, keepdims=True) + eps)
    for _ in range(iters - 1):
        c = c / (c.sum(axis=2, keepdims=True) + eps)
        c = c / (c.sum(axis=1, keepdims=True) + eps)
    return c


def sinkhorn_plain(A, rounds: int, history: bool = False):
    """Plain Sinkhorn-Knopp: per round divide each row by its sum, then each column by its sum.

    "2A · Single-Pass mHC", section 3 (row step then column step, 20 rounds) and section 4 (the
    [[3,1],[1,1]] hand check). No softmax and no eps. A [..., n, n] positive.
    With history=True also returns the list of (after-row-step, after-column-step) pairs.
    """
    c = np.asarray(A, dtype=np.float64)
    steps = []
    for _ in range(rounds):
        r = c / c.sum(axis=-1, keepdims=True)
        c = r / r.sum(axis=-2, keepdims=True)
        steps.append((r, c))
    return (c, steps) if history else c


def hc_mixes(Xp, W, scale, base, iters: int, hc_eps: float, norm_eps: float):
    """hc_mixes on the bf16 streams: m, then (p, u, C). Stream weights for the feed-forward,
    Code: hc_mixes. Returns (m, p, u, C)."""
    n = Xp.shape[1]
    m = hc_mixes_scores(Xp, W, norm_eps)
    p, u, L = hc_split(m, scale, base, n, hc_eps)
    C = sinkhorn(L, iters, hc_eps)
    return m, p, u, C


def rmsnorm(x, gain, eps: float) -> np.ndarray:
    """y = gain * x / sqrt(mean(x^2) + eps), cast to bf16.

    MoE RMSNorm, formula block and Code: RMSNorm (statistics over the feature width).
    x [N,d], gain [d] -> y [N,d] (bf16 values).
    """
    x = np.asarray(x, dtype=np.float64)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + eps)
    return bf16_round(np.asarray(gain, dtype=np.float64)[None, :] * (x * r))


def fused_step(X, F, pre_prev, post_prev, comb_prev, W, scale, base, gain, *, iters: int = 20,
               hc_eps: float = 1e-6, norm_eps: float = 1e-6, comb_row_dest: bool = False):
    """One sublayer's worth of the single-pass mHC step.

    MoE RMSNorm, Code: Block.forward (the FFN half): X' = hc_post(X, F, u_prev, C_prev); the new
    (p, u, C) = hc_mixes(X'); y_hat = hc_pre(X', p_prev); y = RMSNorm(y_hat). The previous tuple is
    what the previous sublayer's hc_mixes produced (Stream weights for the feed-forward, "Why").
    Returns dict with Xp, y, pre, post, comb, mixes.
    """
    Xp = hc_post(X, F, post_prev, comb_prev, comb_row_dest)
    m, p, u, C = hc_mixes(Xp, W, scale, base, iters, hc_eps, norm_eps)
    y_hat = hc_pre(Xp, pre_prev)
    y = rmsnorm(y_hat, gain, norm_eps)
    return {"Xp": Xp, "y": y, "pre": p, "post": u, "comb": C, "mixes": m, "y_hat": y_hat}


# ----------------------------------------------------------------------------------------------
# counts the pages state


def parameter_counts(n: int, d: int) -> dict:
    """Learned parameters of one mHC instance, from the shapes in Block.__init__ (Stream weights
    for the feed-forward, Code: Block.__init__): hc_fn [(2+n)n, n d], hc_base [(2+n)n],
    hc_scale [3]; grouped as the page's "Exact per-instance accounting" table groups them."""
    mix_hc = (2 + n) * n
    hc_dim = n * d
    return {
        "mix projection": mix_hc * hc_dim,
        "reading weights": n + 1,          # base entries 0..n-1 and scale[0]
        "writing weights": n + 1,          # base entries n..2n-1 and scale[1]
        "stream combination": n * n + 1,   # base entries 2n.. and scale[2]
        "total": mix_hc * hc_dim + mix_hc + 3,
    }


def unfused_traffic_steps(n: int, d: int):
    """Per-token (reads, writes) in elements of each kernel of the earlier form: hc_post, hc_mixes,
    hc_pre as three kernels, plus the pre-norm as its own pass (Stream weights for the feed-forward,
    "Why")."""
    return [
        ("hc_post", n * d + d, n * d),     # reads X and F, writes X'
        ("hc_mixes", n * d, 0),            # reads X' (the 24 mix numbers are negligible)
        ("hc_pre", n * d, d),              # reads X', writes y_hat
        ("pre-norm", d, d),                # reads y_hat, writes y
    ]


def fused_traffic_steps(n: int, d: int):
    """Per-token (reads, writes) of the single fused pass: reads X and F once, writes X' and y."""
    return [("fused", n * d + d, n * d + d)]


def traffic_per_token(steps) -> int:
    return sum(r + w for _, r, w in steps)
