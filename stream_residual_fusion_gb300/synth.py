"""Seeded synthetic inputs for the single-pass mHC step.

This module only draws random numbers and lays them out in the shapes the step takes. It holds
none of the step's arithmetic (no sigmoid, no Sinkhorn, no normalisation), so both the CUDA path
and the CPU oracle can be fed from it without sharing any of the method.

Shapes follow the pages' code excerpts (Stream weights for the feed-forward, Code: Block.__init__,
hc_mixes / hc_pre / hc_post; MoE RMSNorm, Code: RMSNorm), flattened to N = B*T tokens:

    X       bf16 [N, n, d]   residual streams
    F       bf16 [N, d]      sublayer output
    pre     fp32 [N, n]      previous reading weights (p_prev)
    post    fp32 [N, n]      previous writing weights (u_prev)
    comb    fp32 [N, n, n]   previous stream combination (C_prev)
    W       fp32 [(2+n)n, n*d]
    scale   fp32 [3]
    base    fp32 [(2+n)n]
    gain    fp32 [d]

The previous tuple is not something the configs draw directly beyond "prev pre U(0,1)". The reading
used here: u_prev ~ U(0,2) (the range of 2*sigmoid) and C_prev a random convex combination of
permutation matrices, which is doubly stochastic by the Birkhoff-von Neumann theorem and in general
not symmetric. No Sinkhorn is needed to make it.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

N_STREAMS = 4
WIDTH = 5120


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: its size and the recipe of its value distributions."""

    name: str
    B: int
    T: int
    n: int = N_STREAMS
    d: int = WIDTH
    x_stream_std: bool = False      # per-stream std ~ U(0.5, 2), one draw per stream index
    scale_uniform: bool = False     # scale ~ U(0.5, 2) instead of ones
    outlier_frac: float = 0.0       # fraction of tokens whose X and F are scaled by 100

    @property
    def N(self) -> int:
        return self.B * self.T


# The five workloads of the benchmark plan: a tiny case, a prefill, a decode batch, the headline
# prefill and a large prefill with outlier tokens.
WORKLOADS = {
    "tiny": Workload("tiny B=1,T=8", 1, 8),
    "prefill4k": Workload("prefill B=1,T=4096", 1, 4096, x_stream_std=True),
    "decode256": Workload("decode B=256,T=1", 256, 1),
    "prefill32k": Workload("prefill B=4,T=8192", 4, 8192, scale_uniform=True),
    "prefill128k": Workload("large prefill B=8,T=16384", 8, 16384, scale_uniform=True,
                            outlier_frac=0.01),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def doubly_stochastic(N: int, n: int, *, seed: int, device="cpu", terms: int = 8) -> torch.Tensor:
    """[N, n, n] fp32: per token a Dirichlet-weighted sum of `terms` random permutation matrices."""
    g = _gen(device, seed)
    keys = torch.rand(N, terms, n, generator=g, device=device)
    perm = keys.argsort(dim=-1)                                   # [N, terms, n]
    onehot = torch.zeros(N, terms, n, n, device=device)
    onehot.scatter_(-1, perm.unsqueeze(-1), 1.0)                  # row r has its 1 at column perm[r]
    w = -torch.log(torch.rand(N, terms, generator=g, device=device).clamp_min(1e-12))
    w = w / w.sum(dim=1, keepdim=True)
    return (w[:, :, None, None] * onehot).sum(dim=1).contiguous()


def make_inputs(N: int, n: int = N_STREAMS, d: int = WIDTH, *, seed: int, device="cpu",
                x_stream_std: bool = False, scale_uniform: bool = False,
                outlier_frac: float = 0.0, w_std: float = 0.02) -> dict:
    """Draw one batch of inputs. Every tensor comes from its own seed (seed*100 + index)."""
    K = n * d
    mix = (2 + n) * n
    dev = torch.device(device)

    def g(i):
        return _gen(dev, seed * 100 + i)

    X = torch.randn(N, n, d, generator=g(0), device=dev)
    if x_stream_std:
        std = torch.empty(n, device=dev).uniform_(0.5, 2.0, generator=g(10))
        X = X * std[None, :, None]
    F = torch.randn(N, d, generator=g(1), device=dev)
    if outlier_frac > 0.0 and N > 0:
        n_out = max(1, int(round(outlier_frac * N)))
        idx = torch.randperm(N, generator=g(11), device=dev)[:n_out]
        X[idx] *= 100.0
        F[idx] *= 100.0
    out = {
        "X": X.to(torch.bfloat16).contiguous(),
        "F": F.to(torch.bfloat16).contiguous(),
        "pre": torch.rand(N, n, generator=g(2), device=dev),
        "post": torch.rand(N, n, generator=g(3), device=dev) * 2.0,
        "comb": doubly_stochastic(N, n, seed=seed * 100 + 4, device=dev),
        "W": torch.randn(mix, K, generator=g(5), device=dev) * w_std,
        "base": torch.randn(mix, generator=g(6), device=dev),
        "scale": (torch.empty(3, device=dev).uniform_(0.5, 2.0, generator=g(7))
                  if scale_uniform else torch.ones(3, device=dev)),
        "gain": torch.ones(d, device=dev),
    }
    if outlier_frac > 0.0 and N > 0:
        out["outliers"] = idx.sort().values
    return out


def make_workload(w: Workload, *, seed: int, device="cpu") -> dict:
    return make_inputs(w.N, w.n, w.d, seed=seed, device=device, x_stream_std=w.x_stream_std,
                       scale_uniform=w.scale_uniform, outlier_frac=w.outlier_frac)


def subset(inputs: dict, tokens) -> dict:
    """The per-token tensors of `inputs` restricted to `tokens` (a 1-D index tensor), parameters
    unchanged. Used to hand a sample of a large batch to the oracle."""
    per_token = ("X", "F", "pre", "post", "comb")
    return {k: (v[tokens] if k in per_token else v) for k, v in inputs.items() if k != "outliers"}


def make_upstream(N: int, n: int = N_STREAMS, d: int = WIDTH, *, seed: int, device="cpu",
                  std: float = 1.0) -> dict:
    """Seeded gradients of the step's outputs for the backward: gXp (of X', bf16 [N,n,d]), gy
    (of y, bf16 [N,d]), gpre, gpost (fp32 [N,n]) and gcomb (fp32 [N,n,n]), all N(0, std^2)."""
    dev = torch.device(device)

    def g(i):
        return _gen(dev, seed * 100 + 50 + i)
    return {
        "gXp": (torch.randn(N, n, d, generator=g(0), device=dev) * std).to(torch.bfloat16),
        "gy": (torch.randn(N, d, generator=g(1), device=dev) * std).to(torch.bfloat16),
        "gpre": torch.randn(N, n, generator=g(2), device=dev) * std,
        "gpost": torch.randn(N, n, generator=g(3), device=dev) * std,
        "gcomb": torch.randn(N, n, n, generator=g(4), device=dev) * std,
    }

