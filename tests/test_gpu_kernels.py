"""Parity of the standalone kernels (split + Sinkhorn, RMSNorm, hc_post, hc_pre, weight packing,
hc_mixes) against the CPU oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle as O
from tests.parity import (TOL_PUC, assert_abs, assert_bf16_within, assert_exact, assert_mixes,
                          near_tie_cases, oracle_step, to64)

pytestmark = pytest.mark.gpu


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


DEV = "cuda"


@pytest.mark.parametrize("N,std,iters", [(1, 1.0, 20), (1000, 3.0, 20), (257, 8.0, 20),
                                         (64, 2.0, 1), (64, 2.0, 3)])
def test_sinkhorn(M, N, std, iters):
    g = torch.Generator(device=DEV).manual_seed(N)
    mixes = torch.randn(N, 24, generator=g, device=DEV) * std
    scale = torch.tensor([0.7, 1.3, 1.9], device=DEV)
    base = torch.randn(24, generator=g, device=DEV)
    o = M.sinkhorn(mixes, scale, base, iters=iters, hc_eps=1e-6)
    p, u, L = O.hc_split(to64(mixes), to64(scale), to64(base), 4, 1e-6)
    C = O.sinkhorn(L, iters, 1e-6)
    assert_abs(to64(o["pre"]), p, TOL_PUC, "pre")
    assert_abs(to64(o["post"]), u, TOL_PUC, "post")
    assert_abs(to64(o["comb"]), C, TOL_PUC, "comb")


def test_sinkhorn_equal_logits_closed_form(M):
    mixes = torch.zeros(5, 24, device=DEV)
    o = M.sinkhorn(mixes, torch.ones(3, device=DEV), torch.zeros(24, device=DEV), iters=20)
    C = O.sinkhorn(np.zeros((5, 4, 4)), 20, 1e-6)
    assert_abs(to64(o["comb"]), C, 1e-6, "comb")
    assert_abs(to64(o["pre"]), np.full((5, 4), 0.5 + 1e-6), 1e-7, "pre")
    assert_abs(to64(o["post"]), np.ones((5, 4)), 1e-7, "post")


@pytest.mark.parametrize("N,d,eps", [(1, 128, 1e-6), (333, 5120, 1e-6), (64, 1024, 1e-20)])
def test_rmsnorm(M, N, d, eps):
    g = torch.Generator(device=DEV).manual_seed(d)
    x = (torch.randn(N, d, generator=g, device=DEV) * 3).to(torch.bfloat16)
    gain = torch.rand(d, generator=g, device=DEV) + 0.5
    y = M.rmsnorm(x, gain, eps)
    assert_bf16_within(to64(y), O.rmsnorm(to64(x), to64(gain), eps))


def test_rmsnorm_zero_row_tiny_eps(M):
    x = torch.zeros(3, 256, dtype=torch.bfloat16, device=DEV)
    y = M.rmsnorm(x, torch.ones(256, device=DEV), 1e-20)
    assert torch.count_nonzero(y).item() == 0 and torch.isfinite(y.float()).all()


@pytest.mark.parametrize("row_dest", [False, True])
def test_hc_post_and_pre_bit_exact(M, synth, row_dest):
    inp = synth.make_inputs(77, 4, 768, seed=3, device=DEV)
    Xp = M.hc_post(inp["X"], inp["F"], inp["post"], inp["comb"],
                   flags=M.COMB_ROW_DEST if row_dest else 0)
    a = O.inputs_to_f64(inp)
    ref = O.hc_post(a["X"], a["F"], a["post"], a["comb"], comb_row_dest=row_dest)
    assert_exact(to64(Xp), ref, "X'")
    yh = M.hc_pre(Xp, inp["pre"])
    assert_exact(to64(yh), O.hc_pre(ref, a["pre"]), "y_hat")


def _planes(M, P, d):
    """hi, mid, lo planes [24, 4d] decoded from the packed image documented at mhc_pack_weights:
    d/B blocks of [4 streams][80 rows][B columns], plane pl of mix row r in row
    36*(r//12)+12*pl+r%12, rows 72..79 zero, chunk c of row r stored at c ^ ((r*2B/128) % (B/8))."""
    B = M.lib.mhc_packed_block_columns()
    ch = B // 8
    img = P.view(torch.bfloat16).float().cpu().numpy().reshape(d // B, 4, 80, ch, 8)
    rows = np.arange(80)
    phys = np.arange(ch)[None, :] ^ ((rows[:, None] * 2 * B // 128) % ch)    # [80, ch]
    logical = np.take_along_axis(img, phys[None, None, :, :, None], axis=3)  # unswizzled
    assert np.all(logical[:, :, 72:] == 0)
    cols = logical.reshape(d // B, 4, 80, B).transpose(2, 1, 0, 3).reshape(80, 4 * d)
    r = np.arange(24)
    base = 36 * (r // 12) + r % 12
    return cols[base], cols[base + 12], cols[base + 24]


def test_pack_weights_reconstructs(M):
    g = torch.Generator(device=DEV).manual_seed(0)
    W = torch.randn(24, 4 * 512, generator=g, device=DEV) * 0.02
    W[0, :8] = torch.tensor([1e-30, -1e-30, 3.0e38, 0.0, -0.0, 1.0, 2.0 ** -126, 1e-40], device=DEV)
    P = M.pack_weights(W)
    assert P.numel() == M.packed_weights_bytes(512)
    hi, mid, lo = _planes(M, P, 512)
    w = W.double().cpu().numpy()
    assert np.array_equal(hi, O.bf16_round(w))                # the hi plane is bf16(W)
    recon = (lo + mid) + hi
    # three bf16 planes hold every float32 down to bf16's subnormal step 2^-133
    np.testing.assert_allclose(recon, w, rtol=2.0 ** -23, atol=2.0 ** -133)


@pytest.mark.parametrize("N,d,split", [(1, 256, 0), (200, 512, 2), (300, 5120, 0), (129, 1024, 4)])
def test_mixes(M, synth, N, d, split):
    inp = synth.make_inputs(N, 4, d, seed=N + d, device=DEV, scale_uniform=True)
    o = M.mixes(inp["X"], inp["W"], inp["scale"], inp["base"], flags=M.split_flag(split))
    a = O.inputs_to_f64(inp)
    m, p, u, C = O.hc_mixes(a["X"], a["W"], a["scale"], a["base"], 20, 1e-6, 1e-6)
    assert_mixes(to64(o["mixes"]), m)
    assert_abs(to64(o["pre"]), p, TOL_PUC, "pre")
    assert_abs(to64(o["post"]), u, TOL_PUC, "post")
    assert_abs(to64(o["comb"]), C, TOL_PUC, "comb")


def test_products_rounded_before_the_sum_on_gpu(M, synth):
    """Constructed near ties (tests/parity.py near_tie_cases): per token, stream 2 of X' sums
    2^-24 * X_0 (X_0 = 1) and p * X_1 (X_1 = x) through comb, stream 3 adds the sublayer term
    p * F (F = x) to 2^-24 * X_0. Products rounded before the sum give exactly 1 in both; a fused
    multiply-add would give 1 + 2^-7. hc_pre with pre = (2^-24, p, 0, 0) over X'_0 = 1,
    X'_1 = x gives 1 the same way. Checked for the standalone hc_post / hc_pre kernels and for
    X' of the fused step, and against the oracle."""
    cases = near_tie_cases()
    N, d = len(cases), 128
    assert N > 10
    p = torch.tensor([c[0] for c in cases], device=DEV)
    x = torch.tensor([c[1] for c in cases], device=DEV)
    inp = synth.make_inputs(N, 4, d, seed=61, device=DEV)
    X = torch.randn(N, 4, d, device=DEV)
    X[:, 0] = 1.0
    X[:, 1] = x[:, None]
    inp["X"] = X.to(torch.bfloat16)
    inp["F"] = x[:, None].expand(N, d).to(torch.bfloat16).contiguous()
    C = torch.zeros(N, 4, 4, device=DEV)
    C[:, 0, 0] = 1.0                     # X'_0 = X_0 = 1
    C[:, 1, 1] = 1.0                     # X'_1 = X_1 = x
    C[:, 0, 2] = 2.0 ** -24
    C[:, 1, 2] = p                       # X'_2 = 2^-24 * 1 + p * x
    C[:, 0, 3] = 2.0 ** -24              # X'_3 = p * F + 2^-24 * 1
    u = torch.zeros(N, 4, device=DEV)
    u[:, 3] = p
    pre = torch.zeros(N, 4, device=DEV)
    pre[:, 0] = 2.0 ** -24
    pre[:, 1] = p
    inp.update(comb=C, post=u, pre=pre)
    Xp = M.hc_post(inp["X"], inp["F"], u, C)
    assert torch.equal(Xp[:, 0], inp["X"][:, 0]) and torch.equal(Xp[:, 1], inp["X"][:, 1])
    assert bool((Xp[:, 2:] == 1.0).all()), "hc_post: a product was fused into its sum"
    yh = M.hc_pre(Xp, pre)
    assert bool((yh == 1.0).all()), "hc_pre: a product was fused into its sum"
    out = M.fused_step(inp["X"], inp["F"], pre, u, C, inp["W"], inp["scale"], inp["base"],
                       inp["gain"], with_mixes=True)
    assert M.get_status() == M.MHC_OK
    assert torch.equal(out["Xp"], Xp)
    ref = oracle_step(inp)
    assert_exact(to64(Xp), ref["Xp"], "X'")
    assert_exact(to64(yh), ref["y_hat"], "y_hat")
