"""Comparison rules for the CUDA path against the CPU oracle.

Tolerances (stated once, used by every GPU test):
  * X' and y_hat: bit-exact. The pages' code fixes the float32 arithmetic before the bf16
    rounding (each product rounded, the products summed over the stream index in order), and
    both sides evaluate exactly that, so the rounding decision is identical.
  * y: within 2 bf16 ulps of the oracle (the RMS statistic is summed in a different order).
  * p, u, C: absolute error <= 1e-5.
  * m (the 24 mix numbers): per token, max |dm| <= 1e-4 * max |m|.
  * MXFP8 y: the codes encode the kernel's bf16 y, which is within Y_ULPS bf16 ulps of the
    oracle's. Scales and codes must equal the oracle's encoding of its y wherever no y within
    that distance would decide otherwise (a block maximum that close to a power of two, y / X
    that close to a boundary between E4M3 values); there the kernel's result must be one of the
    two decisions within reach.
"""
from fractions import Fraction

import numpy as np

import oracle as O

TOL_PUC = 1e-5
TOL_M_REL = 1e-4
Y_ULPS = 2


def to64(t):
    return t.detach().double().cpu().numpy()


def bf16_ulp(ref):
    a = np.abs(np.asarray(ref, dtype=np.float64))
    e = np.frexp(a)[1]
    return np.maximum(np.ldexp(1.0, e - 8), 2.0 ** -133)


def assert_bf16_within(got, ref, ulps=Y_ULPS, name="y"):
    got = np.asarray(got, dtype=np.float64)
    diff = np.abs(got - ref)
    lim = ulps * bf16_ulp(ref)
    bad = diff > lim
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{name}: {int(bad.sum())} of {bad.size} beyond {ulps} bf16 ulps; "
                             f"first at {idx.tolist()}: got {got[tuple(idx[0])]}, "
                             f"want {ref[tuple(idx[0])]}")


def assert_exact(got, ref, name):
    got = np.asarray(got, dtype=np.float64)
    neq = got != ref
    if neq.any():
        idx = np.argwhere(neq)[:5]
        raise AssertionError(f"{name}: {int(neq.sum())} of {neq.size} differ; first at "
                             f"{idx.tolist()}: got {got[tuple(idx[0])]}, want {ref[tuple(idx[0])]}")


def assert_abs(got, ref, tol, name):
    err = np.max(np.abs(np.asarray(got, dtype=np.float64) - ref)) if ref.size else 0.0
    assert err <= tol, f"{name}: max abs error {err:.3e} > {tol:.1e}"


def assert_mixes(got, ref, rel=TOL_M_REL):
    got = np.asarray(got, dtype=np.float64)
    scale = np.max(np.abs(ref), axis=1, keepdims=True)
    err = np.max(np.abs(got - ref), axis=1, keepdims=True)
    worst = float(np.max(err / scale)) if ref.size else 0.0
    assert worst <= rel, f"mixes: worst per-token relative error {worst:.3e} > {rel:.1e}"


def oracle_step(inp, **kw):
    a = O.inputs_to_f64(inp)
    return O.fused_step(a["X"], a["F"], a["pre"], a["post"], a["comb"], a["W"], a["scale"],
                        a["base"], a["gain"], **kw)


def check_step(out, ref, with_mixes=True):
    assert_exact(to64(out["Xp"]), ref["Xp"], "X'")
    assert_bf16_within(to64(out["y"]), ref["y"])
    for k in ("pre", "post", "comb"):
        assert_abs(to64(out[k]), ref[k], TOL_PUC, k)
    if with_mixes:
        assert_mixes(to64(out["mixes"]), ref["mixes"])


def check_mxfp8(codes, scale, y_ref, ulps=Y_ULPS):
    """codes uint8 [N, d], scale uint8 [N, d/32] from the kernel against the oracle's MXFP8
    encoding (oracle.mx) of its bf16 y [N, d]."""
    from oracle import mx
    codes = np.asarray(codes)
    scale = np.asarray(scale).astype(np.int64)
    N, d = y_ref.shape
    wid = ulps * bf16_ulp(y_ref)
    a_lo = np.maximum(np.abs(y_ref) - wid, 0.0).reshape(N, d // mx.MX_BLOCK, mx.MX_BLOCK).max(axis=2)
    a_hi = (np.abs(y_ref) + wid).reshape(N, d // mx.MX_BLOCK, mx.MX_BLOCK).max(axis=2)
    s_lo = mx.mx_scale_code(a_lo).astype(np.int64)
    s_hi = mx.mx_scale_code(a_hi).astype(np.int64)
    ok_s = (scale >= s_lo) & (scale <= s_hi)
    if not ok_s.all():
        i = np.argwhere(~ok_s)[0]
        raise AssertionError(f"y_scale: {int((~ok_s).sum())} of {ok_s.size} blocks differ; first "
                             f"at {i.tolist()}: got {scale[tuple(i)]}, want {s_lo[tuple(i)]}")
    X = np.repeat(np.exp2(scale.astype(np.float64) - 127.0), mx.MX_BLOCK, axis=1)
    got = mx.e4m3_decode(codes)
    lo, hi = mx.e4m3_round((y_ref - wid) / X), mx.e4m3_round((y_ref + wid) / X)
    ok = (got >= lo) & (got <= hi)
    if not ok.all():
        i = np.argwhere(~ok)[0]
        raise AssertionError(f"y codes: {int((~ok).sum())} of {ok.size} differ; first at "
                             f"{i.tolist()}: got {got[tuple(i)]}, want {mx.e4m3_round(y_ref[tuple(i)] / X[tuple(i)])}")
    same = (scale == mx.mx_scale_code(np.abs(y_ref).reshape(N, -1, mx.MX_BLOCK).max(axis=2))).mean()
    assert same > 0.99, f"y_scale: only {same:.4f} of the blocks equal the oracle's"


def near_tie_cases():
    """(p, x) pairs, p float32 and x = 1 + m/128 a bf16 value, whose exact product A lies in
    (1 + 2^-8, 1 + 2^-8 + 2^-24). Rounding A to float32 gives 1 + 2^-8; adding 2^-24 then lands on
    a float32 tie that stays at 1 + 2^-8, a bf16 tie that goes to 1. A fused multiply-add
    A + 2^-24 rounds to 1 + 2^-8 + 2^-23 instead, and that to the bf16 value 1 + 2^-7. Each
    pair is checked with exact rationals."""
    lo = Fraction(1) + Fraction(1, 2 ** 8)
    out = []
    for m in range(1, 128):
        x1 = 1.0 + m / 128.0
        c = np.float32(float((lo + Fraction(1, 2 ** 25)) / Fraction(x1)))
        for p1 in (c, np.nextafter(c, np.float32(2)), np.nextafter(c, np.float32(0))):
            if lo < Fraction(float(p1)) * Fraction(x1) < lo + Fraction(1, 2 ** 24):
                out.append((float(p1), x1))
                break
    return out
