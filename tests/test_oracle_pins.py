"""Pins of the CPU oracle against what the pages and the mathematics fix (no GPU).

Each test fixes part of the oracle by something other than the oracle itself: the pages' worked
example and printed counts (tests/golden/), closed forms, invariants, exact rational brute force on
tiny inputs, and an independent bf16 conversion.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
from tests.parity import near_tie_cases

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line)
    return rows


# ---------------------------------------------------------------------------------------------
# bf16 rounding


def test_bf16_ties_to_even_and_specials():
    one = 1.0
    assert O.bf16_round(one + 2.0 ** -8) == 1.0                   # tie -> even (1.0)
    assert O.bf16_round(one + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6   # tie -> even (…10)
    assert O.bf16_round(one + 2.0 ** -8 + 2.0 ** -30) == 1.0 + 2.0 ** -7
    big = (2.0 - 2.0 ** -7) * 2.0 ** 127
    assert O.bf16_round(big) == big
    assert np.isinf(O.bf16_round(big * (1 + 2.0 ** -8)))        # rounds past max -> inf
    assert O.bf16_round(2.0 ** -133) == 2.0 ** -133               # smallest subnormal
    assert O.bf16_round(2.0 ** -134) == 0.0                       # tie with 0 -> even (0)
    assert O.bf16_round(3 * 2.0 ** -134) == 2.0 ** -132           # tie -> even
    assert O.bf16_round(-0.0) == 0.0 and np.signbit(O.bf16_round(-0.0))


def test_bf16_matches_independent_conversion_from_float32():
    """torch's float32 -> bfloat16 cast (round to nearest even) is an independent implementation;
    on float32 inputs (normal, subnormal, large) both must agree bit for bit."""
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(20000),
        rng.standard_normal(2000) * 1e-39,      # float32 subnormal range
        rng.uniform(-1, 1, 2000) * 3e38,
        (1.0 + (np.arange(4096) + 0.5) * 2.0 ** -8),   # exact halfway cases
    ]).astype(np.float32)
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    got = O.bf16_round(x.astype(np.float64))
    assert np.array_equal(got, ref)


def _round_f32_exact(fr):
    """Nearest float32 to the rational fr, ties to even (by exact comparison)."""
    r = np.float32(float(fr))
    cands = {float(r), float(np.nextafter(r, np.float32(np.inf))), float(np.nextafter(r, np.float32(-np.inf)))}
    best = sorted(cands, key=lambda v: (abs(Fraction(v) - fr),
                                        int(np.float32(v).view(np.uint32)) & 1))
    return np.float32(best[0])


def _round_bf16_exact(fr):
    """Nearest bfloat16 to the rational fr, ties to even, by exact comparison (normal range)."""
    if fr == 0:
        return 0.0
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = math.floor(math.log2(a))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = Fraction(2) ** (e - 7)                     # spacing of bf16 numbers in [2^e, 2^(e+1))
    k = a / q
    lo = math.floor(k)
    rem = k - lo
    k = lo + 1 if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1) else lo
    return sign * float(k * q)


def _f32_sum_in_order(terms):
    """Float32 evaluation of sum(terms) in the given order, every addition rounded once."""
    acc = terms[0]
    for t in terms[1:]:
        acc = Fraction(float(_round_f32_exact(acc + t)))
    return acc


def _hc_post_exact(X, F, u, C, k, i):
    """X'_k at feature i by exact rationals: float32-rounded products, float32 sums over j in
    index order, the rounded sublayer product added last, one bf16 rounding."""
    prods = [Fraction(float(_round_f32_exact(Fraction(C[j, k]) * Fraction(X[j, i]))))
             for j in range(X.shape[0])]
    s = _f32_sum_in_order(prods)
    uf = Fraction(float(_round_f32_exact(Fraction(u[k]) * Fraction(F[i]))))
    return _round_bf16_exact(Fraction(float(_round_f32_exact(uf + s))))


def test_hc_post_hc_pre_float32_brute_force():
    """hc_post and hc_pre against an exact-rational evaluation of the pages' float32 arithmetic
    (Stream weights for the feed-forward, Code: hc_post, hc_pre: each product a float32 tensor,
    summed over the stream index, cast to bf16): float32 weights with full 24-bit mantissas, so
    most products need rounding."""
    rng = np.random.default_rng(31)
    N, n, d = 3, 4, 24
    X, F = _rand_streams(N, n, d, 32)
    u = rng.uniform(0, 2, (N, n)).astype(np.float32).astype(np.float64)
    C = rng.uniform(0, 1, (N, n, n)).astype(np.float32).astype(np.float64)
    p = rng.uniform(0, 1, (N, n)).astype(np.float32).astype(np.float64)
    Xp = O.hc_post(X, F, u, C)
    Xr = O.hc_post(X, F, u, C, comb_row_dest=True)
    yh = O.hc_pre(Xp, p)
    for t in range(N):
        for i in range(d):
            for k in range(n):
                assert Xp[t, k, i] == _hc_post_exact(X[t], F[t], u[t], C[t], k, i)
                assert Xr[t, k, i] == _hc_post_exact(X[t], F[t], u[t], C[t].T, k, i)
            prods = [Fraction(float(_round_f32_exact(Fraction(p[t, j]) * Fraction(Xp[t, j, i]))))
                     for j in range(n)]
            assert yh[t, i] == _round_bf16_exact(_f32_sum_in_order(prods))


def test_hc_products_rounded_before_the_sum():
    """A product that float32 rounds down onto a bf16 tie once added: y_hat = p_0 X'_0 + p_1 X'_1
    with p_0 X'_0 = 2^-24 exact and p_1 X'_1 = A in (1 + 2^-8, 1 + 2^-8 + 2^-24). Rounding A
    first gives 1 + 2^-8, plus 2^-24 is a float32 tie that stays there, a bf16 tie that goes to
    even: 1. A fused multiply-add would keep A's low bits and give 1 + 2^-7."""
    cases = 0
    for p1, x1 in near_tie_cases():
        A = Fraction(float(p1)) * Fraction(x1)
        p1 = np.float32(p1)
        Xp = np.zeros((1, 4, 1))
        Xp[0, 0, 0], Xp[0, 1, 0] = 1.0, x1
        pre = np.array([[2.0 ** -24, float(p1), 0.0, 0.0]])
        assert O.hc_pre(Xp, pre)[0, 0] == 1.0
        assert _round_bf16_exact(Fraction(float(_round_f32_exact(A + Fraction(1, 2 ** 24))))) == 1.0 + 2.0 ** -7
        # the same in hc_post, once through comb (C_0k X_0 + C_1k X_1) and once through the
        # sublayer term (u_k F + C_0k X_0)
        X = np.zeros((1, 4, 1))
        X[0, 0, 0], X[0, 1, 0] = 1.0, x1
        C = np.zeros((1, 4, 4))
        C[0, 0, 2], C[0, 1, 2] = 2.0 ** -24, float(p1)
        assert O.hc_post(X, np.zeros((1, 1)), np.zeros((1, 4)), C)[0, 2, 0] == 1.0
        C[0, 1, 2] = 0.0
        u = np.array([[0.0, 0.0, float(p1), 0.0]])
        assert O.hc_post(X, np.full((1, 1), x1), u, C)[0, 2, 0] == 1.0
        cases += 1
    assert cases > 10


def test_hc_sums_run_in_stream_order():
    """Exact products (X' = 1, weights of few bits) whose float32 sum depends on the order of
    the additions: the oracle follows index order j = 0..3 in hc_pre, and in hc_post adds the
    sublayer term last. The set of cases includes ones where pairwise and reversed orders, and
    adding the sublayer term first, all round differently."""
    vals = [1.0, 2.0 ** -8, 2.0 ** -24, 1.5 * 2.0 ** -24, 2.0 ** -23, -2.0 ** -24, 3.0 * 2.0 ** -9]
    rng = np.random.default_rng(33)
    picks = rng.choice(len(vals), size=(600, 5))
    diff_pw = diff_rev = diff_first = 0

    def bf(terms):
        return _round_bf16_exact(_f32_sum_in_order([Fraction(v) for v in terms]))
    for row in picks:
        q = [vals[i] for i in row]
        Xp = np.ones((1, 4, 1))
        got = O.hc_pre(Xp, np.array([q[:4]]))[0, 0]
        want = bf(q[:4])
        assert got == want
        pw = _round_bf16_exact(Fraction(float(_round_f32_exact(
            Fraction(float(_round_f32_exact(Fraction(q[0]) + Fraction(q[1])))) +
            Fraction(float(_round_f32_exact(Fraction(q[2]) + Fraction(q[3]))))))))
        diff_pw += pw != want
        diff_rev += bf(q[3::-1]) != want
        # hc_post with F = 1, u_k = q[4], C_jk = q[j]: the sublayer term is added last
        X = np.ones((1, 4, 1))
        C = np.zeros((1, 4, 4))
        C[0, :, 0] = q[:4]
        u = np.array([[q[4], 0.0, 0.0, 0.0]])
        post = O.hc_post(X, np.ones((1, 1)), u, C)[0, 0, 0]
        assert post == _round_bf16_exact(Fraction(float(_round_f32_exact(
            Fraction(q[4]) + _f32_sum_in_order([Fraction(v) for v in q[:4]])))))
        diff_first += post != bf([q[4]] + q[:4])
    assert diff_pw > 0 and diff_rev > 0 and diff_first > 0


# ---------------------------------------------------------------------------------------------
# plain Sinkhorn: the page's worked example


def test_sinkhorn_plain_hand_rounds():
    """The two hand-computed rounds on [[3,1],[1,1]] ("2A · Single-Pass mHC", section 4)."""
    rows = _read_golden("sinkhorn_hand_2x2.txt")
    _, hist = O.sinkhorn_plain(np.array([[3.0, 1.0], [1.0, 1.0]]), 2, history=True)
    assert len(rows) == 4
    for line in rows:
        rnd, step, *vals = line.split()
        want = np.array([float(Fraction(v)) for v in vals]).reshape(2, 2)
        got = hist[int(rnd) - 1][0 if step == "row" else 1]
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-15)


def test_sinkhorn_plain_limit_and_tolerance():
    """Diagonal scaling keeps the cross ratio a11 a22 / (a12 a21) = 3, so the doubly stochastic
    limit is [[a, 1-a], [1-a, a]] with a^2 / (1-a)^2 = 3. After 20 rounds the row and column sums
    are within 1e-6 of 1 in float64 without any correction ("2A · Single-Pass mHC", section 4)."""
    C = O.sinkhorn_plain(np.array([[3.0, 1.0], [1.0, 1.0]]), 20)
    a = math.sqrt(3.0) / (1.0 + math.sqrt(3.0))
    np.testing.assert_allclose(C, [[a, 1 - a], [1 - a, a]], atol=1e-12)
    assert np.max(np.abs(C.sum(0) - 1)) < 1e-6
    assert np.max(np.abs(C.sum(1) - 1)) < 1e-6


def test_sinkhorn_plain_fixed_point():
    P = np.array([[0.2, 0.5, 0.3], [0.5, 0.1, 0.4], [0.3, 0.4, 0.3]])
    np.testing.assert_allclose(O.sinkhorn_plain(P, 5), P, atol=1e-15)


# ---------------------------------------------------------------------------------------------
# Sinkhorn in the form of the kernel excerpt (softmax, eps)


def _scalar_recurrence(iters, eps, n=4):
    c = Fraction(1, n) + eps                     # softmax of equal logits, plus eps
    c = c / (n * c + eps)                        # first column step
    for _ in range(iters - 1):
        c = c / (n * c + eps)                    # row step
        c = c / (n * c + eps)                    # column step
    return c


@pytest.mark.parametrize("iters", [1, 2, 3, 20])
@pytest.mark.parametrize("eps", [Fraction(1, 8), Fraction(1e-6)])
def test_sinkhorn_equal_logits_closed_form(iters, eps):
    """All logits equal: by symmetry every entry follows c <- c / (n c + eps) from 1/n + eps."""
    L = np.full((3, 4, 4), 0.7)
    C = O.sinkhorn(L, iters, float(eps))
    want = float(_scalar_recurrence(iters, eps))
    np.testing.assert_allclose(C, want, rtol=1e-14, atol=0)


@pytest.mark.parametrize("eps", [0.0, 0.05])
def test_sinkhorn_one_iteration_softmax_axis(eps):
    """iters = 1 on additive logits L_jk = a_j + b_k: the row softmax gives the same row pi for
    every j, so after + eps and one column step every row equals (pi+eps)/(n(pi+eps)+eps). A
    softmax over the wrong axis would make the rows differ."""
    rng = np.random.default_rng(1)
    a = rng.standard_normal(4) * 3
    b = rng.standard_normal(4)
    L = (a[:, None] + b[None, :])[None]
    pi = np.exp(b) / np.exp(b).sum()
    want = (pi + eps) / (4 * (pi + eps) + eps)
    C = O.sinkhorn(L, 1, eps)[0]
    np.testing.assert_allclose(C, np.tile(want, (4, 1)), rtol=1e-13)


def test_sinkhorn_ends_with_column_step():
    """After the final (column) step every column sums to s/(s+eps) = 1 - eps/(s+eps) <= 1 for its
    pre-step sum s (no column carries less than ~1% of the mass here), rows need not."""
    rng = np.random.default_rng(2)
    L = rng.standard_normal((50, 4, 4)) * 4
    for iters in (1, 2, 20):
        C = O.sinkhorn(L, iters, 1e-6)
        col = C.sum(axis=1)
        assert np.all(col <= 1.0 + 1e-15) and np.all(col > 1.0 - 1e-3)
    C1 = O.sinkhorn(L, 1, 1e-6)
    assert np.max(np.abs(C1.sum(axis=2) - 1)) > 1e-2      # one round leaves rows unbalanced


def test_sinkhorn_exact_small_case():
    """Exact rational brute force, n = 2, two iterations, eps = 1/10, logits = log of integers
    (so the softmax is a ratio of integers)."""
    A = [[3, 1], [1, 2]]
    eps = Fraction(1, 10)
    c = [[Fraction(A[j][k], sum(A[j])) + eps for k in range(2)] for j in range(2)]

    def cols(c):
        s = [c[0][k] + c[1][k] for k in range(2)]
        return [[c[j][k] / (s[k] + eps) for k in range(2)] for j in range(2)]

    def rows(c):
        s = [c[j][0] + c[j][1] for j in range(2)]
        return [[c[j][k] / (s[j] + eps) for k in range(2)] for j in range(2)]

    c = cols(c)
    c = cols(rows(c))
    L = np.log(np.array(A, dtype=np.float64))[None]
    got = O.sinkhorn(L, 2, 0.1)[0]
    np.testing.assert_allclose(got, np.array([[float(v) for v in r] for r in c]), rtol=1e-14)


def test_sinkhorn_permutation_equivariance():
    rng = np.random.default_rng(3)
    L = rng.standard_normal((20, 4, 4)) * 2
    P = np.eye(4)[[2, 0, 3, 1]]
    Q = np.eye(4)[[1, 3, 0, 2]]
    C = O.sinkhorn(L, 20, 1e-6)
    Cp = O.sinkhorn(P @ L @ Q.T, 20, 1e-6)
    np.testing.assert_allclose(Cp, P @ C @ Q.T, atol=1e-14)


def test_sinkhorn_converges_when_well_conditioned():
    rng = np.random.default_rng(4)
    C = O.sinkhorn(rng.standard_normal((100, 4, 4)) * 0.5, 20, 1e-6)
    assert np.all(C > 0)
    assert np.max(np.abs(C.sum(axis=1) - 1)) < 1e-5
    assert np.max(np.abs(C.sum(axis=2) - 1)) < 1e-5


# ---------------------------------------------------------------------------------------------
# the split of the 24 mix numbers


def test_split_at_zero():
    m = np.zeros((2, 24))
    p, u, L = O.hc_split(m, [1.0, 1.0, 1.0], np.zeros(24), 4, 1e-6)
    np.testing.assert_array_equal(p, 0.5 + 1e-6)
    np.testing.assert_array_equal(u, 1.0)
    np.testing.assert_array_equal(L, 0.0)


def test_split_index_layout():
    """Moving one mix number moves exactly one output: index j -> p_j, n+j -> u_j,
    2n + j n + k -> L[j, k], each with its own scale."""
    n, z = 4, 3.0
    s = np.array([0.5, 1.5, 2.5])
    for idx in range(24):
        m = np.zeros((1, 24))
        m[0, idx] = z
        p, u, L = O.hc_split(m, s, np.zeros(24), n, 0.0)
        p0 = np.full(n, 0.5)
        u0 = np.ones(n)
        L0 = np.zeros((n, n))
        if idx < n:
            p0[idx] = 1 / (1 + math.exp(-s[0] * z))
        elif idx < 2 * n:
            u0[idx - n] = 2 / (1 + math.exp(-s[1] * z))
        else:
            j, k = divmod(idx - 2 * n, n)
            L0[j, k] = s[2] * z
        np.testing.assert_allclose(p[0], p0, rtol=1e-15)
        np.testing.assert_allclose(u[0], u0, rtol=1e-15)
        np.testing.assert_allclose(L[0], L0, rtol=1e-15)


def test_split_base_enters_before_sigmoid():
    b = np.linspace(-2, 2, 24)
    p, u, L = O.hc_split(np.zeros((1, 24)), [1, 1, 1], b, 4, 0.0)
    np.testing.assert_allclose(p[0], 1 / (1 + np.exp(-b[:4])), rtol=1e-15)
    np.testing.assert_allclose(u[0], 2 / (1 + np.exp(-b[4:8])), rtol=1e-15)
    np.testing.assert_allclose(L[0], b[8:].reshape(4, 4), rtol=1e-15)


# ---------------------------------------------------------------------------------------------
# the projection and its RMS scale


def test_projection_one_hot_rows_pin_flatten_order():
    """W row r = unit vector at flat index k*d + i picks x[k, i] times the RMS scale."""
    rng = np.random.default_rng(5)
    n, d = 4, 8
    Xp = O.bf16_round(rng.standard_normal((3, n, d)))
    picks = [(k, i) for k in range(n) for i in (0, 5)] + [(3, 7)] * 16
    W = np.zeros((24, n * d))
    for r, (k, i) in enumerate(picks[:24]):
        W[r, k * d + i] = 1.0
    m = O.hc_mixes_scores(Xp, W, 0.0)
    for t in range(3):
        r = 1 / math.sqrt(np.mean(Xp[t] ** 2))
        for row, (k, i) in enumerate(picks[:24]):
            assert m[t, row] == pytest.approx(Xp[t, k, i] * r, rel=1e-14)


@pytest.mark.parametrize("d", [1, 2, 8])
def test_projection_exact_brute_force(d):
    """Exact rational sums at tiny d; only the final 1/sqrt is taken in float."""
    rng = np.random.default_rng(10 + d)
    n = 4
    Xp = O.bf16_round(rng.standard_normal((2, n, d)))
    W = rng.standard_normal((24, n * d)).astype(np.float32).astype(np.float64)
    eps = 1e-6
    m = O.hc_mixes_scores(Xp, W, eps)
    for t in range(2):
        x = [Fraction(v) for v in Xp[t].reshape(-1)]
        ms = sum(v * v for v in x) / len(x) + Fraction(eps)
        r = 1 / math.sqrt(float(ms))
        for row in range(24):
            dot = sum(Fraction(W[row, i]) * x[i] for i in range(n * d))
            assert m[t, row] == pytest.approx(float(dot) * r, rel=1e-14, abs=1e-300)


def test_projection_scale_invariance():
    rng = np.random.default_rng(6)
    Xp = O.bf16_round(rng.standard_normal((4, 4, 64)))
    W = rng.standard_normal((24, 256)) * 0.02
    np.testing.assert_allclose(O.hc_mixes_scores(Xp * 8.0, W, 0.0), O.hc_mixes_scores(Xp, W, 0.0),
                               rtol=1e-13)


# ---------------------------------------------------------------------------------------------
# hc_post


def _rand_streams(N, n, d, seed):
    rng = np.random.default_rng(seed)
    X = O.bf16_round(rng.standard_normal((N, n, d)))
    F = O.bf16_round(rng.standard_normal((N, d)))
    return X, F


def test_hc_post_identity_comb_is_bit_exact():
    X, F = _rand_streams(3, 4, 64, 7)
    Xp = O.hc_post(X, F, np.zeros((3, 4)), np.tile(np.eye(4), (3, 1, 1)))
    np.testing.assert_array_equal(Xp, X)


def test_hc_post_zero_comb_copies_sublayer():
    X, F = _rand_streams(3, 4, 64, 8)
    Xp = O.hc_post(X, F, np.ones((3, 4)), np.zeros((3, 4, 4)))
    for k in range(4):
        np.testing.assert_array_equal(Xp[:, k], F)


@pytest.mark.parametrize("row_dest", [False, True])
def test_hc_post_permutation_direction(row_dest):
    """comb[j, pi(j)] = 1 (non-symmetric pi). The code's reading sums over comb's first index:
    X'_{pi(j)} = X_j. The other reading sums over the second index: X'_j = X_{pi(j)}."""
    pi = [2, 0, 3, 1]
    X, F = _rand_streams(2, 4, 32, 9)
    C = np.zeros((2, 4, 4))
    for j in range(4):
        C[:, j, pi[j]] = 1.0
    Xp = O.hc_post(X, F, np.zeros((2, 4)), C, comb_row_dest=row_dest)
    for j in range(4):
        if row_dest:
            np.testing.assert_array_equal(Xp[:, j], X[:, pi[j]])
        else:
            np.testing.assert_array_equal(Xp[:, pi[j]], X[:, j])


def test_hc_post_against_exact_rationals():
    """The float32 evaluation agrees with the exact value rounded once to bf16, except where the
    float32 error straddles a rounding boundary; there it is one bf16 step away at most."""
    n, d, N = 4, 16, 6
    X, F = _rand_streams(N, n, d, 11)
    rng = np.random.default_rng(12)
    u = rng.uniform(0, 2, (N, n)).astype(np.float32).astype(np.float64)
    C = rng.uniform(0, 1, (N, n, n)).astype(np.float32).astype(np.float64)
    Xp = O.hc_post(X, F, u, C)
    same = 0
    for t in range(N):
        for k in range(n):
            for i in range(d):
                exact = Fraction(u[t, k]) * Fraction(F[t, i]) + sum(
                    Fraction(C[t, j, k]) * Fraction(X[t, j, i]) for j in range(n))
                want = O.bf16_round(float(exact))
                if Xp[t, k, i] == want:
                    same += 1
                else:
                    ulp = 2.0 ** (math.frexp(want)[1] - 8)
                    assert abs(Xp[t, k, i] - want) <= ulp
    assert same >= 0.99 * N * n * d


# ---------------------------------------------------------------------------------------------
# hc_pre and RMSNorm


def test_hc_pre_one_hot_reads_one_stream():
    X, _ = _rand_streams(3, 4, 64, 13)
    for j in range(4):
        p = np.zeros((3, 4))
        p[:, j] = 1.0
        np.testing.assert_array_equal(O.hc_pre(X, p), X[:, j])


def test_hc_pre_weights_exact_small():
    X, _ = _rand_streams(2, 4, 32, 14)
    p = np.array([[0.5, 0.25, 0.125, 2.0], [1.0, 1.0, 1.0, 1.0]])   # sums of bf16 stay exact-ish
    got = O.hc_pre(X, p)
    exact = np.einsum("tj,tji->ti", p, X)
    np.testing.assert_array_equal(got, O.bf16_round(exact))


def test_rmsnorm_constant_row_and_invariances():
    c, eps = 3.0, 1e-6
    x = np.full((1, 128), c)
    y = O.rmsnorm(x, np.ones(128), eps)
    np.testing.assert_array_equal(y, O.bf16_round(c / math.sqrt(c * c + eps)))
    rng = np.random.default_rng(15)
    x = O.bf16_round(rng.standard_normal((5, 256)))
    g = rng.standard_normal(256)
    np.testing.assert_array_equal(O.rmsnorm(2.0 * x, g, 0.0), O.rmsnorm(x, g, 0.0))
    np.testing.assert_array_equal(O.rmsnorm(x, 2.0 * g, 0.0), 2.0 * O.rmsnorm(x, g, 0.0))


def test_rmsnorm_tiny_eps_is_not_flushed():
    """The formula block prints eps = 1e-20; it must still count for an all-zero row."""
    y = O.rmsnorm(np.zeros((1, 8)), np.ones(8), 1e-20)
    np.testing.assert_array_equal(y, 0.0)
    x = np.full((1, 8), 1e-12)
    y = O.rmsnorm(x, np.ones(8), 1e-20)     # mean 1e-24 is 1e4 times eps: result ~ 1/sqrt(1.0001)
    assert y[0, 0] == O.bf16_round(1e-12 / math.sqrt(1e-24 + 1e-20))


# ---------------------------------------------------------------------------------------------
# the whole step: the single-pass shift


def _step_inputs(seed, N=4, n=4, d=64):
    rng = np.random.default_rng(seed)
    X, F = _rand_streams(N, n, d, seed)
    return dict(
        X=X, F=F, pre_prev=rng.uniform(0, 1, (N, n)), post_prev=rng.uniform(0, 2, (N, n)),
        comb_prev=rng.uniform(0, 1, (N, n, n)), W=rng.standard_normal((24, n * d)) * 0.02,
        scale=np.array([1.0, 0.7, 1.3]), base=rng.standard_normal(24), gain=rng.uniform(0.5, 1.5, d))


def test_step_reads_with_previous_weights():
    """hc_pre uses the previous sublayer's reading weights, not the ones this step produces
    (MoE RMSNorm, Code: Block.forward): changing W changes (m, p, u, C) but not y; changing
    pre_prev changes y but not (m, p, u, C)."""
    a = _step_inputs(16)
    r0 = O.fused_step(**a)
    b = dict(a, W=a["W"] * 1.5 + 0.01)
    r1 = O.fused_step(**b)
    np.testing.assert_array_equal(r0["y"], r1["y"])
    np.testing.assert_array_equal(r0["Xp"], r1["Xp"])
    assert np.max(np.abs(r0["pre"] - r1["pre"])) > 1e-3
    c = dict(a, pre_prev=a["pre_prev"][:, ::-1].copy())
    r2 = O.fused_step(**c)
    assert np.max(np.abs(r0["y"] - r2["y"])) > 1e-2
    for k in ("pre", "post", "comb", "mixes"):
        np.testing.assert_array_equal(r0[k], r2[k])


def test_step_identity_tuple_keeps_streams():
    a = _step_inputs(17)
    N = a["X"].shape[0]
    a.update(post_prev=np.zeros((N, 4)), comb_prev=np.tile(np.eye(4), (N, 1, 1)),
             pre_prev=np.tile([0.0, 1.0, 0.0, 0.0], (N, 1)))
    r = O.fused_step(**a)
    np.testing.assert_array_equal(r["Xp"], a["X"])
    np.testing.assert_array_equal(r["y"], O.rmsnorm(a["X"][:, 1], a["gain"], 1e-6))


# ---------------------------------------------------------------------------------------------
# counts printed on the pages


def test_parameter_table():
    want = {}
    for line in _read_golden("parameter_table.txt"):
        name, count = line.split("\t")
        want[name] = int(count)
    assert O.parameter_counts(4, 5120) == want


def test_traffic_formulas():
    rows = {}
    for line in _read_golden("traffic.txt"):
        form, a, b = line.split("\t")
        rows[form] = (int(a), int(b))
    for n, d in [(4, 5120), (2, 128), (8, 4096)]:
        unf = O.traffic_per_token(O.unfused_traffic_steps(n, d))
        fus = O.traffic_per_token(O.fused_traffic_steps(n, d))
        a, b = rows["three-kernel"]
        assert unf == a * n * d + b * d
        a, b = rows["single-pass"]
        assert fus == a * n * d + b * d
        assert unf == 2 * fus
