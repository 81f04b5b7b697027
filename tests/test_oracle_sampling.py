"""Pins for the oracle's inverse-CDF sampler (CPU only)."""
from fractions import Fraction

import numpy as np
from scipy import stats

from oracle.sampling import inverse_cdf, argmax_first


def test_inverse_cdf_exact_on_dyadic_rows():
    # dyadic probabilities: every partial sum is exact in fp64, so the token is the
    # textbook definition F(x-1) <= u < F(x) evaluated with exact rationals.
    rng = np.random.default_rng(0)
    for _ in range(200):
        V = int(rng.integers(1, 12))
        w = rng.integers(0, 9, size=V)
        if w.sum() == 0:
            w[rng.integers(V)] = 1
        tot = int(w.sum())
        scale = 1 << int(np.ceil(np.log2(tot)))
        w = np.append(w, scale - tot)  # pad to a power of two total
        p = w / scale
        u = rng.integers(0, 1 << 24, size=16) / float(1 << 24)
        x, margin = inverse_cdf(np.repeat(p[None], 16, 0), u)
        for ui, xi, mi in zip(u, x, margin):
            F = [Fraction(int(v), scale) for v in np.cumsum(w)]
            uf = Fraction(ui)
            expect = next(i for i, f in enumerate(F) if f > uf)
            assert xi == expect
            lo = F[expect - 1] if expect > 0 else Fraction(0)
            assert mi == float(min(uf - lo, F[expect] - uf))


def test_inverse_cdf_skips_zero_mass():
    p = np.array([[0.0, 0.5, 0.0, 0.5, 0.0]])
    for u, want in ((0.0, 1), (0.49, 1), (0.5, 3), (0.99, 3)):
        x, _ = inverse_cdf(p, np.array([u]))
        assert x[0] == want


def test_inverse_cdf_rounding_fallback_is_last_positive():
    # a row whose fp64 sum is below u for u close to 1: fall back to the last p > 0
    p = np.array([[0.3, 0.3, 0.3, 0.0]])
    x, margin = inverse_cdf(p, np.array([0.95]))
    assert x[0] == 2 and margin[0] == 0.0


def test_inverse_cdf_frequencies():
    rng = np.random.default_rng(1)
    p = rng.dirichlet(np.ones(10))
    u = rng.random(200_000)
    x, _ = inverse_cdf(np.broadcast_to(p, (u.size, 10)), u)
    obs = np.bincount(x, minlength=10)
    assert stats.chisquare(obs, p * u.size).pvalue > 1e-4


def test_argmax_first_ties_and_gap():
    l = np.array([[1.0, 3.0, 3.0, 0.0], [5.0, 1.0, 4.5, 2.0]])
    x, gap = argmax_first(l)
    assert list(x) == [1, 0]
    assert gap[0] == 0.0 and gap[1] == 0.5
