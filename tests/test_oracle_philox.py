"""Pins for the oracle's Philox4x32-10 and its uniform contract (CPU only)."""
import os

import numpy as np
import pytest
from scipy import stats

from oracle import philox

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def _kat_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        rows.append([int(t, 16) for t in line.split()])
    return rows


@pytest.mark.parametrize("row", _kat_rows())
def test_known_answer_vectors(row):
    c0, c1, c2, c3, k0, k1 = row[:6]
    out = philox.philox4x32_10(c0, c1, c2, c3, k0, k1)
    assert [int(x) for x in out] == row[6:]


def test_vectorised_equals_scalar():
    rng = np.random.default_rng(7)
    ctr = rng.integers(0, 2**32, size=(4, 64), dtype=np.uint64)
    key = rng.integers(0, 2**32, size=(2,), dtype=np.uint64)
    vec = philox.philox4x32_10(*ctr, *key)
    for i in range(64):
        one = philox.philox4x32_10(*[int(c[i]) for c in ctr], int(key[0]), int(key[1]))
        assert [int(v[i]) for v in vec] == [int(o) for o in one]


def test_uniform_range_and_grid():
    u = philox.uniform(0x1234_5678_9ABC, np.arange(20000), 3, 0)
    assert u.min() >= 0.0 and u.max() < 1.0
    # exact multiples of 2^-24 (so fp32 and fp64 hold the same value)
    assert np.all(u * 2**24 == np.floor(u * 2**24))
    assert np.all(u.astype(np.float32).astype(np.float64) == u)


def test_uniform_seed_split_into_key():
    # key = (seed mod 2^32, seed >> 32)
    seed = (0xA4093822 << 32) | 0x299F31D0
    u = philox.uniform(seed, 5, 6, 7)
    out0 = philox.philox4x32_10(5, 6, 7, 0, 0x299F31D0, 0xA4093822)[0]
    assert u == (int(out0) >> 8) * 2.0 ** -24


def test_uniformity_ks():
    n = 200_000
    req = np.arange(n) % 997
    pos = np.arange(n) // 997
    u = philox.uniform(42, req, pos, 1)
    assert stats.kstest(u, "uniform").pvalue > 1e-3


def test_draw_streams_uncorrelated():
    n = 100_000
    r = np.arange(n)
    u0 = philox.uniform(9, r, 1, 0)
    u1 = philox.uniform(9, r, 1, 1)
    u2 = philox.uniform(9, r, 2, 0)
    # correlation of independent uniforms ~ N(0, 1/n)
    for a, b in ((u0, u1), (u0, u2), (u1, u2)):
        assert abs(np.corrcoef(a, b)[0, 1]) < 5.0 / np.sqrt(n)
