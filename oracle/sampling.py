"""Inverse-CDF sampling in fp64 with decision margins — test infrastructure only.

Reading (the pages say "sample" and give no procedure): a token is drawn from a
probability row p by inverse CDF in token-id order.  With F(v) = sum_{i<=v} p(i)
and a uniform u in [0, 1):

    x = smallest v with F(v) > u;   if rounding leaves none, x = last v with p(v) > 0.

The margin of the draw is min(u - F(x-1), F(x) - u) (F(-1) = 0).  An
implementation whose CDF differs from this one by less than the margin picks
the same token.
"""
import numpy as np


def inverse_cdf(p: np.ndarray, u: np.ndarray):
    """p [R, V] fp64 rows summing to 1 (each row normalised); u [R] fp64.

    Returns (x [R] int64, margin [R] fp64)."""
    p = np.asarray(p, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    R, V = p.shape
    F = np.cumsum(p, axis=1)
    over = F > u[:, None]
    found = over.any(axis=1)
    x = np.where(found, over.argmax(axis=1), 0)
    if not found.all():
        pos = p > 0
        last = V - 1 - pos[:, ::-1].argmax(axis=1)
        x = np.where(found, x, last)
    rows = np.arange(R)
    Fx = F[rows, x]
    Fprev = np.where(x > 0, F[rows, np.maximum(x - 1, 0)], 0.0)
    margin = np.minimum(u - Fprev, Fx - u)
    margin = np.where(found, margin, 0.0)
    return x.astype(np.int64), margin


def argmax_first(l: np.ndarray):
    """Row argmax with ties to the lowest token id, and the gap between the two
    largest values (0 when the maximum is tied).  l [R, V]."""
    l = np.asarray(l, dtype=np.float64)
    x = l.argmax(axis=1)  # numpy returns the first maximal index
    R, V = l.shape
    if V == 1:
        return x.astype(np.int64), np.full(R, np.inf)
    top2 = np.partition(l, V - 2, axis=1)[:, V - 2:]
    gap = top2[:, 1] - top2[:, 0]
    return x.astype(np.int64), gap
