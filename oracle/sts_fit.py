"""Fitting of the Sequential Temperature Scaling temperatures (oracle).

TEST INFRASTRUCTURE: only tests/, the package smoke check and the bench's CPU
legs may import this module; the product path never does.

[DSpark] 方法细节, "事后校准（Post-hoc Calibration）" (and the survey page's
§4.2.3 "Sequential Temperature Scaling (STS) 校准"): on held-out data the
temperatures are fitted one position at a time, left to right.  At position k a
one-dimensional grid search picks the temperature whose calibrated cumulative
product prod_{i<=k} c'_i has the smallest expected calibration error (ECE),
with the positions before k held at the temperatures already chosen.

Readings where the pages say no more than that:

* ECE is the usual binned estimate (Guo et al., "On Calibration of Modern
  Neural Networks", ICML 2017): M equal-width bins on [0, 1], bin m holds the
  predictions p with m/M <= p < (m+1)/M (p = 1 goes to the last bin), and
  ECE = sum_m (n_m / N) |acc_m - conf_m| = (1/N) sum_m |sum_{n in m} (y_n - p_n)|.
  An empty sample has ECE 0.
* The label of block n at position k is 1 when its first k draft tokens were
  all accepted by a verification of the full block (accept_len[n] >= k); every
  held-out block counts at every position, since the cumulative product is the
  probability that the whole prefix survives.
* The prediction is the scheduler's survival product: c' = fp32(sigmoid(z/tau))
  with the sigmoid in fp64, multiplied left to right in fp32.
* The grid of candidate temperatures is the caller's; ties go to the first
  grid entry.

Parity pins: tests/test_oracle_sts_fit.py (a hand-worked ECE, bin edges, the
one-bin closed form, exact calibration, degenerate label sets with a known
optimum, exact scale equivariance, left-to-right independence, recovery of a
known over-confidence) and tests/test_oracle_mutations.py.
"""
from __future__ import annotations

import numpy as np

from .schedule import sts_calibrate


def bin_index(pred, n_bins: int):
    """Equal-width bin of each prediction in [0, 1]: floor(p * M), p = 1 -> M - 1.

    The product p * M is exact in fp64 for fp32 predictions and M < 2^29."""
    p = np.asarray(pred, dtype=np.float64)
    return np.minimum(np.floor(p * n_bins).astype(np.int64), n_bins - 1)


def ece(pred, label, n_bins: int) -> float:
    """Binned expected calibration error of predictions against 0/1 labels."""
    p = np.asarray(pred, dtype=np.float64).ravel()
    y = np.asarray(label, dtype=np.float64).ravel()
    N = p.size
    if N == 0:
        return 0.0
    m = bin_index(p, n_bins)
    gap = np.bincount(m, weights=y - p, minlength=n_bins)
    return float(np.sum(np.abs(gap)) / N)


def sts_fit(conf_logit, accept_len, grid, n_bins: int = 15):
    """Left-to-right grid search of one temperature per draft position.

    conf_logit [N, g] fp32 confidence logits of held-out draft blocks;
    accept_len [N] draft tokens accepted by a verification of the full block
    (0..g); grid [G] fp32 candidate temperatures (> 0).

    Returns dict(sts_temp [g] float32, grid_index [g] int64, ece [g, G] fp64
    (ECE of the cumulative product at every candidate), ece_best [g],
    ece_gap [g] (second-smallest minus smallest ECE at that position, inf when
    G = 1), ece_raw [g] (ECE with every temperature 1), surv [N, g] float32
    (the calibrated cumulative products))."""
    z = np.asarray(conf_logit, dtype=np.float32)
    N, G_pos = z.shape
    L = np.asarray(accept_len, dtype=np.int64).reshape(N)
    grid = np.asarray(grid, dtype=np.float32).ravel()
    n_grid = grid.size
    if n_grid < 1 or not np.all(grid > 0) or not np.all(np.isfinite(grid)):
        raise ValueError("the temperature grid must hold at least one finite positive value")
    if np.any(L < 0) or np.any(L > G_pos):
        raise ValueError("accept_len must lie in 0..gamma")

    table = np.zeros((G_pos, n_grid), dtype=np.float64)
    index = np.zeros(G_pos, dtype=np.int64)
    raw = np.zeros(G_pos, dtype=np.float64)
    surv = np.empty((N, G_pos), dtype=np.float32)
    prev = np.ones(N, dtype=np.float32)      # calibrated product of positions before k
    prev_raw = np.ones(N, dtype=np.float32)  # the same with every temperature 1
    for k in range(G_pos):
        label = L >= k + 1
        zk = z[:, k:k + 1]
        for g in range(n_grid):
            c, _ = sts_calibrate(zk, grid[g:g + 1])
            p = (prev * c[:, 0]).astype(np.float32)
            table[k, g] = ece(p, label, n_bins)
        index[k] = int(np.argmin(table[k]))  # first minimum
        c, _ = sts_calibrate(zk, grid[index[k]:index[k] + 1])
        prev = (prev * c[:, 0]).astype(np.float32)
        surv[:, k] = prev
        c1, _ = sts_calibrate(zk, np.ones(1, np.float32))
        prev_raw = (prev_raw * c1[:, 0]).astype(np.float32)
        raw[k] = ece(prev_raw, label, n_bins)
    srt = np.sort(table, axis=1)
    gap = srt[:, 1] - srt[:, 0] if n_grid > 1 else np.full(G_pos, np.inf)
    return dict(sts_temp=grid[index].astype(np.float32), grid_index=index, ece=table,
                ece_best=table[np.arange(G_pos), index], ece_gap=gap, ece_raw=raw, surv=surv)
