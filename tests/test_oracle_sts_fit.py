"""Pins of the STS-fitting oracle (oracle/sts_fit.py).

Each check uses something other than the oracle's own formula: ECE values
worked out by hand (as exact fractions), the one-bin closed form, exact
calibration, label sets whose optimum is known in advance, exact power-of-two
scale equivariance, the left-to-right structure, and recovery of a known
over-confidence on data drawn from a logistic acceptance model."""
import numpy as np
import pytest

import synth
from oracle.sts_fit import bin_index, ece, sts_fit


def test_ece_hand_worked_example():
    # M = 5 bins of width 0.2.
    #   bin 0: p = 0.125, 0.1875 with y = 0, 1  -> |1 - 0.3125|    = 0.6875
    #   bin 2: p = 0.5, 0.5625   with y = 1, 0  -> |1 - 1.0625|    = 0.0625
    #   bin 4: p = 0.875, 0.9375, 1.0 (p = 1 closes the last bin), y = 1, 1, 1
    #                                           -> |3 - 2.8125|    = 0.1875
    #   ECE = (0.6875 + 0.0625 + 0.1875) / 7 = 15/112
    p = [0.125, 0.1875, 0.5, 0.5625, 0.875, 0.9375, 1.0]
    y = [0, 1, 1, 0, 1, 1, 1]
    assert ece(p, y, 5) == pytest.approx(15 / 112, rel=0, abs=1e-15)


def test_ece_bin_edges_are_left_closed():
    # M = 4: p = 0.25 opens bin 1 (it does not close bin 0); p = 1 closes bin 3.
    #   bin 0: 0.125 (y 1) -> 0.875;  bin 1: 0.25 (y 0) -> 0.25;
    #   bin 2: 0.5 (y 1) -> 0.5;      bin 3: 1.0, 0.75 (y 1, 0) -> |1 - 1.75| = 0.75
    #   ECE = 2.375 / 5 = 19/40.  (Right-closed bins would put 0.25 in bin 0 with 0.125.)
    p = [0.25, 0.125, 0.5, 1.0, 0.75]
    y = [0, 1, 1, 1, 0]
    assert ece(p, y, 4) == pytest.approx(19 / 40, rel=0, abs=1e-15)
    assert list(bin_index(p, 4)) == [1, 0, 2, 3, 3]


def test_ece_one_bin_is_the_gap_of_the_means():
    rng = np.random.default_rng(0)
    p = rng.random(1000).astype(np.float32)
    y = rng.random(1000) < 0.3
    assert ece(p, y, 1) == pytest.approx(abs(y.mean() - p.astype(np.float64).mean()), rel=1e-12)


def test_ece_counts_only_miscalibrated_bins():
    # with M = 4: the eight 0.25s (bin 1) have accuracy 2/8 and the four 0.75s (bin 3)
    # accuracy 3/4; 0.5 and 0.625 share bin 2 (mean 0.5625 against accuracy 0.5), the only
    # bin that is off, by |1 - 1.125| = 0.125
    p = [0.25] * 8 + [0.75] * 4 + [0.5, 0.625]
    y = [1, 1, 0, 0, 0, 0, 0, 0] + [1, 1, 1, 0] + [1, 0]
    assert ece(p, y, 4) == pytest.approx(0.125 / 14, abs=1e-15)
    assert ece(p[:12], y[:12], 4) == 0.0
    assert ece([], [], 15) == 0.0


def test_ece_is_invariant_to_sample_order():
    rng = np.random.default_rng(1)
    p = rng.random(500)
    y = rng.random(500) < p
    perm = rng.permutation(500)
    assert ece(p[perm], y[perm], 10) == pytest.approx(ece(p, y, 10), rel=1e-13)


def test_fit_all_accepted_picks_the_sharpest_temperature():
    # every block accepted in full and every logit positive: ECE = mean(1 - p), which
    # falls as p rises, i.e. as tau falls -> the smallest temperature at every position
    rng = np.random.default_rng(2)
    z = (0.5 + 3 * rng.random((400, 4))).astype(np.float32)
    L = np.full(400, 4, np.int32)
    grid = np.array([0.5, 0.8, 1.0, 1.7, 3.0], np.float32)
    o = sts_fit(z, L, grid, 10)
    assert list(o["grid_index"]) == [0, 0, 0, 0]


def test_fit_all_rejected_picks_the_sharpest_temperature():
    # nothing accepted and every logit negative: ECE = mean(p), smallest at the smallest tau
    rng = np.random.default_rng(3)
    z = (-0.5 - 3 * rng.random((400, 3))).astype(np.float32)
    L = np.zeros(400, np.int32)
    grid = np.array([0.4, 0.9, 2.0], np.float32)
    o = sts_fit(z, L, grid, 15)
    assert list(o["grid_index"]) == [0, 0, 0]


def test_fit_ties_go_to_the_first_grid_entry():
    # sigmoid(z / tau) rounds to exactly 1.0f for every candidate: all ECEs are 0
    z = np.full((50, 2), 60.0, np.float32)
    L = np.full(50, 2, np.int32)
    grid = np.array([2.0, 0.5, 1.0], np.float32)
    o = sts_fit(z, L, grid, 15)
    assert np.all(o["ece"] == 0.0)
    assert list(o["grid_index"]) == [0, 0]
    assert list(o["sts_temp"]) == [2.0, 2.0]


def test_fit_with_one_candidate_returns_it():
    z, L, _ = synth.sts_heldout(300, 3, 4)
    o = sts_fit(z, L, np.array([1.3], np.float32), 15)
    assert list(o["sts_temp"]) == [np.float32(1.3)] * 3
    assert np.all(np.isinf(o["ece_gap"]))


def test_fit_is_exactly_scale_equivariant():
    # (2 z) / (2 tau) = z / tau exactly, so every decision and every ECE is unchanged
    z, L, _ = synth.sts_heldout(2000, 4, 5, noise=0.5)
    grid = synth.sts_grid(17)
    a = sts_fit(z, L, grid, 15)
    b = sts_fit(z * np.float32(2), L, grid * np.float32(2), 15)
    assert np.array_equal(a["grid_index"], b["grid_index"])
    assert np.array_equal(a["ece"], b["ece"])


def test_fit_runs_left_to_right():
    # positions after k0 do not influence the temperatures up to k0: change their
    # logits, and the accept lengths of blocks that got past k0 (labels up to k0 stay)
    z, L, _ = synth.sts_heldout(3000, 5, 6, noise=0.4)
    grid = synth.sts_grid(21)
    a = sts_fit(z, L, grid, 15)
    k0 = 2
    rng = np.random.default_rng(7)
    z2 = z.copy()
    z2[:, k0:] = rng.normal(size=(3000, 5 - k0)).astype(np.float32) * 4
    L2 = L.copy()
    past = L >= k0
    L2[past] = rng.integers(k0, 6, size=int(past.sum()))
    b = sts_fit(z2, L2, grid, 15)
    assert np.array_equal(a["grid_index"][:k0], b["grid_index"][:k0])
    assert np.array_equal(a["ece"][:k0], b["ece"][:k0])
    assert not np.array_equal(a["ece"][k0:], b["ece"][k0:])


def test_fit_recovers_a_known_overconfidence():
    # the head reports kappa_k times the true acceptance logit; tau_k = kappa_k makes
    # the cumulative product the true prefix survival, which is calibrated
    kappa = np.array([1.5, 2.0, 1.25, 2.5])
    z, L, _ = synth.sts_heldout(200_000, 4, 8, kappa=kappa, mu0=1.5, mu_step=0.2)
    grid = synth.sts_grid(97, 0.5, 4.0)  # steps of 2.2 %
    o = sts_fit(z, L, grid, 15)
    assert np.all(np.abs(o["sts_temp"] / kappa - 1) < 0.08), (o["sts_temp"], kappa)
    assert np.all(o["ece_best"] < 0.01)
    assert np.all(o["ece_raw"] > 0.03)


def test_fit_rejects_bad_arguments():
    z = np.zeros((4, 2), np.float32)
    with pytest.raises(ValueError):
        sts_fit(z, np.array([0, 1, 2, 3]), np.ones(2, np.float32), 15)
    with pytest.raises(ValueError):
        sts_fit(z, np.zeros(4), np.array([1.0, 0.0], np.float32), 15)
