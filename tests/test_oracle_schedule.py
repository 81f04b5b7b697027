"""Pins for the oracle's STS, prefix scheduler and flatten (CPU only)."""
import itertools
import os

import numpy as np
import pytest
from scipy import special

from oracle import schedule as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "appendix_a_counterexample.txt")


def _golden():
    d = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            d[k] = float(v)
    return d


def test_appendix_a_counterexample():
    g = _golden()
    sps = np.array([0.0, g["sps1"], g["sps2"], g["sps3"]])
    a1 = np.float32(g["a1"])
    # with the early stop: Theta_0 = 1.0, Theta_1 = 0.9 -> stop, l = 0
    for c2 in (g["c2_high"], g["c2_low"]):
        a = np.array([[a1, np.float32(a1 * np.float32(c2))]], np.float32)
        res = S.prefix_schedule(a, sps, S.MODE_GREEDY, early_stop=True)
        assert res["ell"][0] == g["early_stop_ell"]
        assert res["thetas"][0] == pytest.approx(g["theta0"], rel=1e-7)
        assert res["thetas"][1] == pytest.approx(g["theta1"], rel=1e-7)
        assert len(res["thetas"]) == 2  # nothing after the first drop is evaluated
        assert res["theta_best"] == pytest.approx(g["theta0"], rel=1e-7)
    # without it, the choice of l depends on c2, i.e. on the value of x1
    a_hi = np.array([[a1, np.float32(a1 * np.float32(g["c2_high"]))]], np.float32)
    res = S.prefix_schedule(a_hi, sps, S.MODE_GREEDY, early_stop=False)
    assert float(a_hi[0, 1]) == pytest.approx(g["a2_high"], rel=1e-7)
    assert res["thetas"][2] == pytest.approx(g["theta2_high"], rel=1e-7)
    assert res["ell"][0] == g["no_stop_ell_high"]
    a_lo = np.array([[a1, np.float32(0.0)]], np.float32)
    res = S.prefix_schedule(a_lo, sps, S.MODE_GREEDY, early_stop=False)
    assert res["ell"][0] == g["no_stop_ell_low"]
    # the page evaluates Theta_2 with a2 = 0 as well
    assert (1.0 + float(a1) + 0.0) * g["sps3"] == pytest.approx(g["theta2_low"], rel=1e-7)


def _theta_of(ell, a, sps):
    R = a.shape[0]
    tau = R + sum(float(a[r, :ell[r]].astype(np.float64).sum()) for r in range(R))
    return tau * sps[R + int(np.sum(ell))]


def _random_case(rng, R, G):
    c = rng.uniform(0.05, 1.0, size=(R, G)).astype(np.float32)
    c[rng.random((R, G)) < 0.1] = 0.0
    a = S.survival(c)
    n = np.arange(R * (1 + G) + 1, dtype=np.float64)
    kind = rng.integers(3)
    if kind == 0:  # smooth decreasing curve
        sps = 100.0 / (1.0 + n / rng.uniform(2, 20))
    elif kind == 1:  # stepped curve with cliffs (non-unimodal paths)
        sps = 100.0 / (1.0 + np.floor(n / rng.integers(2, 5)) * rng.uniform(0.2, 1.0))
    else:  # random decreasing table
        sps = np.sort(rng.uniform(1, 100, size=n.size))[::-1].copy()
    sps[0] = 0.0
    return a, sps


@pytest.mark.parametrize("seed", range(40))
def test_brute_force_enumeration(seed):
    rng = np.random.default_rng(seed)
    R, G = int(rng.integers(1, 5)), int(rng.integers(1, 5))
    a, sps = _random_case(rng, R, G)
    # (i) the best Theta over all (G+1)^R length vectors equals the best prefix of
    #     the sorted path (top-n survival sets dominate for every total n)
    best = max(_theta_of(ell, a, sps) for ell in itertools.product(range(G + 1), repeat=R))
    full = S.prefix_schedule(a, sps, S.MODE_GREEDY, early_stop=False)
    assert full["theta_best"] == pytest.approx(best, rel=1e-12)
    assert _theta_of(full["ell"], a, sps) == pytest.approx(best, rel=1e-12)
    # (ii)/(iii) the early-stop result is the first local maximum along the path
    es = S.prefix_schedule(a, sps, S.MODE_GREEDY, early_stop=True)
    path = full["thetas"]
    i = 0
    while i + 1 < len(path) and path[i + 1] > path[i]:
        i += 1
    assert es["n_admit"] == i
    assert es["theta_best"] == pytest.approx(path[i], rel=1e-15)
    assert _theta_of(es["ell"], a, sps) == pytest.approx(path[i], rel=1e-12)
    if all(path[k + 1] <= path[k] for k in range(i, len(path) - 1)):
        assert es["theta_best"] == pytest.approx(best, rel=1e-12)
    # (iv) every kept set is a prefix: l_r equals the number of kept (r, .) candidates
    rr, jj = S.sorted_candidates(a)
    kept = np.bincount(rr[:es["n_admit"]], minlength=R)
    np.testing.assert_array_equal(kept, es["ell"])
    for r in range(R):
        assert sorted(jj[:es["n_admit"]][rr[:es["n_admit"]] == r]) == list(range(es["ell"][r]))


def test_sorted_candidates_order_and_filter():
    a = np.array([[0.9, 0.5, 0.0], [0.9, 0.9, 0.2]], np.float32)
    rr, jj = S.sorted_candidates(a)
    assert list(zip(rr, jj)) == [(0, 0), (1, 0), (1, 1), (0, 1), (1, 2)]


def test_sts_identity_order_and_shrink():
    rng = np.random.default_rng(2)
    z = (rng.normal(size=(64, 5)) * 3).astype(np.float32)
    c1, margin = S.sts_calibrate(z, np.ones(5, np.float32))
    np.testing.assert_array_equal(c1, special.expit(z.astype(np.float64)).astype(np.float32))
    assert margin.min() > 0
    tau = np.array([0.8, 1.0, 1.5, 2.0, 3.0], np.float32)
    c, _ = S.sts_calibrate(z, tau)
    for k in range(5):
        # order preserving within each position
        assert np.all(np.argsort(z[:, k], kind="stable") == np.argsort(c[:, k], kind="stable"))
    # tau > 1 pulls towards 1/2, tau < 1 pushes away from it
    d1 = np.abs(c1.astype(np.float64) - 0.5)
    d = np.abs(c.astype(np.float64) - 0.5)
    assert np.all(d[:, 2:] <= d1[:, 2:]) and np.all(d[:, 0] >= d1[:, 0])


def test_survival_is_fp32_running_product():
    c = np.array([[0.9, 0.8, 0.7, 0.0, 0.5]], np.float32)
    a = S.survival(c)
    want = [np.float32(0.9)]
    for v in c[0, 1:]:
        want.append(np.float32(want[-1] * v))
    np.testing.assert_array_equal(a[0], np.array(want, np.float32))
    assert np.all(np.diff(a[0].astype(np.float64)) <= 0)


def test_mode_off_and_flatten():
    R, G = 3, 4
    anchor = np.array([7, 8, 9])
    tokens = np.arange(R * G).reshape(R, G) + 100
    res = S.prefix_schedule(np.ones((R, G), np.float32), np.ones(R * (G + 1) + 1), S.MODE_OFF)
    assert list(res["ell"]) == [G] * R
    fl = S.flatten(np.array([2, 0, 4]), anchor, tokens)
    assert list(fl["offsets"]) == [0, 3, 4, 9]
    assert list(fl["flat_tok"]) == [7, 100, 101, 8, 9, 108, 109, 110, 111]
    assert list(fl["mark_req"]) == [0, 0, 0, 1, 2, 2, 2, 2, 2]
    assert list(fl["mark_pos"]) == [0, 1, 2, 0, 0, 1, 2, 3, 4]


def test_schedule_end_to_end_invariants():
    rng = np.random.default_rng(5)
    R, G = 32, 6
    z = (rng.normal(size=(R, G)) * 2 + 1).astype(np.float32)
    tau = rng.uniform(0.8, 1.5, size=G).astype(np.float32)
    n = np.arange(R * (1 + G) + 1, dtype=np.float64)
    sps = 60 * (1 - np.exp(-64.0 / np.maximum(n, 1)))
    res = S.schedule(z, tau, sps, rng.integers(0, 50, R), rng.integers(0, 50, (R, G)))
    assert res["offsets"][-1] == R + res["ell"].sum()
    assert 0 <= res["ell"].min() and res["ell"].max() <= G
    assert res["theta_best"] >= R * sps[R]


# ---- the asynchronous production variant (capacity from earlier confidences) ----

def test_async_appendix_a():
    # with the earlier survivals equal to the current ones the capacity is the
    # global (no early stop) optimum of the appendix: l = 2 when c2 = 0.9, 0 when c2 = 0
    g = _golden()
    sps = np.array([0.0, g["sps1"], g["sps2"], g["sps3"]])
    a1 = np.float32(g["a1"])
    a_hi = np.array([[a1, np.float32(a1 * np.float32(g["c2_high"]))]], np.float32)
    a_lo = np.array([[a1, np.float32(0.0)]], np.float32)
    res = S.async_topk_schedule(a_hi, a_hi, sps)
    assert res["K"] == 2 and res["ell"][0] == g["no_stop_ell_high"]
    assert res["cap_theta"] == pytest.approx(g["theta2_high"], rel=1e-7)
    res = S.async_topk_schedule(a_lo, a_lo, sps)
    assert res["K"] == 0 and res["ell"][0] == g["no_stop_ell_low"]
    # the causal barrier: the capacity comes from the earlier step only; a current
    # step whose x1 ends the candidates admits what it has, up to K
    res = S.async_topk_schedule(a_lo, a_hi, sps)
    assert res["K"] == 2 and res["ell"][0] == 1 and res["n_admit"] == 1


@pytest.mark.parametrize("seed", range(30))
def test_async_capacity_is_the_brute_force_optimum(seed):
    rng = np.random.default_rng(100 + seed)
    R, G = int(rng.integers(1, 5)), int(rng.integers(1, 5))
    a_prev, sps = _random_case(rng, R, G)
    a_now, _ = _random_case(rng, R, G)
    res = S.async_topk_schedule(a_now, a_prev, sps)
    best = max(_theta_of(ell, a_prev, sps) for ell in itertools.product(range(G + 1), repeat=R))
    assert res["cap_theta"] == pytest.approx(best, rel=1e-12)
    # K is the first prefix length reaching the optimum on the earlier path
    assert res["K"] == int(np.argmax(np.asarray(res["thetas"]) >= res["cap_theta"]))
    # the admission is the top min(K, n_now) current candidates, prefix-closed
    rr, jj = S.sorted_candidates(a_now)
    n = min(res["K"], rr.size)
    assert res["n_admit"] == n
    np.testing.assert_array_equal(np.bincount(rr[:n], minlength=R), res["ell"])
    assert res["theta_best"] == pytest.approx(_theta_of(res["ell"], a_now, sps), rel=1e-12)


@pytest.mark.parametrize("seed", range(10))
def test_async_depends_on_current_values_only_through_their_order(seed):
    rng = np.random.default_rng(200 + seed)
    R, G = 6, 4
    a_prev, sps = _random_case(rng, R, G)
    a_now, _ = _random_case(rng, R, G)
    res = S.async_topk_schedule(a_now, a_prev, sps)
    # an order-preserving change of the current values (positive ones stay
    # positive) leaves the admitted set alone
    warped = np.where(a_now > 0, np.sqrt(a_now.astype(np.float64)) * 0.5 + 0.25, 0.0).astype(np.float32)
    res2 = S.async_topk_schedule(warped, a_prev, sps)
    np.testing.assert_array_equal(res["ell"], res2["ell"])


def test_async_equals_algorithm_1_on_a_unimodal_path():
    # same survivals in both steps and a smooth curve: the global optimum is the
    # first local maximum, so the asynchronous and greedy schedules agree
    rng = np.random.default_rng(7)
    for _ in range(20):
        R, G = 5, 4
        c = rng.uniform(0.05, 1.0, size=(R, G)).astype(np.float32)
        a = S.survival(c)
        n = np.arange(R * (1 + G) + 1, dtype=np.float64)
        sps = 100.0 / (1.0 + n / rng.uniform(2, 20))
        sps[0] = 0.0
        path = S.prefix_schedule(a, sps, S.MODE_GREEDY, early_stop=False)["thetas"]
        i = int(np.argmax(path))
        if not all(path[k + 1] > path[k] for k in range(i)) or not all(
                path[k + 1] <= path[k] for k in range(i, len(path) - 1)):
            continue
        res = S.async_topk_schedule(a, a, sps)
        es = S.prefix_schedule(a, sps, S.MODE_GREEDY, early_stop=True)
        np.testing.assert_array_equal(res["ell"], es["ell"])
        assert res["theta_best"] == pytest.approx(es["theta_best"], rel=1e-12)


def test_pack_rows_is_the_marker_gather():
    # brute force: walk the requests and their kept positions in order
    rng = np.random.default_rng(5)
    R, G, V = 6, 4, 5
    target = rng.normal(size=(R, G + 1, V))
    ell = rng.integers(0, G + 1, R)
    fl = S.flatten(ell, rng.integers(0, 9, R), rng.integers(0, 9, (R, G)))
    expect = []
    for r in range(R):
        for j in range(ell[r] + 1):
            expect.append(target[r, j])
    np.testing.assert_array_equal(S.pack_rows(target, fl["mark_req"], fl["mark_pos"]), np.array(expect))
    np.testing.assert_array_equal(S.pack_rows(target, fl["mark_req"], fl["mark_pos"], 3), np.array(expect[:3]))
