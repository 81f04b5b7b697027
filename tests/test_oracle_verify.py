"""Pins for the oracle's lossless verification (CPU only).

* lossless: the emitted token at output slot j follows p_t^j, whatever the draft
  ([DSpark] 背景知识与设计原则; [MTP Survey] §2.2), checked by chi-square over
  10^6 independent requests, with a fixed verify length and with the
  early-stopping scheduler choosing it;
* the acceptance rate at a position equals sum_v min(p_t, p_d) = 1 - TV
  ([DSpark] 置信度头的设计, the soft label c* = 1 - ||p_d - p_t||_1 / 2);
* greedy verification of a draft equal to the target accepts everything and
  emits the argmax chain plus the argmax bonus;
* degenerate cases: p_d = p_t never rejects, l = 0 emits one target sample;
* cap-accept (full-block verification, a committed window): the committed
  tokens follow p_t^j, the committed length has the law of compact
  verification with the same window, and a window of gamma or more commits
  the full output.
"""
import numpy as np
import pytest
from scipy import special, stats

from oracle.draft import draft, draft_row_distribution
from oracle.verify import cap_accept, verify
from oracle import schedule as S

SEED = 0xDEC0DE


def _setup(V, G, r, seed, R):
    rng = np.random.default_rng(seed)
    tgt = rng.normal(size=(G + 1, V)) * 1.5
    U = tgt[:G] + rng.normal(size=(G, V)) * 1.2
    W1 = rng.normal(size=(V, r)) * 0.8
    W2 = rng.normal(size=(r, V)) * 0.8
    H = 3
    h = rng.normal(size=(G, H))
    w = rng.normal(size=H + r)
    x0 = 2
    return dict(tgt=tgt, U=U, W1=W1, W2=W2, h=h, w=w, x0=x0, R=R)


def _run(st, T, ell, seed=SEED):
    R, G, V = st["R"], st["U"].shape[0], st["U"].shape[1]
    d = draft(np.broadcast_to(st["U"], (R, G, V)), st["W1"], st["W2"], np.broadcast_to(st["h"], (R,) + st["h"].shape),
              st["w"], np.full(R, st["x0"]), np.full(R, T), seed, np.arange(R))
    fl = S.flatten(ell, np.full(R, st["x0"]), d["tokens"])
    rows = st["tgt"][fl["mark_pos"]]  # synthetic target rows do not depend on the prefix
    v = verify(rows, fl["offsets"], ell, d["tokens"], d["pd"], d["pd_tok"], np.full(R, T), seed, np.arange(R))
    return d, v


def _check_output_marginals(st, v, T, G):
    pt = special.softmax(st["tgt"] / T, axis=1)
    V = pt.shape[1]
    for j in range(min(G, 3)):
        sel = v["n_out"] > j
        obs = np.bincount(v["out_tok"][sel, j], minlength=V)
        assert sel.sum() > 5_000
        assert stats.chisquare(obs, pt[j] * sel.sum()).pvalue > 1e-4, f"slot {j}"


@pytest.mark.slow
@pytest.mark.parametrize("T", [1.0, 0.7])
def test_lossless_fixed_length(T):
    V, G, R = 8, 3, 1_000_000
    st = _setup(V, G, 3, 1, R)
    d, v = _run(st, T, np.full(R, G))
    _check_output_marginals(st, v, T, G)


@pytest.mark.slow
def test_lossless_with_early_stopping_scheduler():
    V, G, Rb, nb, T = 8, 3, 500, 400, 1.0
    st = _setup(V, G, 3, 2, Rb * nb)
    R = st["R"]
    # per-request hidden states (independent of the draft tokens) spread the confidences
    h = np.random.default_rng(99).normal(size=(R, G, st["h"].shape[1])) * 1.5
    d = draft(np.broadcast_to(st["U"], (R, G, V)), st["W1"], st["W2"], h,
              st["w"], np.full(R, st["x0"]), np.full(R, T), SEED, np.arange(R))
    c, _ = S.sts_calibrate(d["conf_logit"].astype(np.float32), np.ones(G, np.float32))
    a = S.survival(c)
    n = np.arange(Rb * (1 + G) + 1, dtype=np.float64)
    sps = 100.0 * np.exp(-n / (4.0 * Rb))
    ell = np.concatenate([S.prefix_schedule(a[b * Rb:(b + 1) * Rb], sps)["ell"] for b in range(nb)])
    assert 0.2 < ell.mean() < G - 0.2 and len(np.unique(ell)) == G + 1  # lengths really vary
    fl = S.flatten(ell, np.full(R, st["x0"]), d["tokens"])
    v = verify(st["tgt"][fl["mark_pos"]], fl["offsets"], ell, d["tokens"], d["pd"], d["pd_tok"],
               np.full(R, T), SEED, np.arange(R))
    _check_output_marginals(st, v, T, G)


def test_acceptance_equals_one_minus_tv():
    V, G, R, T = 8, 2, 400_000, 1.0
    st = _setup(V, G, 3, 3, R)
    d, v = _run(st, T, np.full(R, G))
    pt = special.softmax(st["tgt"] / T, axis=1)
    pd1 = draft_row_distribution(st["U"][0], st["W1"], st["W2"], st["x0"], T)
    acc = np.minimum(pt[0], pd1).sum()
    rate = np.mean(v["n_accept"] >= 1)
    assert abs(rate - acc) < 4 * np.sqrt(acc * (1 - acc) / R)
    # position 2, conditioned on the accepted first token a: 1 - TV(p_t^2, p_d^2(.|a))
    for a_tok in range(V):
        sel = (v["n_accept"] >= 1) & (d["tokens"][:, 0] == a_tok)
        if sel.sum() < 5000:
            continue
        pd2 = draft_row_distribution(st["U"][1], st["W1"], st["W2"], a_tok, T)
        acc2 = np.minimum(pt[1], pd2).sum()
        rate2 = np.mean(v["n_accept"][sel] >= 2)
        assert abs(rate2 - acc2) < 4.5 * np.sqrt(acc2 * (1 - acc2) / sel.sum())


def test_greedy_draft_equal_to_target():
    rng = np.random.default_rng(4)
    V, G, R = 50, 5, 6
    tgt = rng.normal(size=(R, G + 1, V)) * 3
    d = draft(tgt[:, :G], np.zeros((V, 0)), np.zeros((0, V)), np.zeros((R, G, 1)), np.zeros(1),
              rng.integers(0, V, R), np.zeros(R), SEED, np.arange(R))
    ell = np.full(R, G)
    fl = S.flatten(ell, np.zeros(R), d["tokens"])
    rows = tgt[fl["mark_req"], fl["mark_pos"]]
    v = verify(rows, fl["offsets"], ell, d["tokens"], d["pd"], d["pd_tok"], np.zeros(R), SEED, np.arange(R))
    assert np.all(v["n_accept"] == G)
    np.testing.assert_array_equal(v["out_tok"][:, :G], tgt[:, :G].argmax(axis=2))
    np.testing.assert_array_equal(v["out_tok"][:, G], tgt[:, G].argmax(axis=1))


def test_greedy_rejection_emits_target_argmax():
    V, G = 10, 3
    tgt = np.zeros((1, G + 1, V))
    tgt[0, 0, 4] = tgt[0, 1, 7] = tgt[0, 2, 1] = tgt[0, 3, 9] = 5.0
    tokens = np.array([[4, 2, 1]])  # position 2 disagrees with the target argmax 7
    fl = S.flatten(np.array([G]), np.array([0]), tokens)
    v = verify(tgt[0, fl["mark_pos"]], fl["offsets"], np.array([G]), tokens, np.zeros((1, G, V)),
               np.ones((1, G)), np.zeros(1), SEED, np.arange(1))
    assert v["n_accept"][0] == 1 and list(v["out_tok"][0]) == [4, 7, -1, -1]


def test_draft_equal_target_never_rejects():
    V, G, R, T = 12, 4, 20_000, 0.9
    rng = np.random.default_rng(6)
    tgt = rng.normal(size=(G + 1, V)) * 2
    d = draft(np.broadcast_to(tgt[:G] * 1.0, (R, G, V)), np.zeros((V, 0)), np.zeros((0, V)),
              np.zeros((R, G, 1)), np.zeros(1), np.zeros(R, np.int64), np.full(R, T), SEED, np.arange(R))
    ell = np.full(R, G)
    fl = S.flatten(ell, np.zeros(R), d["tokens"])
    v = verify(tgt[fl["mark_pos"]], fl["offsets"], ell, d["tokens"], d["pd"], d["pd_tok"],
               np.full(R, T), SEED, np.arange(R))
    assert np.all(v["n_accept"] == G)
    obs = np.bincount(v["out_tok"][:, G], minlength=V)
    assert stats.chisquare(obs, special.softmax(tgt[G] / T) * R).pvalue > 1e-4


def test_zero_length_emits_one_target_sample():
    V, G, R, T = 9, 3, 50_000, 1.0
    rng = np.random.default_rng(8)
    tgt = rng.normal(size=(G + 1, V)) * 2
    tokens = rng.integers(0, V, (R, G))
    ell = np.zeros(R, np.int64)
    fl = S.flatten(ell, np.zeros(R), tokens)
    v = verify(tgt[fl["mark_pos"]], fl["offsets"], ell, tokens, np.zeros((R, G, V)), np.ones((R, G)),
               np.full(R, T), SEED, np.arange(R))
    assert np.all(v["n_accept"] == 0) and np.all(v["n_out"] == 1) and np.all(v["out_tok"][:, 1:] == -1)
    obs = np.bincount(v["out_tok"][:, 0], minlength=V)
    assert stats.chisquare(obs, special.softmax(tgt[0] / T) * R).pvalue > 1e-4


def test_residual_zero_mass_falls_back_to_target():
    # inconsistent inputs (p_d row equal to p_t but a large recorded p_d(x)) force a
    # rejection whose residual has no mass; the guard samples p_t instead
    V, G, T = 6, 1, 1.0
    tgt = np.linspace(0, 1, V)[None].repeat(G + 1, 0)
    pt = special.softmax(tgt[0])
    fl = S.flatten(np.array([1]), np.array([0]), np.array([[0]]))
    v = verify(tgt[fl["mark_pos"]], fl["offsets"], np.array([1]), np.array([[0]]), pt[None, None, :],
               np.array([[1e9]]), np.array([T]), SEED, np.array([0]))
    assert v["n_accept"][0] == 0 and v["residual_fallback"][0]
    assert 0 <= v["out_tok"][0, 0] < V


@pytest.mark.slow
def test_cap_accept_is_lossless():
    V, G, R, T = 8, 3, 600_000, 1.0
    st = _setup(V, G, 3, 5, R)
    _, v = _run(st, T, np.full(R, G))
    cap = np.random.default_rng(17).integers(0, G + 1, R)
    c = cap_accept(v, cap)
    _check_output_marginals(st, c, T, G)


@pytest.mark.slow
@pytest.mark.parametrize("window", [0, 1, 2])
def test_cap_accept_commits_like_compact_verification(window):
    # the committed length under cap-accept and the emitted length under compact
    # verification with l = window have the same law (two independent samples)
    V, G, R, T = 8, 3, 200_000, 1.0
    st = _setup(V, G, 3, 6, R)
    _, full = _run(st, T, np.full(R, G), seed=SEED)
    c = cap_accept(full, np.full(R, window))
    _, compact = _run(st, T, np.full(R, window), seed=SEED + 1)
    a = np.bincount(c["n_out"], minlength=window + 2)[1:window + 2]
    b = np.bincount(compact["n_out"], minlength=window + 2)[1:window + 2]
    if window == 0:
        assert a.sum() == b.sum() == R
    else:
        assert stats.chi2_contingency(np.stack([a, b])).pvalue > 1e-4


def test_cap_accept_structure():
    V, G, R, T = 8, 4, 2000, 1.0
    st = _setup(V, G, 3, 7, R)
    _, v = _run(st, T, np.full(R, G))
    same = cap_accept(v, np.full(R, G + 3))
    assert np.array_equal(same["n_out"], v["n_out"]) and np.array_equal(same["out_tok"], v["out_tok"])
    cap = np.random.default_rng(3).integers(0, G + 1, R)
    c = cap_accept(v, cap)
    assert np.array_equal(c["n_accept"], v["n_accept"])  # the observation: the full-block count
    assert np.array_equal(c["n_out"], np.minimum(v["n_accept"], cap) + 1)
    for r in range(R):
        k = c["n_out"][r]
        assert np.array_equal(c["out_tok"][r, :k], v["out_tok"][r, :k]) and np.all(c["out_tok"][r, k:] == -1)
    # a window of 0 commits one token: x_1 if it was accepted, else the correction
    z = cap_accept(v, np.zeros(R))
    assert np.all(z["n_out"] == 1) and np.array_equal(z["out_tok"][:, 0], v["out_tok"][:, 0])


def _rejecting_requests(V, R, seed):
    """R one-position requests with the same p_t and p_d rows, draft tokens drawn from p_d."""
    rng = np.random.default_rng(seed)
    zt = rng.normal(size=(2, V)) * 0.8
    pd_row = special.softmax(rng.normal(size=V) * 0.8)  # independent of the target: p_t > p_d at several tokens
    pt = special.softmax(zt[0])
    tok = rng.choice(V, size=R, p=pd_row)[:, None]
    pd = np.broadcast_to(pd_row, (R, 1, V))
    return zt, pt, pd_row, tok, pd


def _residual_counts(verify_fn, V, R, seed, **kw):
    zt, pt, pd_row, tok, pd = _rejecting_requests(V, R, seed)
    rows = np.tile(zt, (R, 1))
    offsets = np.arange(R + 1) * 2
    v = verify_fn(rows, offsets, np.ones(R, np.int64), tok, pd, pd_row[tok[:, 0]][:, None], np.ones(R), 99,
                  np.arange(R), **kw)
    rej = v["n_accept"] == 0
    return np.bincount(v["out_tok"][rej, 0], minlength=V), rej.sum(), pt, pd_row


def test_residual_by_rejection_samples_the_residual():
    counts, n, pt, pd_row = _residual_counts(verify, 9, 120_000, 4, residual="rejection")
    q = np.maximum(0.0, pt - pd_row)
    q /= q.sum()
    pos = q > 0
    assert n > 20_000 and pos.sum() >= 3
    assert stats.chisquare(counts[pos], q[pos] * n).pvalue > 1e-4
    assert counts[~pos].sum() == 0  # tokens where p_d >= p_t are never the correction


def test_rejection_residual_without_trials_is_the_inverse_cdf_rule():
    zt, pt, pd_row, tok, pd = _rejecting_requests(9, 3000, 4)
    R = tok.shape[0]
    args = (np.tile(zt, (R, 1)), np.arange(R + 1) * 2, np.ones(R, np.int64), tok, pd, pd_row[tok[:, 0]][:, None],
            np.ones(R), 5, np.arange(R))
    a = verify(*args)
    b = verify(*args, residual="rejection", max_trials=0)
    assert np.array_equal(a["out_tok"], b["out_tok"]) and np.array_equal(a["n_accept"], b["n_accept"])
    assert b["residual_fallback"][a["n_accept"] == 0].all()


@pytest.mark.slow
def test_lossless_with_the_rejection_residual():
    V, G, R, T = 8, 3, 300_000, 1.0
    st = _setup(V, G, 3, 8, R)
    d = draft(np.broadcast_to(st["U"], (R, G, V)), st["W1"], st["W2"], np.broadcast_to(st["h"], (R,) + st["h"].shape),
              st["w"], np.full(R, st["x0"]), np.full(R, T), SEED, np.arange(R))
    ell = np.full(R, G)
    fl = S.flatten(ell, np.full(R, st["x0"]), d["tokens"])
    v = verify(st["tgt"][fl["mark_pos"]], fl["offsets"], ell, d["tokens"], d["pd"], d["pd_tok"], np.full(R, T), SEED,
               np.arange(R), residual="rejection")
    _check_output_marginals(st, v, T, G)
