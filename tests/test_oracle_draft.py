"""Pins for the oracle's Markov-head draft sampler (CPU only).

Each pin reduces the sampler to a case fixed by mathematics or by the pages:
* with U = 0, r = V, W1 = I and W2 = log P the Markov head is exactly a
  first-order Markov chain with transition matrix P, so the joint law of
  (x_1, x_2) given the anchor is P[x0, a] P[a, b] (temperature T raises P to 1/T);
* greedy decoding of that chain follows the row argmaxes;
* with r = 0 the head vanishes (DFlash) and each position is softmax(U_k / T);
* the confidence head reads h at the same position and the embedding of the
  previous token.
"""
import numpy as np
import pytest
from scipy import special, stats

from oracle.draft import draft

SEED = 0xC0FFEE


def _chain(V, seed):
    rng = np.random.default_rng(seed)
    P = rng.dirichlet(np.full(V, 0.8), size=V)
    return P


def _markov_inputs(P, R, G, anchor, T):
    V = P.shape[0]
    U = np.zeros((R, G, V))
    W1 = np.eye(V)
    W2 = np.log(P)
    h = np.zeros((R, G, 1))
    w = np.zeros(1 + V)
    return dict(U=U, W1=W1, W2=W2, h=h, w=w, anchor=np.full(R, anchor),
                temp=np.full(R, T), seed=SEED, req_id=np.arange(R))


@pytest.mark.parametrize("T", [1.0, 0.5])
def test_markov_chain_joint_law(T):
    V, R, G, x0 = 5, 200_000, 2, 3
    P = _chain(V, 11)
    out = draft(**_markov_inputs(P, R, G, x0, T), keep_pd=False)
    PT = P ** (1.0 / T)
    PT /= PT.sum(axis=1, keepdims=True)
    expect = np.outer(PT[x0], np.ones(V)) * PT  # [a, b] = PT[x0, a] * PT[a, b]
    cells = out["tokens"][:, 0] * V + out["tokens"][:, 1]
    obs = np.bincount(cells, minlength=V * V)
    assert stats.chisquare(obs, expect.ravel() * R).pvalue > 1e-4


def test_markov_chain_probability_rows():
    V, R, G, x0 = 5, 64, 3, 1
    P = _chain(V, 12)
    out = draft(**_markov_inputs(P, R, G, x0, 1.0))
    prev = np.concatenate([np.full((R, 1), x0), out["tokens"][:, :-1]], axis=1)
    np.testing.assert_allclose(out["pd"], P[prev], rtol=1e-12, atol=0)
    np.testing.assert_allclose(out["pd"].sum(axis=2), 1.0, rtol=0, atol=1e-12)
    rows = np.arange(R)[:, None]
    np.testing.assert_array_equal(out["pd_tok"], out["pd"][rows, np.arange(G)[None], out["tokens"]])


def test_greedy_follows_row_argmax():
    V, G = 7, 6
    # a chain whose most likely successor of v is (3 v + 1) mod V
    P = np.full((V, V), 0.5 / (V - 1))
    for v in range(V):
        P[v, (3 * v + 1) % V] = 0.5
    out = draft(**_markov_inputs(P, 1, G, 2, 0.0))
    want, x = [], 2
    for _ in range(G):
        x = (3 * x + 1) % V
        want.append(x)
    assert list(out["tokens"][0]) == want
    onehot = np.zeros((G, V))
    onehot[np.arange(G), want] = 1.0
    np.testing.assert_array_equal(out["pd"][0], onehot)
    assert out["greedy"][0]


def test_rank_zero_is_parallel_drafting():
    rng = np.random.default_rng(3)
    V, R, G = 6, 100_000, 3
    U1 = rng.normal(size=(G, V)) * 1.5
    U = np.broadcast_to(U1, (R, G, V))
    T = 0.8
    out = draft(U, np.zeros((V, 0)), np.zeros((0, V)), np.zeros((R, G, 2)), np.zeros(2),
                np.zeros(R, np.int64), np.full(R, T), SEED, np.arange(R), keep_pd=False)
    for k in range(G):
        p = special.softmax(U1[k] / T)
        obs = np.bincount(out["tokens"][:, k], minlength=V)
        assert stats.chisquare(obs, p * R).pvalue > 1e-4
    # positions are independent when the head vanishes
    joint = np.bincount(out["tokens"][:, 0] * V + out["tokens"][:, 1], minlength=V * V)
    p0, p1 = special.softmax(U1[0] / T), special.softmax(U1[1] / T)
    assert stats.chisquare(joint, np.outer(p0, p1).ravel() * R).pvalue > 1e-4


def test_confidence_reads_previous_token_and_same_position_hidden():
    V, R, G = 5, 16, 4
    P = _chain(V, 5)
    inp = _markov_inputs(P, R, G, 4, 1.0)
    w_e = np.array([-2.0, -1.0, 0.0, 1.0, 2.0])
    H = 3
    h = np.zeros((R, G, H))
    h[:, :, 0] = np.arange(1, G + 1)[None, :]  # h_k[0] = k
    inp["h"] = h
    inp["w"] = np.concatenate([[0.25, 0.0, 0.0], w_e])
    out = draft(**inp, keep_pd=False)
    prev = np.concatenate([np.full((R, 1), 4), out["tokens"][:, :-1]], axis=1)
    z_expect = 0.25 * np.arange(1, G + 1)[None, :] + w_e[prev]
    np.testing.assert_allclose(out["conf_logit"], z_expect, rtol=0, atol=1e-14)
    np.testing.assert_allclose(out["conf"], special.expit(z_expect), rtol=1e-14)


def test_page_example_markov_bias_direction():
    # [DSpark] 马尔可夫头: after "of" is drawn at position 1 the head raises
    # "course" and lowers "problem" at position 2.  Tokens: 0 of, 1 course, 2 problem, 3 no.
    V, r = 4, 2
    W1 = np.zeros((V, r))
    W1[0] = [1.0, 0.0]       # "of"
    W1[3] = [0.0, 1.0]       # "no"
    W2 = np.zeros((r, V))
    W2[0, 1], W2[0, 2] = 2.0, -2.0   # after "of": +course, -problem
    W2[1, 1], W2[1, 2] = -2.0, 2.0   # after "no": -course, +problem
    U = np.zeros((1, 2, V))
    U[0, 0] = [3.0, -9.0, -9.0, 3.0]  # position 1: "of" or "no"
    U[0, 1] = [-9.0, 1.0, 1.0, -9.0]  # position 2: "course" or "problem", parallel-ambiguous
    R = 40_000
    out = draft(np.broadcast_to(U, (R, 2, V)), W1, W2, np.zeros((R, 2, 1)), np.zeros(1 + r),
                np.zeros(R, np.int64), np.ones(R), SEED, np.arange(R), keep_pd=False)
    t = out["tokens"]
    after_of = t[t[:, 0] == 0, 1]
    after_no = t[t[:, 0] == 3, 1]
    assert after_of.size > 1000 and after_no.size > 1000
    assert np.mean(after_of == 1) > 0.9 and np.mean(after_no == 2) > 0.9


def test_batch_composition_invariance():
    rng = np.random.default_rng(9)
    R, G, V, r, H = 6, 3, 40, 4, 5
    args = dict(U=rng.normal(size=(R, G, V)), W1=rng.normal(size=(V, r)) * 0.3,
                W2=rng.normal(size=(r, V)) * 0.3, h=rng.normal(size=(R, G, H)),
                w=rng.normal(size=H + r), anchor=rng.integers(0, V, R),
                temp=np.array([1.0, 0.0, 0.7, 1.0, 1.3, 0.0]), seed=77, req_id=np.arange(100, 100 + R))
    full = draft(**args)
    sub = [4, 1, 2]
    part = draft(**{k: (v[sub] if isinstance(v, np.ndarray) and v.shape[:1] == (R,) else v)
                    for k, v in args.items()})
    np.testing.assert_array_equal(full["tokens"][sub], part["tokens"])
    np.testing.assert_array_equal(full["pd"][sub], part["pd"])
