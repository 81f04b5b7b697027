"""Pins of the oracle's RNN sequential head (oracle/draft.py, W_rnn).

Each check reduces the head to a case whose answer is known without the
recurrence: an output map that reads only the embedding is a Markov head with a
transformed W1 (itself pinned by the Markov-chain closed form); an output map
that reads only h_k is a token-independent bias, a plain softmax; a saturated
gate either freezes the state at s_0 = 0 or overwrites it each step, and the
resulting rows have closed forms; with a half-open gate the state remembers
x_{k-2}, which a Markov head cannot."""
import numpy as np
import pytest
from scipy import special

from oracle.draft import draft

V, r, H, G = 6, 4, 3, 3


def _inputs(seed, R, T=1.0):
    rng = np.random.default_rng(seed)
    U = rng.normal(size=(R, G, V)) * 1.2
    W1 = rng.normal(size=(V, r))
    W2 = rng.normal(size=(r, V))
    h = rng.normal(size=(R, G, H))
    w = rng.normal(size=H + r) * 0.3
    anchor = rng.integers(0, V, R)
    return dict(U=U, W1=W1, W2=W2, h=h, w=w, anchor=anchor, temp=np.full(R, T), seed=7, req_id=np.arange(R))


def _blocks(rng, g=None, c=None, o=None):
    """W_rnn = [W_g; W_c; W_o], each [r, 2r + H] over z = [s; W1[x]; h]."""
    def blk(x):
        return rng.normal(size=(r, 2 * r + H)) if x is None else x
    return np.concatenate([blk(g), blk(c), blk(o)], axis=0)


@pytest.mark.parametrize("T", [1.0, 0.6, 0.0])
def test_embedding_only_output_is_a_markov_head(T):
    rng = np.random.default_rng(1)
    A = rng.normal(size=(r, r))
    Wo = np.zeros((r, 2 * r + H))
    Wo[:, r:2 * r] = A
    inp = _inputs(2, 300, T)
    rnn = draft(**inp, W_rnn=_blocks(rng, o=Wo))
    markov = draft(**dict(inp, W1=np.tanh(inp["W1"] @ A.T)))
    assert np.array_equal(rnn["tokens"], markov["tokens"])
    np.testing.assert_allclose(rnn["pd"], markov["pd"], rtol=0, atol=1e-12)
    # the confidence head keeps reading W1[x_{k-1}] of the tokens drawn
    prev = np.concatenate([inp["anchor"][:, None], rnn["tokens"][:, :-1]], axis=1)
    zl = inp["h"] @ inp["w"][:H] + inp["W1"][prev] @ inp["w"][H:]
    np.testing.assert_allclose(rnn["conf_logit"], zl, rtol=0, atol=1e-12)


def test_hidden_only_output_is_a_token_independent_softmax():
    rng = np.random.default_rng(3)
    C = rng.normal(size=(r, H))
    Wo = np.zeros((r, 2 * r + H))
    Wo[:, 2 * r:] = C
    inp = _inputs(4, 200)
    out = draft(**inp, W_rnn=_blocks(rng, o=Wo))
    for k in range(G):
        bias = np.tanh(inp["h"][:, k] @ C.T) @ inp["W2"]
        np.testing.assert_allclose(out["pd"][:, k], special.softmax(inp["U"][:, k] + bias, axis=1), rtol=0,
                                   atol=1e-12)


def _gate_on_h0(value):
    # h_k[0] = 1 for every position, the gate reads only that entry
    Wg = np.zeros((r, 2 * r + H))
    Wg[:, 2 * r] = value
    return Wg


def test_open_gate_keeps_the_zero_state():
    # sigmoid(40) = 1 - 4e-18: s_k stays 0, tanh(W_o z) reads only the state -> no bias
    rng = np.random.default_rng(5)
    inp = _inputs(6, 200)
    inp["h"][:, :, 0] = 1.0
    Wo = np.zeros((r, 2 * r + H))
    Wo[:, :r] = rng.normal(size=(r, r)) * 3
    out = draft(**inp, W_rnn=_blocks(rng, g=_gate_on_h0(40.0), o=Wo))
    np.testing.assert_allclose(out["pd"], special.softmax(inp["U"], axis=2), rtol=0, atol=1e-13)


def test_closed_gate_holds_the_previous_embedding():
    # sigmoid(-40) ~ 0: s_k = tanh(a W1[x_{k-1}]); W_o reads the state, so position k
    # sees x_{k-2}: p_1 has no bias, p_2 reads the anchor, p_3 reads x_1
    rng = np.random.default_rng(7)
    a, Bs = 0.8, rng.normal(size=(r, r)) * 2
    inp = _inputs(8, 300)
    inp["h"][:, :, 0] = 1.0
    Wc = np.zeros((r, 2 * r + H))
    Wc[:, r:2 * r] = a * np.eye(r)
    Wo = np.zeros((r, 2 * r + H))
    Wo[:, :r] = Bs
    out = draft(**inp, W_rnn=_blocks(rng, g=_gate_on_h0(-40.0), c=Wc, o=Wo))
    W1, W2, U = inp["W1"], inp["W2"], inp["U"]
    prev2 = [None, inp["anchor"], out["tokens"][:, 0]]
    for k in range(G):
        bias = 0.0 if k == 0 else np.tanh(np.tanh(a * W1[prev2[k]]) @ Bs.T) @ W2
        np.testing.assert_allclose(out["pd"][:, k], special.softmax(U[:, k] + bias, axis=1), rtol=0, atol=1e-12)


def test_half_open_gate_remembers_two_tokens_back():
    # g = 1/2: s_2 = s_1 / 2 + tanh(a W1[x_1]) / 2 and p_3 reads s_2 only, so p_3 is a
    # function of x_1 (the anchor is fixed) and not of x_2
    rng = np.random.default_rng(9)
    R = 4000
    inp = _inputs(10, R)
    inp["U"] = np.broadcast_to(inp["U"][:1], inp["U"].shape).copy()
    inp["h"] = np.broadcast_to(inp["h"][:1], inp["h"].shape).copy()
    inp["anchor"] = np.full(R, 2)
    Wc = np.zeros((r, 2 * r + H))
    Wc[:, r:2 * r] = np.eye(r)
    Wo = np.zeros((r, 2 * r + H))
    Wo[:, :r] = rng.normal(size=(r, r)) * 3
    out = draft(**inp, W_rnn=_blocks(rng, g=np.zeros((r, 2 * r + H)), c=Wc, o=Wo))
    x1, x2, p3 = out["tokens"][:, 0], out["tokens"][:, 1], out["pd"][:, 2]
    seen_x2_variation = seen_x1_variation = False
    for a in range(V):
        rows = np.flatnonzero(x1 == a)
        if rows.size:
            np.testing.assert_array_equal(p3[rows], np.broadcast_to(p3[rows[0]], p3[rows].shape))
            seen_x2_variation |= np.unique(x2[rows]).size > 1
    firsts = [np.flatnonzero(x1 == a)[0] for a in range(V) if np.any(x1 == a)]
    seen_x1_variation = len({tuple(np.round(p3[i], 12)) for i in firsts}) == len(firsts) > 1
    assert seen_x2_variation and seen_x1_variation


def test_row_rounding_matches_the_library_conversions():
    import torch
    from oracle.draft import round_to
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.normal(size=20000), rng.uniform(-1, 1, 20000) * 1e-3, [0.0, -0.0, 1.0, -1.0]])
    np.testing.assert_array_equal(round_to(x, "f32"), x.astype(np.float32).astype(np.float64))
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(round_to(x, "bf16"), ref)


def test_rounded_rows_change_only_the_row_precision():
    # with rounding the rows are the bf16 values of the fp64 rows: the same head with
    # W_o reading only the embedding equals a Markov head with bf16-rounded tanh rows
    from oracle.draft import round_to
    rng = np.random.default_rng(12)
    A = rng.normal(size=(r, r))
    Wo = np.zeros((r, 2 * r + H))
    Wo[:, r:2 * r] = A
    inp = _inputs(13, 200)
    rnn = draft(**inp, W_rnn=_blocks(rng, o=Wo), rnn_row_dtype="bf16")
    markov = draft(**dict(inp, W1=round_to(np.tanh(inp["W1"] @ A.T), "bf16")))
    assert np.array_equal(rnn["tokens"], markov["tokens"])
    np.testing.assert_allclose(rnn["pd"], markov["pd"], rtol=0, atol=1e-12)
