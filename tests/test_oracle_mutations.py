"""The pins have teeth: plant a plausible mistake in a copy of the oracle (on the
CPU) and check that the lossless / acceptance pins reject it.  Each mutation is a
one-token edit of the oracle's source, executed as a throw-away module."""
import importlib.util
import os
import sys
import types

import numpy as np
import pytest
from scipy import special, stats

from oracle.draft import draft
from oracle import schedule as S

ORACLE_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle")


def _mutant(module, old, new):
    src = open(os.path.join(ORACLE_DIR, module + ".py")).read()
    assert src.count(old) == 1, (module, old)
    src = src.replace(old, new)
    mod = types.ModuleType("oracle._mutant_" + module)
    mod.__package__ = "oracle"
    exec(compile(src, f"<mutant {module}>", "exec"), mod.__dict__)
    return mod


def _lossless_pvalues(verify_fn, draft_fn=draft, T=1.0, R=200_000):
    rng = np.random.default_rng(1)
    V, G, r = 8, 3, 3
    tgt = rng.normal(size=(G + 1, V)) * 1.5
    U = tgt[:G] + rng.normal(size=(G, V)) * 1.2
    W1 = rng.normal(size=(V, r)) * 0.8
    W2 = rng.normal(size=(r, V)) * 0.8
    d = draft_fn(np.broadcast_to(U, (R, G, V)), W1, W2, np.zeros((R, G, 1)), np.zeros(1 + r),
                 np.full(R, 2), np.full(R, T), 5, np.arange(R))
    ell = np.full(R, G)
    fl = S.flatten(ell, np.full(R, 2), d["tokens"])
    v = verify_fn(tgt[fl["mark_pos"]], fl["offsets"], ell, d["tokens"], d["pd"], d["pd_tok"],
                  np.full(R, T), 5, np.arange(R))
    pt = special.softmax(tgt / T, axis=1)
    ps = []
    for j in range(G):
        sel = v["n_out"] > j
        obs = np.bincount(v["out_tok"][sel, j], minlength=V)
        ps.append(stats.chisquare(obs, pt[j] * sel.sum()).pvalue)
    return ps


def test_unmutated_oracle_passes():
    from oracle.verify import verify
    assert min(_lossless_pvalues(verify)) > 1e-4


@pytest.mark.parametrize("old,new", [
    ("q = np.maximum(0.0, pt - pdr)", "q = np.maximum(0.0, pdr - pt)"),           # residual sign
    ("acc[s] = lhs < rhs", "acc[s] = lhs > rhs"),                                   # accept test flipped
    ("lhs = u * pd_tok[idx[s], j - 1]", "lhs = u * pd_tok[idx[s], j - 1] * 0.5"),   # wrong ratio
    ("final_rows = offsets[:R] + m", "final_rows = offsets[:R] + np.maximum(m - 1, 0)"),  # off-by-one row
    ("x = tokens[idx, j - 1]", "x = tokens[idx, np.maximum(j - 2, 0)]"),             # wrong draft index
])
def test_verify_mutations_are_caught(old, new):
    mod = _mutant("verify", old, new)
    assert min(_lossless_pvalues(mod.verify)) < 1e-6


@pytest.mark.parametrize("old,new", [
    ("e = W1[x_prev]  ", "e = W1[(x_prev + 1) % V]  "),                      # wrong previous token
    ("logits = U[:, k - 1] + e @ W2", "logits = U[:, k - 1] - e @ W2"),      # wrong bias sign
    ("y = logits[s] / temp[s][:, None]", "y = logits[s] * temp[s][:, None]"),  # temperature inverted
])
def test_draft_mutations_are_caught(old, new):
    # the closed-form pin of the draft sampler: with U = 0, r = V, W1 = I and
    # W2 = log P the head is a Markov chain with transition matrix P, so
    # (x_1, x_2) given the anchor has law P^(1/T)[x0, a] P^(1/T)[a, b] (rows renormalised)
    mod = _mutant("draft", old, new)
    V, R, G, x0, T = 5, 100_000, 2, 3, 0.5
    P = np.random.default_rng(11).dirichlet(np.full(V, 0.8), size=V)
    out = mod.draft(np.zeros((R, G, V)), np.eye(V), np.log(P), np.zeros((R, G, 1)), np.zeros(1 + V),
                    np.full(R, x0), np.full(R, T), 7, np.arange(R), keep_pd=False)
    PT = P ** (1.0 / T)
    PT /= PT.sum(axis=1, keepdims=True)
    expect = np.outer(PT[x0], np.ones(V)) * PT
    obs = np.bincount(out["tokens"][:, 0] * V + out["tokens"][:, 1], minlength=V * V)
    assert stats.chisquare(obs, expect.ravel() * R).pvalue < 1e-6


@pytest.mark.parametrize("old,new", [
    ("cap = prefix_schedule(a_prev, sps, MODE_GREEDY, early_stop=False)",
     "cap = prefix_schedule(a_prev, sps, MODE_GREEDY, early_stop=True)"),       # capacity with the early stop
    ("cap = prefix_schedule(a_prev, sps, MODE_GREEDY, early_stop=False)",
     "cap = prefix_schedule(a_now, sps, MODE_GREEDY, early_stop=False)"),       # capacity from the current step
    ("n_admit = min(K, rr.size)", "n_admit = min(K + 1, rr.size)"),            # one admission too many
])
def test_async_scheduler_mutations_are_caught(old, new):
    # the brute-force and appendix pins of the asynchronous scheduler reject each
    mod = _mutant("schedule", old, new)
    import test_oracle_schedule as T
    failed = 0
    for fn, args in [(T.test_async_appendix_a, ())] + [(T.test_async_capacity_is_the_brute_force_optimum, (s,))
                                                        for s in range(30)]:
        saved = T.S
        T.S = mod
        try:
            fn(*args)
        except AssertionError:
            failed += 1
        finally:
            T.S = saved
    assert failed > 0


def _sts_pins_hold(mod):
    """The STS-fitting pins run against a (possibly mutated) oracle module."""
    import synth
    ok = True
    # hand-worked ECEs (bin edges, weights)
    ok &= abs(mod.ece([0.125, 0.1875, 0.5, 0.5625, 0.875, 0.9375, 1.0], [0, 1, 1, 0, 1, 1, 1], 5) - 15 / 112) < 1e-15
    ok &= abs(mod.ece([0.25, 0.125, 0.5, 1.0, 0.75], [0, 1, 1, 1, 0], 4) - 19 / 40) < 1e-15
    # all accepted: the sharpest temperature everywhere
    rng = np.random.default_rng(2)
    z = (0.5 + 3 * rng.random((400, 4))).astype(np.float32)
    o = mod.sts_fit(z, np.full(400, 4, np.int32), np.array([0.5, 0.8, 1.0, 1.7, 3.0], np.float32), 10)
    ok &= list(o["grid_index"]) == [0, 0, 0, 0]
    # ties go to the first entry
    o = mod.sts_fit(np.full((50, 2), 60.0, np.float32), np.full(50, 2, np.int32),
                    np.array([2.0, 0.5, 1.0], np.float32), 15)
    ok &= list(o["grid_index"]) == [0, 0]
    # recovery of a known over-confidence
    kappa = np.array([1.5, 2.0, 1.25, 2.5])
    z, L, _ = synth.sts_heldout(200_000, 4, 8, kappa=kappa, mu0=1.5, mu_step=0.2)
    o = mod.sts_fit(z, L, synth.sts_grid(97, 0.5, 4.0), 15)
    ok &= bool(np.all(np.abs(o["sts_temp"] / kappa - 1) < 0.08))
    return bool(ok)


def test_unmutated_sts_fit_passes():
    from oracle import sts_fit
    assert _sts_pins_hold(sts_fit)


@pytest.mark.parametrize("old,new", [
    ("label = L >= k + 1", "label = L > k + 1"),                                        # label off by one
    ("p = (prev * c[:, 0]).astype(np.float32)", "p = (prev_raw * c[:, 0]).astype(np.float32)"),  # earlier positions not held at their fit
    ("np.floor(p * n_bins)", "(np.ceil(p * n_bins) - 1).clip(0)"),                      # right-closed bins
    ("return float(np.sum(np.abs(gap)) / N)", "return float(np.mean(np.abs(gap)))"),   # bins not weighted by size
    ("index[k] = int(np.argmin(table[k]))",
     "index[k] = int(n_grid - 1 - np.argmin(table[k][::-1]))"),                        # ties to the last entry
    ("gap = np.bincount(m, weights=y - p, minlength=n_bins)",
     "gap = np.bincount(m, weights=np.abs(y - p), minlength=n_bins)"),                 # per-sample instead of per-bin gap
])
def test_sts_fit_mutations_are_caught(old, new):
    assert not _sts_pins_hold(_mutant("sts_fit", old, new))


def _cap_accept_pvalues(cap_fn):
    from oracle.verify import verify
    rng = np.random.default_rng(1)
    V, G, r, R, T = 8, 3, 3, 300_000, 1.0
    tgt = rng.normal(size=(G + 1, V)) * 1.5
    U = tgt[:G] + rng.normal(size=(G, V)) * 1.2
    W1 = rng.normal(size=(V, r)) * 0.8
    W2 = rng.normal(size=(r, V)) * 0.8
    d = draft(np.broadcast_to(U, (R, G, V)), W1, W2, np.zeros((R, G, 1)), np.zeros(1 + r),
              np.full(R, 2), np.full(R, T), 5, np.arange(R))
    ell = np.full(R, G)
    fl = S.flatten(ell, np.full(R, 2), d["tokens"])
    v = verify(tgt[fl["mark_pos"]], fl["offsets"], ell, d["tokens"], d["pd"], d["pd_tok"], np.full(R, T), 5,
               np.arange(R))
    c = cap_fn(v, np.random.default_rng(9).integers(0, G + 1, R))
    pt = special.softmax(tgt / T, axis=1)
    ps = []
    for j in range(G):
        sel = c["n_out"] > j
        ps.append(stats.chisquare(np.bincount(c["out_tok"][sel, j], minlength=V), pt[j] * sel.sum()).pvalue)
    return ps


def test_unmutated_cap_accept_passes():
    from oracle.verify import cap_accept
    assert min(_cap_accept_pvalues(cap_accept)) > 1e-4


@pytest.mark.parametrize("old,new", [
    # the window's last slot takes the full output's final token (a later correction or bonus)
    ("out = np.where(np.arange(G1)[None, :] < n_out[:, None], v[\"out_tok\"], -1)",
     "out = np.where(np.arange(G1)[None, :] < n_out[:, None], v[\"out_tok\"], -1)\n"
     "    out[np.arange(m.size), n_out - 1] = v[\"out_tok\"][np.arange(m.size), m]"),
])
def test_cap_accept_mutations_are_caught(old, new):
    mod = _mutant("verify", old, new)
    assert min(_cap_accept_pvalues(mod.cap_accept)) < 1e-6


def _rnn_pins_hold(mod):
    """The RNN-head pins (tests/test_oracle_rnn_head.py) run against a draft module."""
    import test_oracle_rnn_head as P
    saved = P.draft
    P.draft = mod.draft
    try:
        P.test_embedding_only_output_is_a_markov_head(1.0)
        P.test_hidden_only_output_is_a_token_independent_softmax()
        P.test_open_gate_keeps_the_zero_state()
        P.test_closed_gate_holds_the_previous_embedding()
        P.test_half_open_gate_remembers_two_tokens_back()
        return True
    except AssertionError:
        return False
    finally:
        P.draft = saved


def test_unmutated_rnn_head_passes():
    import oracle.draft as D
    assert _rnn_pins_hold(D)


@pytest.mark.parametrize("old,new", [
    ("state = gate * state + (1.0 - gate) * cand", "state = (1.0 - gate) * state + gate * cand"),  # gate inverted
    ("zk = np.concatenate([state, e, h[:, k - 1]], axis=1)",
     "zk = np.concatenate([np.zeros_like(state), e, h[:, k - 1]], axis=1)"),                   # state not carried
    ("e = np.tanh(pre[:, 2 * r:])", "e = np.tanh(pre[:, r:2 * r])"),                          # output from the candidate rows
    ("gate = 1.0 / (1.0 + np.exp(-pre[:, :r]))", "gate = 1.0 / (1.0 + np.exp(pre[:, :r]))"),  # gate sign
])
def test_rnn_head_mutations_are_caught(old, new):
    assert not _rnn_pins_hold(_mutant("draft", old, new))


def _rejection_residual_pvalue(mod):
    import test_oracle_verify as P
    counts, n, pt, pd_row = P._residual_counts(mod.verify, 9, 60_000, 4, residual="rejection")
    q = np.maximum(0.0, pt - pd_row)
    q /= q.sum()
    pos = q > 0
    return stats.chisquare(counts[pos], q[pos] * counts[pos].sum()).pvalue if counts[~pos].sum() == 0 else 0.0


def test_unmutated_rejection_residual_passes():
    import oracle.verify as Vm
    assert _rejection_residual_pvalue(Vm) > 1e-4


@pytest.mark.parametrize("old,new", [
    ("v, mg = inverse_cdf(pt[pend], u)", "v, mg = inverse_cdf(pdr[pend], u)"),          # proposals from the draft
    ("acc = lhs < rhs", "acc = lhs > rhs"),                                               # acceptance inverted
    ("lhs, rhs = w * pt[pend, v], pt[pend, v] - pdr[pend, v]",
     "lhs, rhs = w * pt[pend, v], pt[pend, v]"),                                          # p_d left out of the test
])
def test_rejection_residual_mutations_are_caught(old, new):
    assert _rejection_residual_pvalue(_mutant("verify", old, new)) < 1e-6
