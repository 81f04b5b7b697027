"""Lossless rejection-sampling verification in fp64 — test infrastructure only.

[DSpark] 背景知识与设计原则, "投机解码的延迟建模": at draft position k the
target distribution p_t^k is compared with the draft distribution p_d^k and x_k
is accepted with probability min(1, p_t^k(x_k) / p_d^k(x_k)); verification runs
left to right and the first rejection discards every later token.
[MTP Survey] §2.2 "拒绝采样（Rejection Sampling）：无损校验的数学": at the
rejecting position a correction token is drawn from
q^k = norm(max(0, p_t^k - p_d^k)); when every draft token is accepted one bonus
token comes from the target; at temperature 0 the rule degenerates to "accept
iff x_k = argmax p_t^k, else emit that argmax".

Readings where the pages are silent (this library's contract):
* verify rows: request r's rows in the flattened batch are [x0, x_1..x_l]; row
  j (0-based) holds the target logits that give p_t^{j+1}.  All l accepted ->
  the bonus comes from row l, i.e. p_t^{l+1} (the only reading consistent with
  1 + l rows per request);
* p_t = softmax(z / T_r) with the request's temperature T_r (same as the
  draft's); T_r <= 0 means greedy, argmax ties to the lowest token id;
* accept test: u * p_d(x) < p_t(x) with u = Philox(seed, req, j, draw 1), which
  equals u < min(1, p_t/p_d) for u in [0, 1); decision margin
  |u p_d - p_t| / max(u p_d, p_t);
* residual: draw 2 at the rejecting position, inverse CDF of
  max(0, p_t - p_d) / sum; if that sum is 0 in the implementation's arithmetic
  (reachable only through rounding), sample p_t instead;
* bonus: draw 3 at position l + 1, inverse CDF of p_t^{l+1}.
* residual by rejection (residual="rejection", the p_d-row-free mode): the
  same distribution norm(max(0, p_t - p_d)) sampled by rejection from p_t.
  Trial t proposes v = InvCDF(p_t, u) with u from draw 2, trial t, and accepts
  it iff w p_t(v) < p_t(v) - p_d(v) with w from draw 4, trial t, i.e. with
  probability max(0, 1 - p_d(v)/p_t(v)); the accepted v is a sample of the
  residual, so only p_d at the proposed tokens is needed.  After max_trials
  rejected proposals the residual is sampled by inverse CDF with u from draw
  2, trial max_trials (max_trials = 0 is the inverse-CDF rule above).
"""
import numpy as np

from .philox import uniform, DRAW_ACCEPT, DRAW_RESIDUAL, DRAW_BONUS, DRAW_RESID_ACCEPT

MAX_TRIALS = 256  # residual proposals before the inverse-CDF fallback
from .sampling import inverse_cdf, argmax_first


def _softmax_rows(z, T):
    y = z / T[:, None]
    ey = np.exp(y - y.max(axis=1, keepdims=True))
    return ey / ey.sum(axis=1, keepdims=True)


def _residual_by_rejection(pt, pdr, seed, req, j, max_trials):
    """Rejecting requests: (tokens, margins, fell_back) of the residual drawn by
    rejection from p_t (see the module notes), trial by trial over the requests
    still pending.  pt, pdr [n, V] fp64; req, j [n] int."""
    n = pt.shape[0]
    tok = np.full(n, -1, np.int64)
    margin = np.full(n, np.inf)
    pend = np.arange(n)
    for t in range(max_trials):
        if pend.size == 0:
            break
        u = uniform(seed, req[pend], j[pend], DRAW_RESIDUAL, t)
        v, mg = inverse_cdf(pt[pend], u)
        margin[pend] = np.minimum(margin[pend], mg)
        w = uniform(seed, req[pend], j[pend], DRAW_RESID_ACCEPT, t)
        lhs, rhs = w * pt[pend, v], pt[pend, v] - pdr[pend, v]
        margin[pend] = np.minimum(margin[pend], np.abs(lhs - rhs) / np.maximum(pt[pend, v], 1e-300))
        acc = lhs < rhs
        tok[pend[acc]] = v[acc]
        pend = pend[~acc]
    fell = np.zeros(n, bool)
    if pend.size:
        q = np.maximum(0.0, pt[pend] - pdr[pend])
        Q = q.sum(axis=1)
        zero = ~(Q > 0)
        q = np.where(zero[:, None], pt[pend], q / np.where(zero, 1.0, Q)[:, None])
        u = uniform(seed, req[pend], j[pend], DRAW_RESIDUAL, max_trials)
        v, mg = inverse_cdf(q, u)
        tok[pend] = v
        margin[pend] = np.minimum(margin[pend], mg)
        fell[pend] = True
    return tok, margin, fell


def verify(target_rows, offsets, ell, tokens, pd_rows, pd_tok, temp, seed, req_id, residual="inverse_cdf",
           max_trials=MAX_TRIALS):
    """Verify R requests.

    target_rows [N, V] (row offsets[r] + j -> p_t^{j+1} of request r),
    offsets [R+1], ell [R], tokens [R, g], pd_tok [R, g], temp [R], req_id [R];
    pd_rows: [R, g, V] array or a callable (r, k0) -> row of p_d^{k0+1}.

    residual: "inverse_cdf" or "rejection" (see the module notes).

    Returns dict(n_accept [R], out_tok [R, g+1] (-1 after the emitted tokens),
    n_out [R], accept_margin [R] (smallest accept-test margin met before the
    last decision; inf if none), sample_margin [R] (CDF margin of the final
    draw, or the smallest margin of any proposal and acceptance decision of a
    rejection-sampled residual; inf for greedy rows), residual_fallback [R]
    bool (inverse-CDF rule: zero residual mass; rejection: no proposal
    accepted))."""
    offsets = np.asarray(offsets, dtype=np.int64)
    ell = np.asarray(ell, dtype=np.int64)
    tokens = np.asarray(tokens, dtype=np.int64)
    pd_tok = np.asarray(pd_tok, dtype=np.float64)
    temp = np.asarray(temp, dtype=np.float64)
    req_id = np.asarray(req_id, dtype=np.int64)
    R, G = tokens.shape
    sampled = temp > 0
    get_pd = pd_rows if callable(pd_rows) else None

    m = np.zeros(R, np.int64)
    alive = np.ones(R, bool)  # no rejection seen yet
    acc_margin = np.full(R, np.inf)
    for j in range(1, G + 1):
        act = alive & (ell >= j)
        if not act.any():
            break
        idx = np.flatnonzero(act)
        z = np.asarray(target_rows[offsets[idx] + j - 1], dtype=np.float64)
        x = tokens[idx, j - 1]
        acc = np.zeros(idx.size, bool)
        s = sampled[idx]
        if s.any():
            pt = _softmax_rows(z[s], temp[idx[s]])
            u = uniform(seed, req_id[idx[s]], j, DRAW_ACCEPT)
            lhs = u * pd_tok[idx[s], j - 1]
            rhs = pt[np.arange(pt.shape[0]), x[s]]
            acc[s] = lhs < rhs
            mg = np.abs(lhs - rhs) / np.maximum(np.maximum(lhs, rhs), 1e-300)
            acc_margin[idx[s]] = np.minimum(acc_margin[idx[s]], mg)
        if (~s).any():
            am, _ = argmax_first(z[~s])
            acc[~s] = x[~s] == am
        m[idx[acc]] += 1
        alive[idx[~acc]] = False

    # final token: row m of each request (the rejecting row, or row l = m for the bonus)
    out_tok = np.full((R, G + 1), -1, np.int64)
    out_tok[:, :G] = np.where(np.arange(G)[None, :] < m[:, None], tokens, -1)
    sample_margin = np.full(R, np.inf)
    fallback = np.zeros(R, bool)
    rejected = m < ell
    final_rows = offsets[:R] + m
    g = np.flatnonzero(~sampled)
    if g.size:
        am, _ = argmax_first(np.asarray(target_rows[final_rows[g]], dtype=np.float64))
        out_tok[g, m[g]] = am
    for idx, is_rej in ((np.flatnonzero(sampled & rejected), True),
                        (np.flatnonzero(sampled & ~rejected), False)):
        if idx.size == 0:
            continue
        z = np.asarray(target_rows[final_rows[idx]], dtype=np.float64)
        pt = _softmax_rows(z, temp[idx])
        if is_rej and residual == "rejection":
            pdr = np.stack([get_pd(int(r), int(m[r])) for r in idx]) if callable(pd_rows) \
                else np.asarray(pd_rows[idx, m[idx]], dtype=np.float64)
            x, mg, fb = _residual_by_rejection(pt, pdr, seed, req_id[idx], m[idx] + 1, max_trials)
            out_tok[idx, m[idx]] = x
            sample_margin[idx] = mg
            fallback[idx] = fb
            continue
        if is_rej:
            pdr = np.stack([get_pd(int(r), int(m[r])) for r in idx]) if callable(pd_rows) \
                else np.asarray(pd_rows[idx, m[idx]], dtype=np.float64)
            q = np.maximum(0.0, pt - pdr)
            Q = q.sum(axis=1)
            zero = ~(Q > 0)
            q = np.where(zero[:, None], pt, q / np.where(zero, 1.0, Q)[:, None])
            fallback[idx] = zero
            u = uniform(seed, req_id[idx], m[idx] + 1, DRAW_RESIDUAL)
        else:
            q = pt
            u = uniform(seed, req_id[idx], ell[idx] + 1, DRAW_BONUS)
        x, mg = inverse_cdf(q, u)
        out_tok[idx, m[idx]] = x
        sample_margin[idx] = mg
    return dict(n_accept=m, out_tok=out_tok, n_out=m + 1, accept_margin=acc_margin,
                sample_margin=sample_margin, residual_fallback=fallback)


def cap_accept(v, cap):
    """Cap-accept verification ([MTP Survey] §8, the SGLang integration notes:
    three verify modes, static (full block), compact (truncated by the
    scheduler) and cap-accept: the full block is verified but only the
    scheduled window is committed, to observe the upper bound).

    Reading: with m draft tokens accepted by the full-block verification `v`
    (the output of verify() with every l_r = gamma) and a window of cap_r
    tokens, the engine commits the first min(m, cap_r) + 1 emitted tokens.
    When m > cap_r the last committed token is the accepted draft token
    x_{cap_r + 1}, itself a sample of p_t^{cap_r + 1} given the prefix, so the
    commit is lossless like compact verification; n_accept keeps the
    full-block count m as the observation.

    Returns dict(n_accept [R] (m), n_out [R] (committed tokens),
    out_tok [R, g+1] (committed tokens, then -1))."""
    m = np.asarray(v["n_accept"], dtype=np.int64)
    G1 = v["out_tok"].shape[1]
    cap = np.clip(np.asarray(cap, dtype=np.int64), 0, G1 - 1)
    n_out = np.minimum(m, cap) + 1
    out = np.where(np.arange(G1)[None, :] < n_out[:, None], v["out_tok"], -1)
    return dict(n_accept=m, n_out=n_out, out_tok=out)
