"""Markov-head draft sampler and confidence head in fp64 — test infrastructure only.

[DSpark] 方法细节, "序列阶段的依赖注入": the sequential stage induces the causal
block distribution
    p_k(v | x0, x<k) = exp(U_k(v) + B_k(v)) / sum_u exp(U_k(u) + B_k(u)),
sampled left to right, x0 being the anchor (the previous round's bonus token).
[DSpark] 方法细节, "马尔可夫头（Markov head）的实现": the Markov head restricts
B_k to the previous token through a rank-r factorisation,
    B(x_{k-1}, .) = W1[x_{k-1}] W2,  W1 in R^{V x r}, W2 in R^{r x V}.
[DSpark] 方法细节, "置信度头的设计": c_k = sigmoid(w^T [h_k; W1[x_{k-1}]]).
[DSpark] 方法细节, "RNN头的实现" (the optional head): a recurrent state s_k
(s_0 = 0) carries the block's whole prefix.  With z_k = [s_{k-1}; W1[x_{k-1}];
h_k] in R^{2r+H} and one linear map split into gate, candidate and output parts
W_g, W_c, W_o in R^{r x (2r+H)}:
    s_k = sigmoid(W_g z_k) * s_{k-1} + (1 - sigmoid(W_g z_k)) * tanh(W_c z_k),
    B_k(x_{<k}, .) = W2^T tanh(W_o z_k),
i.e. the Markov head's row W1[x_{k-1}] is replaced by tanh(W_o z_k).
[DSpark] 方法细节, "并行阶段的局限与设计": the anchor is the first predicted
position, so gamma backbone inputs give gamma base-logit rows U_1..U_gamma.
[DeepSpec analysis] §2.2 (DFlash): markov_rank = 0 turns the head into a zero
matrix, i.e. plain parallel drafting.

Readings where the pages are silent:
* temperature T_r per request: p_k = softmax((U_k + B_k) / T_r); T_r <= 0 (or
  NaN) means greedy: x_k = argmax with ties to the lowest token id and p_d^k is
  one-hot at x_k;
* the confidence weight splits as w = [w_h (H entries); w_e (r entries)], no bias;
* the draft draw at position k uses Philox uniform (seed, req_id, k, draw 0),
  positions counted from 1;
* sampling is inverse CDF in token-id order (see `oracle.sampling`);
* RNN head: the map is one [3r, 2r+H] matrix, rows W_g, then W_c, then W_o;
  the confidence head keeps its definition (w_e . W1[x_{k-1}]); the row
  tanh(W_o z_k) enters the bias product in that product's operand precision
  (rnn_row_dtype "bf16" or "f32", as the Markov head's W1 rows do; None keeps
  fp64), i.e. it is rounded to nearest-even in that format.
"""
import numpy as np

from .philox import uniform, DRAW_DRAFT
from .sampling import inverse_cdf, argmax_first


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def round_to(x, fmt):
    """Round fp64 values to nearest-even in fp32 or bfloat16 (bf16 through fp32,
    which is how a kernel holding the fp32 value rounds it)."""
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    if fmt == "f32":
        return x32.astype(np.float64)
    assert fmt == "bf16"
    b = x32.view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def draft(U, W1, W2, h, w, anchor, temp, seed, req_id, keep_pd=True, W_rnn=None, rnn_row_dtype=None):
    """Run the draft sampler for R requests.

    U [R, g, V], W1 [V, r], W2 [r, V], h [R, g, H], w [H + r]: real arrays (any
    float dtype; read as fp64).  anchor [R] int, temp [R] float, req_id [R] int,
    seed int.  W_rnn [3r, 2r + H] selects the RNN head (None: Markov head);
    rnn_row_dtype ("bf16", "f32" or None) is the precision its rows take.

    Returns a dict:
      tokens [R, g] int64        sampled / greedy draft tokens x_1..x_g
      pd [R, g, V] fp64          draft probability rows (None unless keep_pd)
      pd_tok [R, g] fp64         p_d^k(x_k)
      conf_logit [R, g] fp64     z_k = w_h . h_k + w_e . W1[x_{k-1}]
      conf [R, g] fp64           c_k = sigmoid(z_k)
      margin [R, g] fp64         sampled rows: CDF margin of the draw;
                                 greedy rows: top-2 logit gap / max(1, |l_max|)
      greedy [R] bool
    """
    U = _f64(U)
    W1 = _f64(W1)
    W2 = _f64(W2)
    h = _f64(h)
    w = _f64(w)
    R, G, V = U.shape
    H = h.shape[2]
    r = W1.shape[1]
    assert W1.shape == (V, r) and W2.shape == (r, V) and w.shape == (H + r,)
    w_h, w_e = w[:H], w[H:]
    temp = np.asarray(temp, dtype=np.float64)
    sampled = temp > 0
    req_id = np.asarray(req_id, dtype=np.int64)
    x_prev = np.asarray(anchor, dtype=np.int64).copy()
    assert ((x_prev >= 0) & (x_prev < V)).all()
    rnn = W_rnn is not None
    if rnn:
        W_rnn = _f64(W_rnn)
        assert W_rnn.shape == (3 * r, 2 * r + H)
        state = np.zeros((R, r))                    # s_0 = 0

    tokens = np.zeros((R, G), np.int64)
    pd = np.zeros((R, G, V), np.float64) if keep_pd else None
    pd_tok = np.zeros((R, G))
    zl = np.zeros((R, G))
    margin = np.zeros((R, G))
    rows = np.arange(R)
    for k in range(1, G + 1):
        e = W1[x_prev]                              # W1[x_{k-1}]      [R, r]
        zl[:, k - 1] = h[:, k - 1] @ w_h + e @ w_e  # confidence logit
        if rnn:
            zk = np.concatenate([state, e, h[:, k - 1]], axis=1)   # [s_{k-1}; W1[x_{k-1}]; h_k]
            pre = zk @ W_rnn.T
            gate = 1.0 / (1.0 + np.exp(-pre[:, :r]))
            cand = np.tanh(pre[:, r:2 * r])
            e = np.tanh(pre[:, 2 * r:])             # tanh(W_o z_k) takes the place of W1[x_{k-1}]
            if rnn_row_dtype is not None:
                e = round_to(e, rnn_row_dtype)
            state = gate * state + (1.0 - gate) * cand
        logits = U[:, k - 1] + e @ W2               # U_k + B_k
        p = np.zeros((R, V))
        x = np.zeros(R, np.int64)
        if sampled.any():
            s = sampled
            y = logits[s] / temp[s][:, None]
            y = y - y.max(axis=1, keepdims=True)
            ey = np.exp(y)
            ps = ey / ey.sum(axis=1, keepdims=True)
            u = uniform(seed, req_id[s], k, DRAW_DRAFT)
            xs, ms = inverse_cdf(ps, u)
            p[s] = ps
            x[s] = xs
            margin[s, k - 1] = ms
        if (~sampled).any():
            gmask = ~sampled
            lg = logits[gmask]
            xg, gap = argmax_first(lg)
            x[gmask] = xg
            p[np.flatnonzero(gmask), xg] = 1.0
            margin[gmask, k - 1] = gap / np.maximum(1.0, np.abs(lg.max(axis=1)))
        tokens[:, k - 1] = x
        pd_tok[:, k - 1] = p[rows, x]
        if keep_pd:
            pd[:, k - 1] = p
        x_prev = x
    conf = 1.0 / (1.0 + np.exp(-zl))
    return dict(tokens=tokens, pd=pd, pd_tok=pd_tok, conf_logit=zl, conf=conf,
                margin=margin, greedy=~sampled)


def draft_row_distribution(U_k, W1, W2, x_prev, T):
    """p_d^k for one request and one position, given the previous token (fp64).

    Used by the statistical pins to state the conditional distribution of
    x_k given x_{k-1}."""
    logits = _f64(U_k) + _f64(W1)[int(x_prev)] @ _f64(W2)
    if T > 0:
        y = logits / T
        ey = np.exp(y - y.max())
        return ey / ey.sum()
    p = np.zeros_like(logits)
    p[int(np.argmax(logits))] = 1.0
    return p
