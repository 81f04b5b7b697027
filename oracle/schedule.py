"""Sequential Temperature Scaling, the hardware-aware prefix scheduler and the
flattened verify batch — test infrastructure only.

[DSpark] 方法细节, "事后校准（Post-hoc Calibration）": STS applies one
temperature per draft position to the confidence; temperature scaling keeps the
order of the scores.  The formula is not printed; reading: standard temperature
scaling of the pre-sigmoid logit, c'_k = sigmoid(z_k / tau_k) (tau_k = 1 is the
identity).

[DSpark] 方法细节, "硬件感知前缀调度器": survival a_{r,j} = prod_{i<=j} c_{r,i};
verify batch size B = sum_r (1 + l_r); expected accepted tokens
tau = sum_r (1 + sum_{j<=l_r} a_{r,j}); objective Theta = tau * SPS(B).

[DSpark] 方法细节, "贪心求解与因果性保证", Algorithm 1: candidates
E = {(r, j) : a_{r,j} > 0} sorted by a descending; start from l_r = 0,
B = R, tau = R, Theta_best = R * SPS(R); admit candidates in order, updating B,
tau and Theta; keep the admission while Theta > Theta_best, stop at the first
candidate with Theta <= Theta_best.

[DSpark] 附录, "无早停机制导致的选择偏差反例": the counterexample for a
search without the early stop (used as a pin in the tests).

[DSpark] 补充细节, "高吞吐量与低延迟推理": the kept tokens of all requests are
flattened into one batch and a marker tensor carries the intra-sequence
dependency.

[DSpark] 补充细节, "生产环境中的硬件感知前缀调度器" (and the engineering
compromise of section 4.2.5 / 8.5 of the MTP survey page): in production the
scheduler runs asynchronously.  The confidences of two steps earlier fix the
verify capacity K by a global search over their sorted path (no early stop,
because the real SPS curve steps down in cliffs); the current step still ranks
its candidates by their current cumulative confidence and admits the top K.
K depends only on the earlier information, which is the causal barrier that
keeps the search lossless.

Readings where the pages are silent (this library's contract):
* asynchronous mode: the earlier confidences are given as a [R, g] array for
  the current batch's requests (the caller maps its history onto them); K is the
  number of admissions of the best prefix of their sorted path (the first
  maximum of Theta_i, i = 0 .. n_prev); the current step admits its first
  min(K, n_now) candidates in the usual order; theta_best reports Theta of that
  admission with the current survivals;
* c'_k is the fp32 rounding of sigmoid(z/tau) evaluated in fp64, and a_{r,j} is
  the left-to-right fp32 product of the c'; both are sort keys, so both sides
  must produce the same bits;
* ties in a are broken by request index, then position (ascending), which
  keeps every request's kept set a prefix;
* tau and Theta are accumulated in fp64, in sorted order;
* the SPS table is given per total verify-token count n (entries 0..R(1+g));
* "scheduler off" verifies every draft token (l_r = g);
* flattened layout: request-major rows, position ascending, row (r, 0) is the
  anchor and row (r, j) the draft token x_j; marker = (request, position).
"""
import numpy as np

MODE_OFF = 0
MODE_GREEDY = 1
MODE_ASYNC_TOPK = 2


def sts_calibrate(conf_logit, sts_temp):
    """c' = fp32(sigmoid(z / tau)) with the sigmoid evaluated in fp64.

    conf_logit [R, g] fp32 values, sts_temp [g] fp32 values.
    Returns (c [R, g] float32, margin [R, g] fp64): margin is the relative
    distance of the fp64 sigmoid to the nearest fp32 rounding midpoint."""
    z = np.asarray(conf_logit, dtype=np.float32).astype(np.float64)
    tau = np.asarray(sts_temp, dtype=np.float32).astype(np.float64)
    t = z / tau[None, :]
    with np.errstate(over="ignore"):
        s = 1.0 / (1.0 + np.exp(-t))
    c = s.astype(np.float32)
    up = np.nextafter(c, np.float32(np.inf)).astype(np.float64)
    dn = np.nextafter(c, np.float32(0)).astype(np.float64)
    cd = c.astype(np.float64)
    mid_up = 0.5 * (cd + up)
    mid_dn = 0.5 * (cd + dn)
    dist = np.minimum(np.abs(s - mid_up), np.abs(s - mid_dn))
    with np.errstate(divide="ignore", invalid="ignore"):
        margin = np.where(s > 0, dist / s, np.inf)
    return c, margin


def survival(c):
    """a_{r,j} = c_{r,1} * ... * c_{r,j}, left to right in fp32.  c [R, g] float32."""
    c = np.asarray(c, dtype=np.float32)
    a = np.empty_like(c)
    run = np.ones(c.shape[0], dtype=np.float32)
    for j in range(c.shape[1]):
        run = (run * c[:, j]).astype(np.float32)
        a[:, j] = run
    return a


def sorted_candidates(a):
    """E = {(r, j): a > 0} in admission order (a desc, r asc, j asc).

    Returns (r_idx, j_idx) int64 arrays; j is 0-based (paper position j+1)."""
    a = np.asarray(a, dtype=np.float32)
    R, G = a.shape
    rr, jj = np.nonzero(a > 0)
    vals = a[rr, jj].astype(np.float64)
    order = np.lexsort((jj, rr, -vals))
    return rr[order], jj[order]


def prefix_schedule(a, sps, mode=MODE_GREEDY, early_stop=True):
    """Algorithm 1 on survival products a [R, g] (fp32) and the SPS table.

    mode MODE_OFF returns l_r = g for every request (the "static" full-block
    verify) with theta_best = 0.
    With early_stop=False the search walks the whole sorted list and returns
    the best prefix of it (the search the appendix warns about).

    Returns dict(ell [R] int64, theta_best fp64, n_admit int, thetas list
    (Theta_0, Theta_1, ... as evaluated), theta_margin fp64 = smallest relative
    gap |Theta_i - Theta_best| / Theta_i over the comparisons made)."""
    a = np.asarray(a, dtype=np.float32)
    sps = np.asarray(sps, dtype=np.float64)
    R, G = a.shape
    if mode == MODE_OFF:
        return dict(ell=np.full(R, G, np.int64), theta_best=0.0, n_admit=R * G,
                    thetas=[], theta_margin=np.inf)
    rr, jj = sorted_candidates(a)
    B = R
    tau = float(R)
    theta_best = R * sps[R]
    thetas = [theta_best]
    ell = np.zeros(R, np.int64)
    best_ell = ell.copy()
    n_admit = 0
    best_n = 0
    margin = np.inf
    for i, (r, j) in enumerate(zip(rr, jj)):
        ell[r] = j + 1
        B += 1
        tau += float(a[r, j])
        theta = tau * sps[B]
        thetas.append(theta)
        margin = min(margin, abs(theta - theta_best) / max(abs(theta), abs(theta_best)))
        if theta > theta_best:
            theta_best = theta
            best_ell = ell.copy()
            best_n = i + 1
        elif early_stop:
            break
    n_admit = best_n
    return dict(ell=best_ell, theta_best=theta_best, n_admit=n_admit, thetas=thetas,
                theta_margin=margin)


def async_topk_schedule(a_now, a_prev, sps):
    """The production variant: capacity K from a_prev, top-K admission of a_now.

    a_now, a_prev [R, g] fp32 survival products; sps the SPS table.
    Returns dict(ell [R] int64, theta_best fp64 (Theta of the admission with the
    current survivals), n_admit int, K int, cap_theta fp64 (Theta_K on the
    earlier path), cap_margin fp64 = relative gap between Theta_K and the best
    Theta at any other prefix length of the earlier path (inf if there is no
    other), thetas (Theta_0 .. Theta_{n_prev} of the earlier path))."""
    a_now = np.asarray(a_now, dtype=np.float32)
    sps = np.asarray(sps, dtype=np.float64)
    R, G = a_now.shape
    cap = prefix_schedule(a_prev, sps, MODE_GREEDY, early_stop=False)
    K = cap["n_admit"]
    th = np.asarray(cap["thetas"], dtype=np.float64)
    others = np.delete(th, K)
    cap_margin = (float(np.min(np.abs(th[K] - others)) / abs(th[K])) if others.size else np.inf)
    rr, jj = sorted_candidates(a_now)
    n_admit = min(K, rr.size)
    ell = np.zeros(R, np.int64)
    tau = float(R)
    for i in range(n_admit):
        r, j = rr[i], jj[i]
        ell[r] = max(ell[r], j + 1)
        tau += float(a_now[r, j])
    return dict(ell=ell, theta_best=tau * sps[R + n_admit], n_admit=n_admit, K=K, cap_theta=float(th[K]),
                cap_margin=cap_margin, thetas=list(th), theta_margin=np.inf)


def flatten(ell, anchor, tokens):
    """Flattened verify batch and marker tensor.

    Returns dict(offsets [R+1], flat_tok [N], mark_req [N], mark_pos [N]) as
    int64; N = sum_r (1 + l_r)."""
    ell = np.asarray(ell, dtype=np.int64)
    anchor = np.asarray(anchor, dtype=np.int64)
    tokens = np.asarray(tokens, dtype=np.int64)
    R = ell.shape[0]
    offsets = np.zeros(R + 1, np.int64)
    offsets[1:] = np.cumsum(1 + ell)
    N = int(offsets[-1])
    flat_tok = np.zeros(N, np.int64)
    mark_req = np.zeros(N, np.int64)
    mark_pos = np.zeros(N, np.int64)
    for r in range(R):
        o = offsets[r]
        L = ell[r]
        flat_tok[o] = anchor[r]
        flat_tok[o + 1:o + 1 + L] = tokens[r, :L]
        mark_req[o:o + 1 + L] = r
        mark_pos[o:o + 1 + L] = np.arange(L + 1)
    return dict(offsets=offsets, flat_tok=flat_tok, mark_req=mark_req, mark_pos=mark_pos)


def schedule(conf_logit, sts_temp, sps, anchor, tokens, mode=MODE_GREEDY, early_stop=True, conf_logit_prev=None):
    """STS -> survival -> Algorithm 1 (or the asynchronous top-K variant, which
    takes the earlier confidences conf_logit_prev) -> flatten, as one call.

    Returns the union of the dicts above plus c (calibrated, fp32), a (fp32) and
    sts_margin (smallest rounding margin of c over the batch, and of the earlier
    confidences in the asynchronous mode)."""
    c, m = sts_calibrate(conf_logit, sts_temp)
    a = survival(c)
    if mode == MODE_ASYNC_TOPK:
        c_prev, m_prev = sts_calibrate(conf_logit_prev, sts_temp)
        res = async_topk_schedule(a, survival(c_prev), sps)
        m = np.minimum(m, m_prev)
    else:
        res = prefix_schedule(a, sps, mode, early_stop)
    res.update(flatten(res["ell"], anchor, tokens))
    res["c"] = c
    res["a"] = a
    res["sts_margin"] = float(m.min()) if m.size else np.inf
    return res


def pack_rows(target, mark_req, mark_pos, n_rows=None):
    """The packed verify batch ([DSpark] 补充细节, "高吞吐量与低延迟推理": the
    variable-length prefixes are flattened into one buffer; the SGLang notes
    pack the ragged requests into a compact buffer before the target forward):
    row i is target[mark_req[i], mark_pos[i]] for i < n_rows.

    target [R, g+1, V]; mark_req, mark_pos [>= n_rows] int.  Returns [n_rows, V]."""
    target = np.asarray(target)
    n = len(mark_req) if n_rows is None else int(n_rows)
    req = np.asarray(mark_req, dtype=np.int64)[:n]
    pos = np.asarray(mark_pos, dtype=np.int64)[:n]
    return target[req, pos]
