"""One full step through the three C-ABI calls on the GPU (draft -> schedule ->
target stand-in -> verify), compared with the oracle's own step on the same
inputs.  Where a draw is exempted (margin below the contract), every output that
depends on it is left out of the comparison; the tests bound how often that
happens."""
import numpy as np
import pytest
import torch

import synth
from oracle.draft import draft as oracle_draft
from oracle import schedule as S
from oracle.verify import verify as oracle_verify
from parity import MARGIN, compare_draft, compare_verify, gpu_np, np_inputs, rtol_for, to_np64
from gpu_common import check_no_error, gather_target_rows, gpu_draft, require_gpu
from draft_sampling_lossless_markov_gb300 import torch_api as T

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def gpu_step(inp, ws=None):
    d, ws = gpu_draft(inp, ws)
    sch = T.schedule(ws, d["conf_logit"], inp["sts"], inp["sps"], inp["anchor"], d["tokens"], inp["sched"])
    torch.cuda.synchronize()
    n = int(sch["n_verify"][0])
    rows = gather_target_rows(inp["target"], sch["mark_req"], sch["mark_pos"], n)
    v = T.verify(ws, rows, sch["offsets"], sch["ell"], d["tokens"], d["pd_rows"], d["pd_tok"], inp["temp"],
                 inp["req_id"], inp["seed"])
    torch.cuda.synchronize()
    check_no_error(ws)
    return d, sch, v


def oracle_step(inp, idx=None):
    ni = np_inputs(inp, idx)
    d = oracle_draft(**ni)
    wl_sps = inp["sps"]
    sts = inp["sts"].cpu().numpy()
    sch = S.schedule(d["conf_logit"].astype(np.float32), sts, wl_sps, ni["anchor"], d["tokens"],
                     mode=inp["sched"])
    tgt = inp["target"] if idx is None else inp["target"].index_select(0, idx)
    rows = to_np64(tgt[torch.from_numpy(sch["mark_req"]).to(tgt.device),
                       torch.from_numpy(sch["mark_pos"]).to(tgt.device)])
    v = oracle_verify(rows, sch["offsets"], sch["ell"], d["tokens"], d["pd"], d["pd_tok"], ni["temp"],
                      ni["seed"], ni["req_id"])
    return d, sch, v


def _cut_gap(osch):
    # relative gap between the last admitted and the first rejected survival value
    rr, jj = S.sorted_candidates(osch["a"])
    n = osch["n_admit"]
    vals = osch["a"][rr, jj].astype(np.float64)
    if n == 0 or n >= len(vals):
        return np.inf
    return (vals[n - 1] - vals[n]) / vals[n - 1]


def test_tiny_step_end_to_end():
    wl = synth.WORKLOADS["tiny"]
    full = 0
    for seed in range(24):
        inp = synth.make_inputs(wl, "cuda", seed=seed)
        d, sch, v = gpu_step(inp)
        od, osch, ov = oracle_step(inp)
        st = compare_draft(gpu_np(d), od, rtol_for(wl.dtype))
        if st["n_exempt_requests"]:
            continue  # a draw inside the margin changes the scheduler's inputs downstream
        g_s = gpu_np(sch)
        # the scheduler runs on each side's own confidences (fp32 on the GPU, fp64
        # rounded to fp32 in the oracle), which may differ in the last bits: compare
        # only when no decision lies within that drift
        if osch["theta_margin"] < 1e-4 or _cut_gap(osch) < 1e-4:
            continue
        np.testing.assert_array_equal(g_s["ell"], osch["ell"])
        np.testing.assert_array_equal(g_s["offsets"], osch["offsets"])
        n = int(osch["offsets"][-1])
        for k in ("flat_tok", "mark_req", "mark_pos"):
            np.testing.assert_array_equal(g_s[k][:n], osch[k])
        if osch["theta_best"]:
            assert abs(g_s["theta_best"][0] - osch["theta_best"]) <= 1e-5 * osch["theta_best"]
        compare_verify(gpu_np(v), ov, ~(inp["temp"].cpu().numpy() > 0))
        full += 1
    assert full >= 8


def test_qwen3_4b_step_sampled_requests():
    # scheduler off (l = gamma): each request's verify depends on its own draft only
    wl = synth.WORKLOADS["qwen3_4b"]
    inp = synth.make_inputs(wl, "cuda")
    d, sch, v = gpu_step(inp)
    assert int(sch["n_verify"][0]) == wl.B * (wl.gamma + 1)
    subset = [0, 5, 17, 63]
    idx = torch.tensor(subset, device="cuda")
    od, osch, ov = oracle_step(inp, idx)
    g = {k: t.index_select(0, idx).cpu().numpy() for k, t in d.items()}
    st = compare_draft(g, od, rtol_for(wl.dtype))
    exempt = (od["margin"] < MARGIN).any(axis=1)
    gv = {k: t.index_select(0, idx).cpu().numpy() for k, t in v.items()}
    ok = ~exempt
    if ok.any():
        compare_verify({k: a[ok] for k, a in gv.items()}, {k: a[ok] for k, a in ov.items()},
                       np.zeros(ok.sum(), bool))
    # acceptance statistics of the whole batch: the output lengths are plausible
    n_out = v["n_out"].cpu().numpy()
    assert n_out.min() >= 1 and n_out.max() <= wl.gamma + 1


def _step_modes(inp, head, sched, verify_mode, Wr, zprev, ws=None):
    """GPU step in the requested modes, and the oracle's step in the same modes."""
    from oracle.verify import cap_accept
    B, G, V = inp["U"].shape
    if ws is None:
        from gpu_common import workspace_for
        ws = workspace_for(B, G, V, inp["W1"].shape[1], inp["h"].shape[2], inp["U"].dtype)
    d = T.draft_sample(ws, inp["U"], inp["W1"], inp["W2"], inp["h"], inp["w"], inp["anchor"], inp["temp"],
                       inp["req_id"], inp["seed"], W_rnn=Wr if head == "rnn" else None)
    zp = torch.from_numpy(zprev).cuda() if sched == S.MODE_ASYNC_TOPK else None
    sch = T.schedule(ws, d["conf_logit"], inp["sts"], inp["sps"], inp["anchor"], d["tokens"], sched,
                     conf_logit_prev=zp)
    cap_rows = B * (G + 1)
    if verify_mode == "cap_accept":
        full = torch.arange(B + 1, device="cuda", dtype=torch.int32) * (G + 1)
        v = T.verify(ws, inp["target"].reshape(-1, V), full, torch.full((B,), G, dtype=torch.int32, device="cuda"),
                     d["tokens"], d["pd_rows"], d["pd_tok"], inp["temp"], inp["req_id"], inp["seed"],
                     commit_cap=sch["ell"])
    else:
        rows = torch.empty((cap_rows, V), dtype=inp["target"].dtype, device="cuda")
        T.pack_rows(inp["target"], sch["mark_req"], sch["mark_pos"], sch["n_verify"], rows, ws)
        v = T.verify(ws, rows, sch["offsets"], sch["ell"], d["tokens"], d["pd_rows"], d["pd_tok"], inp["temp"],
                     inp["req_id"], inp["seed"])
    torch.cuda.synchronize()
    check_no_error(ws)

    ni = np_inputs(inp)
    od = oracle_draft(**ni, W_rnn=to_np64(Wr) if head == "rnn" else None,
                      rnn_row_dtype=("bf16" if inp["U"].dtype == torch.bfloat16 else "f32") if head == "rnn" else None)
    osch = S.schedule(od["conf_logit"].astype(np.float32), inp["sts"].cpu().numpy(), inp["sps"], ni["anchor"],
                      od["tokens"], mode=sched, conf_logit_prev=zprev)
    tgt = to_np64(inp["target"])
    if verify_mode == "cap_accept":
        fl = S.flatten(np.full(B, G), ni["anchor"], od["tokens"])
        ofull = oracle_verify(tgt[fl["mark_req"], fl["mark_pos"]], fl["offsets"], np.full(B, G), od["tokens"],
                              od["pd"], od["pd_tok"], ni["temp"], ni["seed"], ni["req_id"])
        ov = dict(cap_accept(ofull, osch["ell"]), accept_margin=ofull["accept_margin"],
                  sample_margin=ofull["sample_margin"])
    else:
        ov = oracle_verify(tgt[osch["mark_req"], osch["mark_pos"]], osch["offsets"], osch["ell"], od["tokens"],
                           od["pd"], od["pd_tok"], ni["temp"], ni["seed"], ni["req_id"])
    return (d, sch, v), (od, osch, ov)


@pytest.mark.parametrize("head,sched,verify_mode", [
    ("rnn", S.MODE_GREEDY, "compact"),
    ("markov", S.MODE_ASYNC_TOPK, "compact"),
    ("markov", S.MODE_GREEDY, "cap_accept"),
    ("rnn", S.MODE_ASYNC_TOPK, "cap_accept"),
])
def test_tiny_step_in_the_other_modes(head, sched, verify_mode):
    # the RNN head, the asynchronous scheduler and cap-accept verification, alone and together
    wl = synth.WORKLOADS["tiny"]
    full = 0
    for seed in range(24):
        inp = synth.make_inputs(wl, "cuda", seed=seed)
        Wr = synth.rnn_weights(wl.r, wl.H, wl.dtype, seed, "cuda")
        zprev = synth.random_conf_logits(wl.B, wl.gamma, 500 + seed)
        (d, sch, v), (od, osch, ov) = _step_modes(inp, head, sched, verify_mode, Wr, zprev)
        st = compare_draft(gpu_np(d), od, rtol_for(wl.dtype))
        if st["n_exempt_requests"]:
            continue
        if osch["theta_margin"] < 1e-4 or _cut_gap(osch) < 1e-4 or osch.get("cap_margin", np.inf) <= 1e-12:
            continue
        g_s = gpu_np(sch)
        np.testing.assert_array_equal(g_s["ell"], osch["ell"])
        np.testing.assert_array_equal(g_s["offsets"], osch["offsets"])
        compare_verify(gpu_np(v), ov, ~(inp["temp"].cpu().numpy() > 0))
        full += 1
    assert full >= 8
