"""GPU parity of the p_d-row-free mode: the draft writes no p_d rows (its
select yields p_d(x_k) and each row's (max, sum)), and verify draws the
residual by rejection from p_t, recomputing p_d at the proposed tokens from
U, W1 and W2.  Compared with the draft in the row mode (same select: equal
tokens) and with the oracle's step using the rejection residual."""
import numpy as np
import pytest
import torch

import synth
from oracle.draft import draft as oracle_draft
from oracle import schedule as S
from oracle.verify import verify as oracle_verify
from parity import MARGIN, compare_draft, compare_verify, gpu_np, np_inputs, rtol_for, to_np64
from gpu_common import check_no_error, require_gpu, workspace_for
from draft_sampling_lossless_markov_gb300 import capi
from draft_sampling_lossless_markov_gb300 import torch_api as T

pytestmark = pytest.mark.gpu

LOG2E = 1.4426950408889634


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _draft(inp, rows):
    U = inp["U"]
    B, G, V = U.shape
    ws = workspace_for(B, G, V, inp["W1"].shape[1], inp["h"].shape[2], U.dtype)
    out = T.draft_sample(ws, U, inp["W1"], inp["W2"], inp["h"], inp["w"], inp["anchor"], inp["temp"], inp["req_id"],
                         inp["seed"], rows=rows, want_pd_stat=True)
    torch.cuda.synchronize()
    check_no_error(ws)
    return out, ws


def _workload(B, G, V, r, H, temp="mixed", seed=5):
    return synth.Workload("rowfree", B, G, V, H, r, "bf16", temp, synth.SCHED_GREEDY, "exp2048", seed=seed)


@pytest.mark.parametrize("B,G,V,r,H", [(40, 3, 1024, 256, 8), (130, 5, 8200, 128, 16), (256, 7, 151936, 256, 4096),
                                       (300, 1, 2056, 64, 8), (260, 16, 2048, 192, 32),
                                       # small batches (the vocabulary on the MMA's M side)
                                       (1, 7, 151936, 256, 4096), (8, 4, 8200, 256, 16), (16, 5, 4104, 64, 24)])
def test_row_free_draft_matches_the_row_mode(B, G, V, r, H):
    wl = _workload(B, G, V, r, H)
    inp = synth.make_inputs(wl, "cuda", with_target=False)
    a, _ = _draft(inp, rows=True)
    b, _ = _draft(inp, rows=False)
    assert "pd_rows" not in b
    for k in ("tokens", "conf_logit", "conf", "pd_stat"):
        assert torch.equal(a[k], b[k]), k  # the same select
    # p_d(x_k): from the emitted row in the row mode, from the select's walk here
    torch.testing.assert_close(b["pd_tok"], a["pd_tok"], rtol=2e-6, atol=0)
    # (max, sum) reproduce the emitted rows: 2^(y - m) / S with y = l log2(e) / T
    pd_rows = a["pd_rows"]
    n = min(B, 8)
    U, W1, W2 = (to_np64(inp[k]) for k in ("U", "W1", "W2"))
    tok = a["tokens"].cpu().numpy()
    anchor, temp = inp["anchor"].cpu().numpy(), inp["temp"].cpu().numpy()
    st = a["pd_stat"].cpu().numpy()
    for rq in range(n):
        if not temp[rq] > 0:
            continue
        for k in range(G):
            xp = anchor[rq] if k == 0 else tok[rq, k - 1]
            y = (U[rq, k] + W1[xp] @ W2) * LOG2E / temp[rq]
            p = np.exp2(y - st[rq, k, 0]) / st[rq, k, 1]
            np.testing.assert_allclose(p, pd_rows[rq, k].cpu().numpy(), rtol=2e-3, atol=1e-30)


def test_row_free_draft_against_the_oracle():
    wl = _workload(40, 4, 2048, 64, 16, seed=6)
    inp = synth.make_inputs(wl, "cuda", with_target=False)
    b, _ = _draft(inp, rows=False)
    g = gpu_np(b)
    o = oracle_draft(**np_inputs(inp))
    st = compare_draft(g, o, rtol_for("bf16"), check_pd_rows=False)
    assert st["n_tokens_compared"] >= 0.5 * wl.B * wl.gamma


@pytest.mark.parametrize("temp", ["1.0", "mixed"])
def test_row_free_step_against_the_oracle(temp):
    # draft without rows -> schedule -> packed rows -> verify with the rejection residual;
    # the oracle verifies the same scheduled lengths, request by request (requests with
    # a draft draw inside the margin are left out)
    n_cmp = 0
    for seed in range(6):
        wl = _workload(40, 4, 2048, 64, 16, temp=temp, seed=20 + seed)
        inp = synth.make_inputs(wl, "cuda")
        B, G, V = wl.B, wl.gamma, wl.V
        d, ws = _draft(inp, rows=False)
        sch = T.schedule(ws, d["conf_logit"], inp["sts"], inp["sps"], inp["anchor"], d["tokens"], wl.sched)
        rows = torch.empty((B * (G + 1), V), dtype=torch.bfloat16, device="cuda")
        T.pack_rows(inp["target"], sch["mark_req"], sch["mark_pos"], sch["n_verify"], rows, ws)
        v = T.verify(ws, rows, sch["offsets"], sch["ell"], d["tokens"], None, d["pd_tok"], inp["temp"],
                     inp["req_id"], inp["seed"],
                     rejection=dict(U=inp["U"], W1=inp["W1"], W2=inp["W2"], anchor=inp["anchor"],
                                    pd_stat=d["pd_stat"]))
        torch.cuda.synchronize()
        check_no_error(ws)
        ni = np_inputs(inp)
        od = oracle_draft(**ni)
        ok = (od["margin"] >= MARGIN).all(axis=1)
        np.testing.assert_array_equal(d["tokens"].cpu().numpy()[ok], od["tokens"][ok])
        ell = sch["ell"].cpu().numpy().astype(np.int64)
        fl = S.flatten(ell, ni["anchor"], od["tokens"])
        tgt = to_np64(inp["target"])
        ov = oracle_verify(tgt[fl["mark_req"], fl["mark_pos"]], fl["offsets"], ell, od["tokens"], od["pd"],
                           od["pd_tok"], ni["temp"], ni["seed"], ni["req_id"], residual="rejection")
        g = gpu_np(v)
        st = compare_verify({k: a[ok] for k, a in g.items()},
                            {k: a[ok] for k, a in ov.items() if isinstance(a, np.ndarray)}, ~(ni["temp"][ok] > 0))
        n_cmp += st["n_requests"] - st["n_exempt"]
        # some of the compared requests rejected a sampled draft token: the residual ran
        assert np.any((ov["n_accept"] < ell)[ok] & (ni["temp"][ok] > 0)) or temp == "mixed"
    assert n_cmp >= 100


def test_rejection_residual_fallback_after_the_trials():
    # a draft that differs from the target at two tokens only: rejections are rare and
    # their residual mass tiny, so most of them exhaust the proposals and fall back to
    # the inverse-CDF draw over a recomputed residual
    B, G, V, r = 65536, 1, 64, 64
    rng = np.random.default_rng(7)
    zt = rng.normal(size=V).astype(np.float32) * 0.5
    x1, x2 = 5, 9
    Urow = zt.copy()
    Urow[x1] += 0.02          # p_d > p_t at x1, p_d < p_t elsewhere (mostly at x2 after the shift below)
    Urow[x2] -= 0.02
    dev = "cuda"
    U = torch.from_numpy(np.broadcast_to(Urow, (B, G, V)).copy()).to(torch.bfloat16).to(dev)
    Ub = U[0, 0].float().cpu().numpy().astype(np.float64)
    W1 = torch.zeros((V, r), dtype=torch.bfloat16, device=dev)
    W2 = torch.zeros((r, V), dtype=torch.bfloat16, device=dev)
    anchor = torch.zeros(B, dtype=torch.int32, device=dev)
    temp = torch.ones(B, dtype=torch.float32, device=dev)
    req_id = torch.arange(B, dtype=torch.int32, device=dev)
    y = Ub * LOG2E
    m = y.max()
    Ssum = np.exp2(y - m).sum()
    pd_row = np.exp2(y - m) / Ssum
    tokens = torch.full((B, G), x1, dtype=torch.int32, device=dev)
    pd_tok = torch.full((B, G), float(pd_row[x1]), dtype=torch.float32, device=dev)
    pd_stat = torch.tensor([m, Ssum], dtype=torch.float32).repeat(B * G).view(B, G, 2).to(dev)
    target = torch.from_numpy(np.tile(zt, (B, G + 1, 1))).to(torch.bfloat16).to(dev)
    tgt_rows = target.view(-1, V)
    offsets = torch.arange(B + 1, dtype=torch.int32, device=dev) * (G + 1)
    ell = torch.full((B,), G, dtype=torch.int32, device=dev)
    ws = workspace_for(B, G, V, r, 0, torch.bfloat16)
    seed = 1234
    v = T.verify(ws, tgt_rows, offsets, ell, tokens, None, pd_tok, temp, req_id, seed,
                 rejection=dict(U=U, W1=W1, W2=W2, anchor=anchor, pd_stat=pd_stat))
    torch.cuda.synchronize()
    check_no_error(ws)
    g = gpu_np(v)
    pd_full = np.broadcast_to(pd_row, (B, G, V))
    ov = oracle_verify(to_np64(tgt_rows), offsets.cpu().numpy(), ell.cpu().numpy(), tokens.cpu().numpy(), pd_full,
                       pd_tok.cpu().numpy().astype(np.float64), temp.cpu().numpy(), seed, req_id.cpu().numpy(),
                       residual="rejection")
    rej = ov["n_accept"] == 0
    assert rej.sum() >= 5 and ov["residual_fallback"][rej].sum() >= 3
    compare_verify(g, ov, np.zeros(B, bool))


def test_row_free_draft_unsupported_off_the_fused_path():
    wl = synth.Workload("rowfree32", 8, 3, 1000, 16, 16, "f32", "1.0", synth.SCHED_GREEDY, "tiny", seed=1)
    inp = synth.make_inputs(wl, "cuda", with_target=False)
    with pytest.raises(T.DsparkError) as e:
        _draft(inp, rows=False)
    assert e.value.status == capi.DSPARK_UNSUPPORTED


def test_row_free_step_full_size_sampled_requests():
    # the headline batch in the row-free mode; the oracle recomputes 24 requests
    # (draws are keyed by request id) on the GPU's scheduled lengths
    wl = synth.get_workload("sweep_B256_g7")
    inp = synth.make_inputs(wl, "cuda")
    B, G, V = wl.B, wl.gamma, wl.V
    d, ws = _draft(inp, rows=False)
    sch = T.schedule(ws, d["conf_logit"], inp["sts"], inp["sps"], inp["anchor"], d["tokens"], wl.sched)
    rows = torch.empty((B * (G + 1), V), dtype=torch.bfloat16, device="cuda")
    T.pack_rows(inp["target"], sch["mark_req"], sch["mark_pos"], sch["n_verify"], rows, ws)
    v = T.verify(ws, rows, sch["offsets"], sch["ell"], d["tokens"], None, d["pd_tok"], inp["temp"], inp["req_id"],
                 inp["seed"], rejection=dict(U=inp["U"], W1=inp["W1"], W2=inp["W2"], anchor=inp["anchor"],
                                             pd_stat=d["pd_stat"]))
    torch.cuda.synchronize()
    check_no_error(ws)
    subset = list(range(0, 256, 11))  # 24 requests across the batch
    idx = torch.tensor(subset, device="cuda")
    ni = np_inputs(inp, idx)
    od = oracle_draft(**ni)
    ok = (od["margin"] >= MARGIN).all(axis=1)
    np.testing.assert_array_equal(d["tokens"][idx].cpu().numpy()[ok], od["tokens"][ok])
    ell = sch["ell"][idx].cpu().numpy().astype(np.int64)
    fl = S.flatten(ell, ni["anchor"], od["tokens"])
    tgt = inp["target"].index_select(0, idx)
    ov = oracle_verify(to_np64(tgt[torch.from_numpy(fl["mark_req"]).cuda(), torch.from_numpy(fl["mark_pos"]).cuda()]),
                       fl["offsets"], ell, od["tokens"], od["pd"], od["pd_tok"], ni["temp"], ni["seed"], ni["req_id"],
                       residual="rejection")
    g = {k: t.index_select(0, idx).cpu().numpy() for k, t in v.items()}
    st = compare_verify({k: a[ok] for k, a in g.items()},
                        {k: a[ok] for k, a in ov.items() if isinstance(a, np.ndarray)}, ~(ni["temp"][ok] > 0))
    assert st["n_requests"] - st["n_exempt"] >= 8
