"""GPU parity of dspark_verify against the oracle.

Verify inputs (tokens, p_d rows, p_d(x)) come from the oracle's own draft,
rounded to the fp32 the C ABI takes; both sides read those same fp32 values.
Target logits are synthetic; verify lengths come from the oracle scheduler.
"""
import numpy as np
import pytest
import torch

import synth
from oracle.draft import draft as oracle_draft
from oracle import schedule as S
from oracle.verify import verify as oracle_verify
from parity import compare_verify, np_inputs, to_np64
from gpu_common import check_no_error, require_gpu, to_dev_f32, to_dev_i32, workspace_for
from draft_sampling_lossless_markov_gb300 import torch_api as T

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _verify_both(target_rows_np, target_rows_dev, offsets, ell, tokens, pd32, pdtok32, temp, seed, req_id):
    B, G = tokens.shape
    V = target_rows_np.shape[1]
    ws = workspace_for(B, G, V, 0, 0, target_rows_dev.dtype)
    out = T.verify(ws, target_rows_dev, to_dev_i32(offsets), to_dev_i32(ell), to_dev_i32(tokens),
                   pd32 if isinstance(pd32, torch.Tensor) else to_dev_f32(pd32), to_dev_f32(pdtok32),
                   to_dev_f32(temp), to_dev_i32(req_id), seed)
    torch.cuda.synchronize()
    check_no_error(ws)
    g = {k: v.cpu().numpy() for k, v in out.items()}
    pd_host = pd32.cpu().numpy() if isinstance(pd32, torch.Tensor) else pd32
    o = oracle_verify(target_rows_np, offsets, ell, tokens, pd_host, pdtok32, temp, seed, req_id)
    st = compare_verify(g, o, ~(np.asarray(temp) > 0))
    # structure of the outputs
    assert np.all(g["n_out"] == g["n_accept"] + 1)
    assert np.all(g["n_accept"] <= ell)
    for r in range(B):
        m = g["n_accept"][r]
        np.testing.assert_array_equal(g["out_tok"][r, :m], tokens[r, :m])
        assert 0 <= g["out_tok"][r, m] < V and np.all(g["out_tok"][r, m + 1:] == -1)
    return g, o, st


def _pipeline_inputs(wl, seed, n_oracle=None, temp=None):
    inp = synth.make_inputs(wl, "cuda", seed=seed, temp=temp)
    B, G = wl.B, wl.gamma
    n_or = B if n_oracle is None else n_oracle
    idx = torch.arange(n_or, device="cuda")
    d = oracle_draft(**np_inputs(inp, idx))
    # tile the oracle's draft over the batch (request r uses draft r mod n_or, own id)
    src = np.arange(B) % n_or
    tokens = d["tokens"][src].astype(np.int32)
    pd32 = d["pd"][src].astype(np.float32)
    pdtok32 = d["pd_tok"][src].astype(np.float32)
    zl32 = d["conf_logit"][src].astype(np.float32)
    temp = inp["temp"].cpu().numpy()
    req_id = inp["req_id"].cpu().numpy()
    anchor = inp["anchor"].cpu().numpy()[src]
    return inp, tokens, pd32, pdtok32, zl32, temp, req_id, anchor


@pytest.mark.parametrize("temp", ["mixed", "1.0", "0", "0.7"])
@pytest.mark.parametrize("sched", [0, 1])
def test_verify_tiny(temp, sched):
    wl = synth.WORKLOADS["tiny"]
    tot = dict(n=0, ex=0)
    for seed in range(6):
        inp, tokens, pd32, pdtok32, zl32, tempv, req_id, anchor = _pipeline_inputs(wl, seed, temp=temp)
        sch = S.schedule(zl32, np.ones(wl.gamma, np.float32), synth.sps_table(wl.sps, wl.B, wl.gamma), anchor,
                         tokens, mode=sched)
        rows = inp["target"][torch.from_numpy(sch["mark_req"]).cuda(), torch.from_numpy(sch["mark_pos"]).cuda()]
        g, o, st = _verify_both(to_np64(rows), rows.contiguous(), sch["offsets"], sch["ell"], tokens, pd32,
                                pdtok32, tempv, inp["seed"], req_id)
        tot["n"] += st["n_requests"]
        tot["ex"] += st["n_exempt"]
    assert tot["ex"] <= 0.25 * tot["n"]


@pytest.mark.parametrize("name,n_oracle", [("qwen3_4b", 8), ("sweep_B256_g7", 8), ("deepseek_vocab", 8)])
def test_verify_full_size(name, n_oracle):
    wl = synth.get_workload(name)
    inp, tokens, pd32, pdtok32, zl32, tempv, req_id, anchor = _pipeline_inputs(wl, 0, n_oracle=n_oracle)
    G = wl.gamma
    sts = inp["sts"].cpu().numpy()
    sch = S.schedule(zl32, sts, synth.sps_table(wl.sps, wl.B, G), anchor, tokens, mode=wl.sched)
    rows = inp["target"][torch.from_numpy(sch["mark_req"]).cuda(), torch.from_numpy(sch["mark_pos"]).cuda()]
    rows = rows.contiguous()
    g, o, st = _verify_both(to_np64(rows), rows, sch["offsets"], sch["ell"], tokens, to_dev_f32(pd32), pdtok32,
                            tempv, inp["seed"], req_id)
    assert st["n_exempt"] <= 0.3 * st["n_requests"]


def test_verify_zero_length_and_draft_equal_target():
    rng = np.random.default_rng(3)
    B, G, V = 40, 4, 3000
    tgt = torch.randn((B, G + 1, V), device="cuda") * 3
    tokens = rng.integers(0, V, (B, G)).astype(np.int32)
    # l = 0 for every request: one target sample (bonus) each
    ell = np.zeros(B, np.int64)
    fl = S.flatten(ell, np.zeros(B), tokens)
    rows = tgt[torch.from_numpy(fl["mark_req"]).cuda(), torch.from_numpy(fl["mark_pos"]).cuda()].contiguous()
    temp = np.where(np.arange(B) % 3 == 0, 0.0, 0.9).astype(np.float32)
    pd = np.zeros((B, G, V), np.float32)
    pdt = np.ones((B, G), np.float32)
    g, o, st = _verify_both(to_np64(rows), rows, fl["offsets"], ell, tokens, pd, pdt, temp, 77, np.arange(B))
    assert np.all(g["n_accept"] == 0)
    # draft equal to the target (p_d = p_t): every token is accepted
    ell = np.full(B, G)
    fl = S.flatten(ell, np.zeros(B), tokens)
    rows = tgt[torch.from_numpy(fl["mark_req"]).cuda(), torch.from_numpy(fl["mark_pos"]).cuda()].contiguous()
    T_ = torch.from_numpy(np.where(temp > 0, temp, 1.0)).cuda()[:, None, None]
    pt = torch.softmax(tgt[:, :G].double() / T_, dim=2)
    tok = torch.multinomial(pt.reshape(-1, V).float(), 1, generator=torch.Generator("cuda").manual_seed(1))
    tok = tok.reshape(B, G).to(torch.int32)
    greedy = torch.from_numpy(temp <= 0).cuda()
    tok = torch.where(greedy[:, None], tgt[:, :G].argmax(dim=2).to(torch.int32), tok)
    pdrow = pt.float()
    pdtok = torch.gather(pdrow, 2, tok.long()[:, :, None])[:, :, 0]
    tok_np = tok.cpu().numpy()
    g, o, st = _verify_both(to_np64(rows), rows, fl["offsets"], ell, tok_np, pdrow.contiguous(),
                            pdtok.cpu().numpy(), temp, 78, np.arange(B))
    assert np.all(g["n_accept"][temp > 0] == G)


@pytest.mark.parametrize("V,dt", [(1001, torch.float32), (1003, torch.bfloat16), (4099, torch.float32)])
def test_verify_vocabulary_not_a_multiple_of_8(V, dt):
    # rows that are not 16-byte aligned take the scalar paths of every verify kernel
    rng = np.random.default_rng(V)
    B, G = 24, 3
    tgt = (torch.randn((B, G + 1, V), device="cuda") * 3).to(dt)
    tokens = rng.integers(0, V, (B, G)).astype(np.int32)
    ell = rng.integers(0, G + 1, B).astype(np.int64)
    fl = S.flatten(ell, np.zeros(B), tokens)
    rows = tgt[torch.from_numpy(fl["mark_req"]).cuda(), torch.from_numpy(fl["mark_pos"]).cuda()].contiguous()
    temp = np.where(np.arange(B) % 4 == 0, 0.0, 0.8).astype(np.float32)
    pd = rng.dirichlet(np.full(V, 0.3), size=(B, G)).astype(np.float32)
    pdt = np.take_along_axis(pd, tokens[:, :, None].astype(np.int64), axis=2)[:, :, 0]
    _verify_both(to_np64(rows), rows, fl["offsets"], ell, tokens, pd, pdt, temp, 91, np.arange(B))


def _cap_accept_both(inp, tokens, pd32, pdtok32, tempv, req_id, anchor, cap):
    from oracle.verify import cap_accept
    B, G = tokens.shape
    full = S.flatten(np.full(B, G), anchor, tokens)  # the whole block is verified
    rows = inp["target"][torch.from_numpy(full["mark_req"]).cuda(), torch.from_numpy(full["mark_pos"]).cuda()]
    rows = rows.contiguous()
    V = rows.shape[1]
    ws = workspace_for(B, G, V, 0, 0, rows.dtype)
    out = T.verify(ws, rows, to_dev_i32(full["offsets"]), to_dev_i32(np.full(B, G)), to_dev_i32(tokens),
                   to_dev_f32(pd32), to_dev_f32(pdtok32), to_dev_f32(tempv), to_dev_i32(req_id), inp["seed"],
                   commit_cap=to_dev_i32(cap))
    torch.cuda.synchronize()
    check_no_error(ws)
    g = {k: v.cpu().numpy() for k, v in out.items()}
    o_full = oracle_verify(to_np64(rows), full["offsets"], np.full(B, G), tokens, pd32, pdtok32, tempv, inp["seed"],
                           req_id)
    o = dict(cap_accept(o_full, cap), accept_margin=o_full["accept_margin"], sample_margin=o_full["sample_margin"])
    st = compare_verify(g, o, ~(np.asarray(tempv) > 0))
    assert np.all(g["n_out"] == np.minimum(g["n_accept"], cap) + 1)
    for r in range(B):
        k = g["n_out"][r]
        assert np.all(g["out_tok"][r, k:] == -1) and np.all(g["out_tok"][r, :k] >= 0)
    return g, o, st


@pytest.mark.parametrize("temp", ["mixed", "1.0", "0"])
def test_verify_cap_accept_tiny(temp):
    wl = synth.WORKLOADS["tiny"]
    tot = dict(n=0, ex=0)
    for seed in range(6):
        inp, tokens, pd32, pdtok32, zl32, tempv, req_id, anchor = _pipeline_inputs(wl, seed, temp=temp)
        # windows from the scheduler on even seeds, uniform 0..gamma on odd ones
        if seed % 2 == 0:
            cap = S.schedule(zl32, np.ones(wl.gamma, np.float32), synth.sps_table(wl.sps, wl.B, wl.gamma), anchor,
                             tokens, mode=1)["ell"]
        else:
            cap = np.random.default_rng(seed).integers(0, wl.gamma + 1, wl.B)
        g, o, st = _cap_accept_both(inp, tokens, pd32, pdtok32, tempv, req_id, anchor, cap.astype(np.int32))
        tot["n"] += st["n_requests"]
        tot["ex"] += st["n_exempt"]
    assert tot["ex"] <= 0.25 * tot["n"]


def test_verify_cap_accept_full_size():
    wl = synth.get_workload("sweep_B256_g7")
    inp, tokens, pd32, pdtok32, zl32, tempv, req_id, anchor = _pipeline_inputs(wl, 0, n_oracle=8)
    cap = S.schedule(zl32, inp["sts"].cpu().numpy(), synth.sps_table(wl.sps, wl.B, wl.gamma), anchor, tokens,
                     mode=1)["ell"].astype(np.int32)
    cap[:3] = [0, wl.gamma, 1]
    g, o, st = _cap_accept_both(inp, tokens, pd32, pdtok32, tempv, req_id, anchor, cap)
    assert st["n_exempt"] <= 0.3 * st["n_requests"]


def test_verify_cap_accept_reports_a_window_out_of_range():
    wl = synth.WORKLOADS["tiny"]
    inp, tokens, pd32, pdtok32, zl32, tempv, req_id, anchor = _pipeline_inputs(wl, 1)
    B, G = tokens.shape
    full = S.flatten(np.full(B, G), anchor, tokens)
    rows = inp["target"][torch.from_numpy(full["mark_req"]).cuda(), torch.from_numpy(full["mark_pos"]).cuda()]
    ws = workspace_for(B, G, rows.shape[1], 0, 0, rows.dtype)
    cap = np.full(B, 1, np.int32)
    cap[2] = G + 1
    out = T.verify(ws, rows.contiguous(), to_dev_i32(full["offsets"]), to_dev_i32(np.full(B, G)), to_dev_i32(tokens),
                   to_dev_f32(pd32), to_dev_f32(pdtok32), to_dev_f32(tempv), to_dev_i32(req_id), inp["seed"],
                   commit_cap=to_dev_i32(cap))
    torch.cuda.synchronize()
    from draft_sampling_lossless_markov_gb300 import capi
    assert ws.read_error() == (capi.DSPARK_BAD_INPUT, 2)
    # clamped to gamma: the full output for that request
    assert int(out["n_out"][2]) == int(out["n_accept"][2]) + 1
