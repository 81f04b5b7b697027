"""GPU parity at the benchmark's full sizes (V = 151936 or 129280), against the
fp64 oracle run request by request on a spread-out sample.

The whole batch runs on the GPU in the launch configuration the benchmark
times (the fused tensor-core draft kernel for these shapes); the oracle
recomputes a sample of requests one by one.  Draws are keyed by request id, so
a request's outputs do not depend on the rest of the batch.  The samples cover
every 128-row M-tile of the batch, greedy and sampled requests where the
workload mixes them, and both ends of the batch.  Each test reports how many
draft tokens it compared bit for bit (tokens after the first draw inside the
1e-5 CDF margin are not compared, as the tolerance contract says).

Workloads: the Qwen3-8B-shaped step with scheduling (B256, gamma 15, T 0.7,
STS temperatures), the headline sweep point (B256, gamma 7), the DeepSeek
vocabulary (B1024, half greedy) and the two ends of the batch sweep (B1 and
B4096 at gamma 7).
"""
import numpy as np
import pytest
import torch

import synth
from oracle.draft import draft as oracle_draft
from oracle import schedule as S
from oracle.verify import verify as oracle_verify
from parity import compare_draft, compare_verify, np_inputs, rtol_for, to_np64
from gpu_common import check_no_error, gpu_draft, require_gpu, to_dev_f32, to_dev_i32, workspace_for
from draft_sampling_lossless_markov_gb300 import torch_api as T

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _spread(B, n):
    """n request indices spread over the batch, first and last included."""
    if B <= n:
        return list(range(B))
    idx = np.unique(np.round(np.linspace(0, B - 1, n)).astype(int))
    return [int(i) for i in idx]


def _draft_sample_parity(name, subset, min_tokens, sampling_seeds=(None,)):
    tot = 0
    for ss in sampling_seeds:
        st = _draft_sample_parity_once(name, subset, ss)
        tot += st["n_tokens_compared"]
    assert tot >= min_tokens, (name, tot)


def _draft_sample_parity_once(name, subset, sampling_seed):
    wl = synth.get_workload(name)
    inp = synth.make_inputs(wl, "cuda", with_target=False, sampling_seed=sampling_seed)
    out, ws = gpu_draft(inp)
    check_no_error(ws)
    idx = torch.tensor(subset, device="cuda")
    g = {k: v.index_select(0, idx).cpu().numpy() for k, v in out.items()}
    o = oracle_draft(**np_inputs(inp, idx))
    st = compare_draft(g, o, rtol_for(wl.dtype))
    # p_d(x_k) is the emitted row's entry at the drawn token, bit for bit
    pick = np.take_along_axis(g["pd_rows"], g["tokens"][:, :, None].astype(np.int64), axis=2)[:, :, 0]
    np.testing.assert_array_equal(pick, g["pd_tok"])
    # whole-batch properties
    tok = out["tokens"]
    assert int(tok.min()) >= 0 and int(tok.max()) < wl.V
    s = out["pd_rows"].sum(dim=2)
    assert float((s - 1).abs().max()) < 5e-4
    c = out["conf"]
    assert float(c.min()) >= 0 and float(c.max()) <= 1
    print(f"{name} (sampling seed {sampling_seed}): {st['n_tokens_compared']} draft tokens compared bit-exact over "
          f"{len(subset)} requests ({st['n_exempt_requests']} requests met a draw inside the margin)")
    return st


@pytest.mark.parametrize("name,n_req,min_tokens,n_seeds", [
    ("sweep_B256_g7", 64, 150, 1),    # the headline point: both M-tiles, 64 requests
    ("qwen3_8b_sched", 48, 150, 1),   # gamma 15, T 0.7
    ("deepseek_vocab", 64, 150, 1),   # V 129280, even request ids greedy, odd sampled; 8 M-tiles
    ("sweep_B1_g7", 1, 12, 6),        # one request: six sampling seeds (six draw sequences)
    ("sweep_B8_g7", 8, 40, 2),
    ("sweep_B4096_g7", 48, 100, 1),   # 32 M-tiles
])
def test_draft_full_size(name, n_req, min_tokens, n_seeds):
    wl = synth.get_workload(name)
    seeds = (None,) if n_seeds == 1 else tuple(1000 + i for i in range(n_seeds))
    _draft_sample_parity(name, _spread(wl.B, n_req), min_tokens, seeds)


def test_draft_deepseek_vocab_covers_greedy_and_sampled_requests():
    # the sample above takes both parities of request id; check that explicitly
    wl = synth.get_workload("deepseek_vocab")
    sub = _spread(wl.B, 64)
    ids = np.asarray(sub)
    assert (ids % 2 == 0).sum() >= 16 and (ids % 2 == 1).sum() >= 16
    assert len({i // 128 for i in sub}) == (wl.B + 127) // 128


def _verify_sample(name, n_oracle):
    """Verify at full size: the oracle's draft of n_oracle requests tiled over the
    batch (request r takes draft r mod n_oracle, its own id), the oracle
    scheduler's lengths, the kept target rows packed by the marker tensor."""
    wl = synth.get_workload(name)
    inp = synth.make_inputs(wl, "cuda")
    B, G, V = wl.B, wl.gamma, wl.V
    idx = torch.arange(n_oracle, device="cuda")
    d = oracle_draft(**np_inputs(inp, idx))
    src = np.arange(B) % n_oracle
    tokens = d["tokens"][src].astype(np.int32)
    pd32 = d["pd"][src].astype(np.float32)
    pdtok32 = d["pd_tok"][src].astype(np.float32)
    zl32 = d["conf_logit"][src].astype(np.float32)
    temp = inp["temp"].cpu().numpy()
    req_id = inp["req_id"].cpu().numpy()
    anchor = inp["anchor"].cpu().numpy()[src]
    sch = S.schedule(zl32, inp["sts"].cpu().numpy(), synth.sps_table(wl.sps, B, G), anchor, tokens, mode=wl.sched)
    rows = inp["target"][torch.from_numpy(sch["mark_req"]).cuda(), torch.from_numpy(sch["mark_pos"]).cuda()]
    rows = rows.contiguous()
    ws = workspace_for(B, G, V, 0, 0, rows.dtype)
    out = T.verify(ws, rows, to_dev_i32(sch["offsets"]), to_dev_i32(sch["ell"]), to_dev_i32(tokens),
                   to_dev_f32(pd32), to_dev_f32(pdtok32), to_dev_f32(temp), to_dev_i32(req_id), inp["seed"])
    torch.cuda.synchronize()
    check_no_error(ws)
    g = {k: v.cpu().numpy() for k, v in out.items()}
    o = oracle_verify(to_np64(rows), sch["offsets"], sch["ell"], tokens, pd32, pdtok32, temp, inp["seed"], req_id)
    st = compare_verify(g, o, ~(temp > 0))
    assert np.all(g["n_out"] == g["n_accept"] + 1)
    assert np.all(g["n_accept"] <= sch["ell"])
    print(f"{name}: verify compared {st['n_requests'] - st['n_exempt']} of {st['n_requests']} requests, "
          f"{int(sch['offsets'][-1])} kept rows")
    return st


def test_verify_qwen3_8b_sched_full_size():
    # every one of the 256 requests is compared (the oracle verifies the whole batch)
    st = _verify_sample("qwen3_8b_sched", 16)
    assert st["n_exempt"] <= 0.3 * st["n_requests"]


def test_qwen3_8b_sched_step_on_the_gpu():
    # the three calls chained on the GPU at full size; the oracle recomputes a sample
    # of requests' drafts, and the scheduler's outputs are checked against the
    # oracle scheduler run on the GPU's own confidences and tokens
    wl = synth.get_workload("qwen3_8b_sched")
    inp = synth.make_inputs(wl, "cuda")
    B, G, V = wl.B, wl.gamma, wl.V
    d, ws = gpu_draft(inp)
    sch = T.schedule(ws, d["conf_logit"], inp["sts"], inp["sps"], inp["anchor"], d["tokens"], wl.sched)
    torch.cuda.synchronize()
    n = int(sch["n_verify"][0])
    rows = torch.empty((B * (G + 1), V), dtype=inp["target"].dtype, device="cuda")
    T.pack_rows(inp["target"], sch["mark_req"], sch["mark_pos"], sch["n_verify"], rows, ws)
    v = T.verify(ws, rows, sch["offsets"], sch["ell"], d["tokens"], d["pd_rows"], d["pd_tok"], inp["temp"],
                 inp["req_id"], inp["seed"])
    torch.cuda.synchronize()
    check_no_error(ws)
    # scheduler: the oracle on the GPU's fp32 confidence logits and tokens
    osch = S.schedule(d["conf_logit"].cpu().numpy(), inp["sts"].cpu().numpy(), inp["sps"],
                      inp["anchor"].cpu().numpy(), d["tokens"].cpu().numpy(), mode=wl.sched)
    if osch["theta_margin"] > 1e-12:
        np.testing.assert_array_equal(sch["ell"].cpu().numpy(), osch["ell"])
        np.testing.assert_array_equal(sch["offsets"].cpu().numpy(), osch["offsets"])
        for k in ("flat_tok", "mark_req", "mark_pos"):
            np.testing.assert_array_equal(sch[k].cpu().numpy()[:n], osch[k])
    # verify: the oracle on the GPU's draft outputs and the packed rows
    tok = d["tokens"].cpu().numpy()
    o = oracle_verify(to_np64(rows[:n]), sch["offsets"].cpu().numpy(), sch["ell"].cpu().numpy(), tok,
                      d["pd_rows"].cpu().numpy(), d["pd_tok"].cpu().numpy(), inp["temp"].cpu().numpy(), inp["seed"],
                      inp["req_id"].cpu().numpy())
    g = {k: t.cpu().numpy() for k, t in v.items()}
    st = compare_verify(g, o, ~(inp["temp"].cpu().numpy() > 0))
    assert st["n_exempt"] <= 0.3 * st["n_requests"]
    # the draft sample
    sub = _spread(B, 16)
    idx = torch.tensor(sub, device="cuda")
    od = oracle_draft(**np_inputs(inp, idx))
    gd = {k: t.index_select(0, idx).cpu().numpy() for k, t in d.items()}
    compare_draft(gd, od, rtol_for(wl.dtype))
