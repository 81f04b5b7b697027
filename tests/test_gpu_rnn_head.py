"""GPU parity of the RNN sequential head (dspark_draft_sample, head = RNN)
against the fp64 oracle, through the C ABI.  The oracle takes the rows
tanh(W_o z_k) in the bias product's operand precision (the workload's dtype),
as the library does; bf16 tensor-core shapes run the tensor-core passes, the
others the CUDA-core path (a child process forces the latter for bf16 too)."""
import numpy as np
import pytest
import torch

import synth
from oracle.draft import draft as oracle_draft
from parity import compare_draft, gpu_np, np_inputs, rtol_for, to_np64
from gpu_common import check_no_error, require_gpu, workspace_for
from draft_sampling_lossless_markov_gb300 import torch_api as T

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _run(inp, W_rnn):
    U = inp["U"]
    B, G, V = U.shape
    r, H = inp["W1"].shape[1], inp["h"].shape[2]
    ws = workspace_for(B, G, V, r, H, U.dtype)
    out = T.draft_sample(ws, U, inp["W1"], inp["W2"], inp["h"] if H else None, inp["w"], inp["anchor"],
                         inp["temp"], inp["req_id"], inp["seed"], W_rnn=W_rnn)
    torch.cuda.synchronize()
    return out, ws


def _invariants(g, V):
    assert g["tokens"].min() >= 0 and g["tokens"].max() < V
    pick = np.take_along_axis(g["pd_rows"], g["tokens"][:, :, None].astype(np.int64), axis=2)[:, :, 0]
    np.testing.assert_array_equal(pick, g["pd_tok"])
    np.testing.assert_allclose(g["pd_rows"].sum(axis=2), 1.0, rtol=0, atol=5e-5)


@pytest.mark.parametrize("temp", ["mixed", "0", "1.0", "0.7"])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_rnn_head_tiny(temp, seed):
    wl = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(wl, "cuda", seed=seed, temp=temp, with_target=False)
    Wr = synth.rnn_weights(wl.r, wl.H, wl.dtype, seed, "cuda")
    out, ws = _run(inp, Wr)
    g = gpu_np(out)
    _invariants(g, wl.V)
    o = oracle_draft(**np_inputs(inp), W_rnn=to_np64(Wr), rnn_row_dtype=wl.dtype)
    st = compare_draft(g, o, rtol_for(wl.dtype))
    assert st["n_tokens_compared"] >= 0.5 * wl.B * wl.gamma
    check_no_error(ws)


@pytest.mark.parametrize("B,G,V,r,H,dt", [
    (1, 1, 7, 1, 0, "f32"),         # one request, one position, rank 1, no hidden state
    (3, 5, 1000, 16, 40, "f32"),    # vocabulary not a multiple of the tile width
    (17, 3, 1031, 7, 5, "f32"),     # rank below one column tile, odd sizes
    (130, 4, 2000, 48, 0, "f32"),   # no hidden state, ragged request and column tiles
    (5, 4, 4104, 64, 24, "bf16"),   # bf16 inputs, fp32 recurrent rows
    (33, 2, 2056, 1, 8, "bf16"),    # rank 1
    (40, 6, 1024, 256, 8, "bf16"),  # rank 256 over six positions: tensor-core passes
    (130, 5, 8200, 128, 16, "bf16"),  # two M-tiles, an 8-column last tile: tensor-core passes
    (1, 7, 8200, 256, 16, "bf16"),    # one request: the small-batch form with the recurrent units
    (16, 5, 8200, 128, 8, "bf16"),    # the small-batch form's largest batch
    (9, 3, 4104, 192, 0, "bf16"),     # small batch, rank 192, no hidden state
])
def test_rnn_head_ragged_shapes(B, G, V, r, H, dt):
    wl = synth.Workload("rnn", B, G, V, H, r, dt, "mixed", synth.SCHED_GREEDY, "tiny", seed=5)
    inp = synth.make_inputs(wl, "cuda", with_target=False)
    Wr = synth.rnn_weights(r, H, dt, 3, "cuda")
    out, ws = _run(inp, Wr)
    g = gpu_np(out)
    _invariants(g, V)
    o = oracle_draft(**np_inputs(inp), W_rnn=to_np64(Wr), rnn_row_dtype=dt)
    compare_draft(g, o, rtol_for(dt))
    check_no_error(ws)


@pytest.mark.parametrize("name,subset,min_tokens", [
    # the whole B256 batch at V151936, r256, H4096 (the 128-row form); 24 requests
    # spread over both M-tiles
    ("sweep_B256_g7", list(range(0, 256, 11)), 40),
    # one request at full size: the small-batch form with its recurrent units
    ("sweep_B1_g7", [0], 1),
])
def test_rnn_head_full_size_sampled_requests(name, subset, min_tokens):
    wl = synth.get_workload(name)
    inp = synth.make_inputs(wl, "cuda", with_target=False)
    Wr = synth.rnn_weights(wl.r, wl.H, wl.dtype, 0, "cuda")
    out, ws = _run(inp, Wr)
    idx = torch.tensor(subset, device="cuda")
    g = {k: v.index_select(0, idx).cpu().numpy() for k, v in out.items()}
    _invariants(g, wl.V)
    o = oracle_draft(**np_inputs(inp, idx), W_rnn=to_np64(Wr), rnn_row_dtype=wl.dtype)
    st = compare_draft(g, o, rtol_for(wl.dtype))
    assert st["n_tokens_compared"] >= min_tokens
    check_no_error(ws)


@pytest.mark.parametrize("B,G,V,r,H,subset", [
    # about 6 recurrent units per CTA in the fused form: unit ranges cross row
    # blocks and M-tiles, a ragged last row block (20 rows) and M-tile (116 rows)
    (500, 3, 8200, 256, 16, [0, 31, 32, 127, 128, 300, 383, 384, 479, 480, 499]),
    # above 512 requests: the pass kernels with the recurrent step on the tensor cores
    (1000, 3, 8200, 256, 16, [0, 31, 32, 127, 128, 300, 511, 767, 895, 896, 991, 999]),
    # no hidden state (no h projection), rank 64: a ragged 12-row last block
    (300, 3, 4104, 64, 0, [0, 63, 64, 127, 128, 255, 256, 287, 288, 299]),
    # rank 192: six of the eight segments of z' in use
    (200, 4, 8200, 192, 8, [0, 31, 32, 127, 128, 191, 192, 199]),
])
def test_rnn_head_many_units_per_cta(B, G, V, r, H, subset):
    wl = synth.Workload("rnn_units", B, G, V, H, r, "bf16", "mixed", synth.SCHED_GREEDY, "tiny", seed=9)
    inp = synth.make_inputs(wl, "cuda", with_target=False)
    Wr = synth.rnn_weights(r, H, "bf16", 6, "cuda")
    out, ws = _run(inp, Wr)
    _invariants(gpu_np(out), V)
    idx = torch.tensor(subset, device="cuda")
    g = {k: v.index_select(0, idx).cpu().numpy() for k, v in out.items()}
    o = oracle_draft(**np_inputs(inp, idx), W_rnn=to_np64(Wr), rnn_row_dtype="bf16")
    st = compare_draft(g, o, rtol_for("bf16"))
    assert st["n_tokens_compared"] >= len(subset)
    check_no_error(ws)


def test_rnn_head_differs_from_the_markov_head():
    # same inputs: the recurrent rows change the draft distribution
    wl = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(wl, "cuda", seed=4, temp="1.0", with_target=False)
    inp["W2"] = inp["W2"] * 50  # a bias large enough to move the rows visibly
    Wr = synth.rnn_weights(wl.r, wl.H, wl.dtype, 4, "cuda")
    rnn, _ = _run(inp, Wr)
    ws = workspace_for(wl.B, wl.gamma, wl.V, wl.r, wl.H, inp["U"].dtype)
    mk = T.draft_sample(ws, inp["U"], inp["W1"], inp["W2"], inp["h"], inp["w"], inp["anchor"], inp["temp"],
                        inp["req_id"], inp["seed"])
    torch.cuda.synchronize()
    assert float((rnn["pd_rows"][:, 0] - mk["pd_rows"][:, 0]).abs().max()) > 1e-3


CHILD = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import synth, torch
from oracle.draft import draft as oracle_draft
from parity import compare_draft, gpu_np, np_inputs, rtol_for, to_np64
from gpu_common import check_no_error, workspace_for
from draft_sampling_lossless_markov_gb300 import torch_api as T
for B, G, V, r, H in [(130, 5, 8200, 128, 16), (5, 4, 4104, 64, 24), (600, 3, 8200, 256, 16)]:
    wl = synth.Workload("paths", B, G, V, H, r, "bf16", "mixed", synth.SCHED_GREEDY, "tiny", seed=11)
    inp = synth.make_inputs(wl, "cuda", with_target=False)
    Wr = synth.rnn_weights(r, H, "bf16", 2, "cuda")
    ws = workspace_for(B, G, V, r, H, torch.bfloat16)
    out = T.draft_sample(ws, inp["U"], inp["W1"], inp["W2"], inp["h"], inp["w"], inp["anchor"], inp["temp"],
                         inp["req_id"], inp["seed"], W_rnn=Wr)
    torch.cuda.synchronize()
    o = oracle_draft(**np_inputs(inp), W_rnn=to_np64(Wr), rnn_row_dtype="bf16")
    compare_draft(gpu_np(out), o, rtol_for("bf16"))
    check_no_error(ws)
print("ok")
"""


@pytest.mark.parametrize("env", [{"DSPARK_DRAFT_PATH": "cuda_core"}, {"DSPARK_DRAFT_LAUNCH": "per_pass"},
                                 {"DSPARK_DRAFT_LAUNCH": "two_pass"},
                                 {"DSPARK_DRAFT_LAUNCH": "two_pass", "DSPARK_RNN_STEP": "cuda_core"},
                                 {"DSPARK_DRAFT_FORM": "wide"}, {"DSPARK_DRAFT_LAUNCH": "fused"}])
def test_rnn_head_on_the_other_launch_paths(env):
    # bf16 tensor-core shapes on the CUDA-core path, with one launch per pass,
    # with one launch per position (the recurrent step between launches, on the
    # tensor cores or on the CUDA cores), a small batch on the 128-row form, and
    # the fused form above 512 requests
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = CHILD.format(root=root, tests=os.path.join(root, "tests"))
    res = subprocess.run([sys.executable, "-c", code], env={**os.environ, **env}, cwd=root,
                         capture_output=True, text=True, timeout=600)
    assert res.returncode == 0 and res.stdout.strip().endswith("ok"), res.stdout[-2000:] + res.stderr[-4000:]
