"""GPU parity of dspark_draft_sample against the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import synth
from oracle.draft import draft as oracle_draft
from parity import compare_draft, gpu_np, np_inputs, rtol_for
from gpu_common import check_no_error, gpu_draft, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _invariants(g, V):
    # p_d(x_k) is the row entry at the drawn token, bit for bit; rows are distributions
    B, G = g["tokens"].shape
    assert g["tokens"].min() >= 0 and g["tokens"].max() < V
    rows = g["pd_rows"]
    pick = np.take_along_axis(rows, g["tokens"][:, :, None].astype(np.int64), axis=2)[:, :, 0]
    np.testing.assert_array_equal(pick, g["pd_tok"])
    np.testing.assert_allclose(rows.sum(axis=2), 1.0, rtol=0, atol=5e-5)


@pytest.mark.parametrize("temp", ["mixed", "0", "1.0", "0.7"])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_draft_tiny(temp, seed):
    wl = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(wl, "cuda", seed=seed, temp=temp)
    out, ws = gpu_draft(inp)
    g = gpu_np(out)
    _invariants(g, wl.V)
    o = oracle_draft(**np_inputs(inp))
    st = compare_draft(g, o, rtol_for(wl.dtype))
    assert st["n_tokens_compared"] >= 0.5 * wl.B * wl.gamma
    check_no_error(ws)


@pytest.mark.parametrize("B,G,V,r,H,dt", [
    (1, 1, 7, 0, 0, "f32"),        # tiny vocabulary, no head, no hidden
    (3, 5, 1000, 16, 40, "f32"),   # vocabulary not a multiple of the tile width
    (17, 3, 1031, 7, 5, "f32"),    # odd sizes everywhere
    (5, 4, 4104, 64, 24, "bf16"),  # several tiles plus a ragged tail, bf16
    (33, 2, 2056, 1, 8, "bf16"),   # rank 1, more rows than one row block
    # tensor-core shapes (bf16, r a multiple of 64, V and H multiples of 8)
    (130, 5, 8200, 128, 16, "bf16"),   # two M-tiles (the second with 2 rows), an 8-column last tile
    (40, 3, 1024, 256, 8, "bf16"),     # 8 vocabulary tiles for many CTAs: most claim no tile
    (260, 16, 2048, 192, 32, "bf16"),  # gamma 16, rank 192, three M-tiles
    # small batches on the tensor-core path (the vocabulary on the MMA's M side)
    (1, 3, 8200, 256, 16, "bf16"),     # one row, an 8-column last tile
    (2, 5, 1032, 128, 32, "bf16"),     # two rows, rank 128, 9 tiles
    (3, 4, 4104, 64, 24, "bf16"),      # three rows, rank 64
    (4, 7, 16384, 256, 64, "bf16"),    # four rows
])
def test_draft_ragged_shapes(B, G, V, r, H, dt):
    wl = synth.Workload("ragged", B, G, V, H, r, dt, "mixed", synth.SCHED_GREEDY, "tiny", seed=5)
    inp = synth.make_inputs(wl, "cuda", with_target=False)
    out, ws = gpu_draft(inp)
    g = gpu_np(out)
    _invariants(g, V)
    o = oracle_draft(**np_inputs(inp))
    compare_draft(g, o, rtol_for(dt))
    check_no_error(ws)


@pytest.mark.parametrize("temp", ["0", "1.0", "0.7", "mixed"])
@pytest.mark.parametrize("B,G,V,r,H", [
    (1, 4, 8200, 256, 16),     # one request, an 8-column last tile
    (5, 4, 8200, 256, 16),
    (16, 4, 8200, 256, 16),    # the largest batch of the small-batch form
    (16, 16, 2048, 192, 32),   # gamma 16, rank 192 (three K blocks)
    (9, 3, 1032, 64, 8),       # rank 64, 9 tiles for 152 CTAs
    (17, 3, 4104, 128, 24),    # one past the small-batch form: the 128-row tile
])
def test_draft_small_batch_form(B, G, V, r, H, temp):
    # small batches put the vocabulary on the MMA's M side (the batch is N = 16)
    wl = synth.Workload("small", B, G, V, H, r, "bf16", temp, synth.SCHED_GREEDY, "tiny", seed=13)
    inp = synth.make_inputs(wl, "cuda", with_target=False)
    out, ws = gpu_draft(inp)
    g = gpu_np(out)
    _invariants(g, V)
    o = oracle_draft(**np_inputs(inp))
    compare_draft(g, o, rtol_for("bf16"))
    check_no_error(ws)


@pytest.mark.parametrize("temp", ["1.0", "mixed"])
def test_rank_zero_against_the_oracles_rank_zero_path(temp):
    # rank 0 (no Markov bias, the DFlash mode): the oracle's own r = 0 path, whose
    # reduction to softmax(U / T) is pinned on the CPU
    wl = synth.Workload("dflash", 6, 3, 3000, 32, 0, "bf16", temp, synth.SCHED_GREEDY, "tiny", seed=9)
    inp = synth.make_inputs(wl, "cuda", with_target=False)
    out, ws = gpu_draft(inp)
    g = gpu_np(out)
    _invariants(g, wl.V)
    o = oracle_draft(**np_inputs(inp))
    assert o["pd"].shape == g["pd_rows"].shape
    st = compare_draft(g, o, rtol_for(wl.dtype))
    assert st["n_tokens_compared"] >= wl.B
    check_no_error(ws)


@pytest.mark.parametrize("name,subset", [
    ("qwen3_4b", [0, 1, 31, 63]),
    ("sweep_B256_g7", [0, 100, 255]),
    ("deepseek_vocab", [0, 1, 512, 1023]),
])
def test_draft_full_size_sampled_requests(name, subset):
    # the full batch runs on the GPU in the benchmark's launch configuration; the
    # oracle recomputes a few requests one by one (draws are keyed by request id)
    wl = synth.get_workload(name)
    inp = synth.make_inputs(wl, "cuda", with_target=False)
    out, ws = gpu_draft(inp)
    idx = torch.tensor(subset, device="cuda")
    g = {k: v.index_select(0, idx).cpu().numpy() for k, v in out.items()}
    _invariants(g, wl.V)
    o = oracle_draft(**np_inputs(inp, idx))
    compare_draft(g, o, rtol_for(wl.dtype))
    # whole-batch properties
    tok = out["tokens"]
    assert int(tok.min()) >= 0 and int(tok.max()) < wl.V
    s = out["pd_rows"].sum(dim=2)
    assert float((s - 1).abs().max()) < 5e-4
    c = out["conf"]
    assert float(c.min()) >= 0 and float(c.max()) <= 1  # fp32 sigmoid saturates to 1 for z > ~17
    check_no_error(ws)


def test_bad_anchor_is_reported_and_replaced():
    wl = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(wl, "cuda", temp="1.0")
    inp["anchor"][2] = wl.V + 5
    out, ws = gpu_draft(inp)
    code, detail = ws.read_error()
    assert code == 5 and detail == wl.V + 5  # DSPARK_BAD_INPUT
    inp2 = dict(inp)
    inp2["anchor"] = inp["anchor"].clone()
    inp2["anchor"][2] = 0
    o = oracle_draft(**np_inputs(inp2))
    compare_draft(gpu_np(out), o, rtol_for(wl.dtype))
    check_no_error(ws)  # read_error cleared the word


def test_repeat_calls_are_deterministic():
    wl = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(wl, "cuda", temp="mixed")
    a, ws = gpu_draft(inp)
    a = {k: v.clone() for k, v in a.items()}
    b, _ = gpu_draft(inp, ws)
    for k in a:
        assert torch.equal(a[k], b[k]), k
