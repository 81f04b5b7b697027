"""dspark_draft_and_schedule: the draft and the schedule in one call, the
scheduler running beside the draft kernel's last sweep where it can (either
fused tensor-core form with p_d rows and a schedule that fits one CTA's shared
memory), else one after the other.  Every output must equal, bit for bit, what dspark_draft_sample followed
by dspark_schedule give on the same inputs (both checked against the oracle
elsewhere); the schedule is also compared with the oracle's scheduler run on
the GPU's own confidences and tokens."""
import numpy as np
import pytest
import torch

import synth
from oracle import schedule as S
from parity import compare_schedule, gpu_np
from gpu_common import check_no_error, require_gpu, workspace_for
from draft_sampling_lossless_markov_gb300 import torch_api as T

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


# B, gamma, V, r, H, dtype, head, scheduler mode: which path the call takes
CASES = [
    (256, 7, 8200, 256, 16, "bf16", "markov", synth.SCHED_GREEDY),       # overlapped, two M-tiles
    (130, 5, 8200, 128, 16, "bf16", "markov", synth.SCHED_GREEDY),       # overlapped, ragged M-tile
    (300, 6, 4104, 192, 8, "bf16", "markov", synth.SCHED_GREEDY),        # overlapped, three M-tiles
    (64, 7, 4104, 64, 8, "bf16", "markov", synth.SCHED_ASYNC_TOPK),      # overlapped, asynchronous scheduler
    (200, 4, 8200, 128, 8, "bf16", "rnn", synth.SCHED_GREEDY),           # overlapped, RNN head in the fused form
    (256, 7, 8200, 256, 16, "bf16", "markov", synth.SCHED_OFF),          # overlapped, scheduler off
    (8, 4, 8200, 256, 16, "bf16", "markov", synth.SCHED_GREEDY),         # overlapped, small-batch form
    (1, 7, 8200, 256, 16, "bf16", "markov", synth.SCHED_GREEDY),         # overlapped, small-batch form, one request
    (12, 3, 4104, 128, 8, "bf16", "rnn", synth.SCHED_GREEDY),            # overlapped, small-batch RNN form
    (600, 4, 4104, 128, 8, "bf16", "markov", synth.SCHED_GREEDY),        # overlapped, 2400 candidates
    (1024, 7, 2056, 64, 8, "bf16", "markov", synth.SCHED_GREEDY),        # overlapped, 8192 slots (the keys
                                                                         # calibrated in the one CTA)
    (1100, 8, 2056, 64, 8, "bf16", "markov", synth.SCHED_GREEDY),        # overlapped, 16384 slots: the radix
                                                                         # kernel forming its own keys
    (2100, 16, 1000, 64, 8, "bf16", "markov", synth.SCHED_GREEDY),       # overlapped, 33600 candidates
    (1100, 8, 2056, 64, 8, "bf16", "markov", synth.SCHED_OFF),           # overlapped, radix kernel, scheduler off
    (40, 3, 1000, 16, 8, "f32", "markov", synth.SCHED_GREEDY),           # CUDA-core path: in sequence
]


def _run(inp, head, Wr, zprev, mode, combined):
    B, G, V = inp["U"].shape
    ws = workspace_for(B, G, V, inp["W1"].shape[1], inp["h"].shape[2], inp["U"].dtype)
    args = (inp["U"], inp["W1"], inp["W2"], inp["h"], inp["w"], inp["anchor"], inp["temp"], inp["req_id"],
            inp["seed"])
    kw = dict(W_rnn=Wr if head == "rnn" else None)
    zp = torch.from_numpy(zprev).cuda() if mode == synth.SCHED_ASYNC_TOPK else None
    if combined:
        d, s = T.draft_and_schedule(ws, *args, inp["sts"], inp["sps"], mode, want_surv=True, conf_logit_prev=zp,
                                    **kw)
    else:
        d = T.draft_sample(ws, *args, **kw)
        s = T.schedule(ws, d["conf_logit"], inp["sts"], inp["sps"], inp["anchor"], d["tokens"], mode,
                       want_surv=True, conf_logit_prev=zp)
    torch.cuda.synchronize()
    check_no_error(ws)
    return gpu_np(d), {k: v for k, v in gpu_np(s).items() if not k.startswith("_")}


@pytest.mark.parametrize("B,G,V,r,H,dtype,head,mode", CASES)
def test_draft_and_schedule_equals_the_two_calls(B, G, V, r, H, dtype, head, mode):
    wl = synth.Workload("ds", B, G, V, H, r, dtype, "mixed", mode, "tiny", seed=B + G)
    inp = synth.make_inputs(wl, "cuda", with_target=False)
    Wr = synth.rnn_weights(r, H, dtype, B, "cuda") if head == "rnn" else None
    zprev = synth.random_conf_logits(B, G, 700 + B)
    d1, s1 = _run(inp, head, Wr, zprev, mode, combined=False)
    d2, s2 = _run(inp, head, Wr, zprev, mode, combined=True)
    for k in d1:
        np.testing.assert_array_equal(d2[k], d1[k], err_msg=f"draft {k}")
    for k in s1:
        np.testing.assert_array_equal(s2[k], s1[k], err_msg=f"schedule {k}")
    # the schedule against the oracle's, on the GPU's confidences and tokens
    osch = S.schedule(d2["conf_logit"].astype(np.float32), inp["sts"].cpu().numpy(), inp["sps"],
                      inp["anchor"].cpu().numpy(), d2["tokens"], mode=mode,
                      conf_logit_prev=zprev if mode == synth.SCHED_ASYNC_TOPK else None)
    np.testing.assert_array_equal(s2["surv"], osch["a"])  # fp32 survival products, bit for bit
    compare_schedule(s2, osch, surv_equal=True)


def test_draft_and_schedule_repeated_on_one_workspace():
    # back-to-back combined calls on one stream and workspace: the counters the
    # overlap uses are reset by each call, and the results do not drift
    wl = synth.Workload("ds", 256, 7, 8200, 16, 256, "bf16", "1.0", synth.SCHED_GREEDY, "tiny", seed=3)
    inp = synth.make_inputs(wl, "cuda", with_target=False)
    ws = workspace_for(256, 7, 8200, 256, 16, inp["U"].dtype)
    args = (inp["U"], inp["W1"], inp["W2"], inp["h"], inp["w"], inp["anchor"], inp["temp"], inp["req_id"],
            inp["seed"])
    first = None
    for _ in range(4):
        d, s = T.draft_and_schedule(ws, *args, inp["sts"], inp["sps"], synth.SCHED_GREEDY)
        torch.cuda.synchronize()
        got = (d["tokens"].cpu().numpy(), s["ell"].cpu().numpy(), s["flat_tok"].cpu().numpy())
        if first is None:
            first = got
        for a, b in zip(got, first):
            np.testing.assert_array_equal(a, b)
    check_no_error(ws)


@pytest.mark.parametrize("B,G", [(256, 7), (8, 4)])
def test_draft_and_schedule_in_a_cuda_graph(B, G):
    # the call captured into a CUDA graph (the programmatic dependency becomes a
    # graph edge) and replayed: the same outputs as the eager call
    wl = synth.Workload("ds", B, G, 8200, 16, 256, "bf16", "mixed", synth.SCHED_GREEDY, "tiny", seed=7)
    inp = synth.make_inputs(wl, "cuda", with_target=False)
    ws = workspace_for(B, G, 8200, 256, 16, inp["U"].dtype)
    sps = torch.from_numpy(np.ascontiguousarray(inp["sps"], dtype=np.float64)).cuda()
    args = (inp["U"], inp["W1"], inp["W2"], inp["h"], inp["w"], inp["anchor"], inp["temp"], inp["req_id"],
            inp["seed"])
    d0, s0 = T.draft_and_schedule(ws, *args, inp["sts"], sps, synth.SCHED_GREEDY)
    torch.cuda.synchronize()
    ref = {k: v.clone() for k, v in list(d0.items()) + [("s_" + k, v) for k, v in s0.items() if not k.startswith("_")]}
    st = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        T.draft_and_schedule(ws, *args, inp["sts"], sps, synth.SCHED_GREEDY, out=d0, sched_out=s0, stream=st)
    st.synchronize()
    with torch.cuda.graph(g, stream=st):
        T.draft_and_schedule(ws, *args, inp["sts"], sps, synth.SCHED_GREEDY, out=d0, sched_out=s0,
                             stream=torch.cuda.current_stream())
    for _ in range(2):
        for v in list(d0.values()) + [v for k, v in s0.items() if not k.startswith("_")]:
            v.fill_(-7) if v.dtype != torch.float64 else v.fill_(-7.0)
        g.replay()
        st.synchronize()
        for k, v in d0.items():
            assert torch.equal(v, ref[k]), k
        for k, v in s0.items():
            if not k.startswith("_"):
                assert torch.equal(v, ref["s_" + k]), k
    check_no_error(ws)
