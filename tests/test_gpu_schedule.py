"""GPU parity of dspark_schedule against the oracle (bit-exact integer outputs)."""
import os

import numpy as np
import pytest
import torch

import synth
from oracle import schedule as S
from parity import compare_schedule
from gpu_common import check_no_error, require_gpu, to_dev_f32, to_dev_i32, workspace_for
from draft_sampling_lossless_markov_gb300 import torch_api as T

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _run(z, tau, sps, anchor, tokens, mode):
    B, G = z.shape
    ws = workspace_for(B, G, 1, 0, 0, torch.float32)
    host = torch.zeros(1, dtype=torch.int32).pin_memory()
    out = T.schedule(ws, to_dev_f32(z), to_dev_f32(tau), sps, to_dev_i32(anchor), to_dev_i32(tokens), mode,
                     n_verify_host=host, want_surv=True)
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in out.items() if isinstance(v, torch.Tensor) and k != "_sps"}
    g["n_verify_host"] = int(host[0])
    check_no_error(ws)
    return g


def _oracle(z, tau, sps, anchor, tokens, mode):
    return S.schedule(z, tau, sps, anchor, tokens, mode=mode)


def _case(seed, B, G, sps_kind="exp2048", z_scale=2.5, z_shift=0.5, tau=None):
    rng = np.random.default_rng(seed)
    z = synth.random_conf_logits(B, G, seed, scale=z_scale, shift=z_shift)
    if tau is None:
        tau = np.ones(G, np.float32)
    sps = synth.sps_table(sps_kind, B, G) if sps_kind in ("tiny", "exp2048") else sps_kind
    anchor = rng.integers(0, 1000, B).astype(np.int32)
    tokens = synth.random_tokens(B, G, 1000, seed + 1)
    return z, np.asarray(tau, np.float32), sps, anchor, tokens


def _check(z, tau, sps, anchor, tokens, mode):
    g = _run(z, tau, sps, anchor, tokens, mode)
    o = _oracle(z, tau, sps, anchor, tokens, mode)
    np.testing.assert_array_equal(g["surv"], o["a"])  # fp32 survival products, bit for bit
    compared = compare_schedule(g, o, surv_equal=True)
    assert g["n_verify_host"] == int(o["offsets"][-1]) or not compared
    return compared, g, o


@pytest.mark.parametrize("seed", range(12))
def test_schedule_random_small(seed):
    rng = np.random.default_rng(100 + seed)
    B, G = int(rng.integers(1, 40)), int(rng.integers(1, 9))
    tau = rng.uniform(0.8, 1.5, G).astype(np.float32)
    kind = ["tiny", "exp2048"][seed % 2]
    n = np.arange(B * (1 + G) + 1, dtype=np.float64)
    if seed % 3 == 2:  # stepped cost table with cliffs
        kind = 100.0 / (1.0 + np.floor(n / 3) * 0.05)
    z = synth.random_conf_logits(B, G, seed)
    sps = synth.sps_table(kind, B, G) if isinstance(kind, str) else kind
    compared, g, o = _check(z, tau, sps, rng.integers(0, 1000, B), synth.random_tokens(B, G, 1000, seed), 1)
    assert compared


@pytest.mark.parametrize("B,G", [(256, 15), (256, 7), (1024, 7), (4096, 16), (65536, 1),
                                 (2500, 2), (3000, 1)])
def test_schedule_workload_sizes(B, G):
    # up to the 65536-candidate limit; config-2 STS temperatures and SPS curve.
    # B2500 gamma2 and B3000 gamma1 take the shared-memory merge with 8 and 4
    # outputs per thread over runs of 2 and 1 slots (a thread's outputs span
    # several run pairs in the first passes)
    rng = np.random.default_rng(B + G)
    tau = rng.uniform(0.8, 1.5, G).astype(np.float32)
    z, _, sps, anchor, tokens = _case(B * 7 + G, B, G)
    compared, g, o = _check(z, tau, sps, anchor, tokens, 1)
    assert compared
    assert 0 <= g["ell"].min() and g["ell"].max() <= G


def test_schedule_survival_sums_past_2048():
    # confident drafts at B1024 gamma8 (8192 slots, the shared-memory path): the
    # admitted survival products sum to about 7300, past 2^11, where a sum with
    # 52 fraction bits would no longer fit a signed 64-bit integer
    B, G = 1024, 8
    z, tau, sps, anchor, tokens = _case(21, B, G, z_scale=0.5, z_shift=4.0)
    compared, g, o = _check(z, tau, sps, anchor, tokens, 1)
    assert compared
    assert int(g["ell"].sum()) > 7000 and float(o["a"][o["a"] > 0].sum()) > 4096


def test_schedule_off_mode():
    z, tau, sps, anchor, tokens = _case(3, 50, 6)
    compared, g, o = _check(z, tau, None, anchor, tokens, 0)
    assert compared and np.all(g["ell"] == 6) and g["n_verify"][0] == 50 * 7


def test_schedule_all_survival_zero():
    z, tau, sps, anchor, tokens = _case(4, 20, 5)
    z[:] = -1.0e4  # sigmoid underflows: c' = 0, no candidate
    compared, g, o = _check(z, tau, sps, anchor, tokens, 1)
    assert compared and np.all(g["ell"] == 0) and g["n_verify"][0] == 20


def test_schedule_always_improving_admits_everything():
    B, G = 30, 4
    z, tau, _, anchor, tokens = _case(5, B, G)
    sps = np.ones(B * (1 + G) + 1)  # flat cost: every candidate with a > 0 raises Theta
    compared, g, o = _check(z, tau, sps, anchor, tokens, 1)
    assert compared and np.all(g["ell"] == G)


def test_schedule_ties_break_by_request_then_position():
    B, G = 64, 4
    z = np.full((B, G), 1.25, np.float32)  # every request identical
    tau = np.ones(G, np.float32)
    sps = synth.sps_table("exp2048", B, G) * 0 + 100.0 / (1.0 + np.arange(B * (1 + G) + 1) / 40.0)
    anchor = np.arange(B, dtype=np.int32)
    tokens = synth.random_tokens(B, G, 50, 3)
    compared, g, o = _check(z, tau, sps, anchor, tokens, 1)
    assert compared
    # lengths differ by at most one and longer requests come first
    assert g["ell"].max() - g["ell"].min() <= 1
    assert np.all(np.diff(g["ell"]) <= 0)


def test_schedule_appendix_a_on_gpu():
    # [DSpark] 附录 (Appendix A): R = 1, a1 = 0.8, SPS(1..3) = 1.0, 0.5, 0.45 -> l = 0
    golden = {}
    for line in open(os.path.join(os.path.dirname(__file__), "golden", "appendix_a_counterexample.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            golden[k] = float(v)
    z1 = np.float32(np.log(golden["a1"] / (1 - golden["a1"])))
    for c2 in (golden["c2_high"], 0.5):
        z2 = np.float32(np.log(c2 / (1 - c2)))
        z = np.array([[z1, z2]], np.float32)
        sps = np.array([0.0, golden["sps1"], golden["sps2"], golden["sps3"]])
        compared, g, o = _check(z, np.ones(2, np.float32), sps, np.array([1]), np.array([[2, 3]]), 1)
        assert compared
        assert g["ell"][0] == golden["early_stop_ell"]
        assert g["theta_best"][0] == pytest.approx(golden["theta0"], rel=1e-6)


def test_schedule_empty_batch_is_a_no_op():
    ws = workspace_for(1, 2, 1, 0, 0, torch.float32)
    from draft_sampling_lossless_markov_gb300 import capi
    a = capi.dspark_sched_args()
    a.B, a.gamma, a.mode = 0, 2, 1
    assert capi.dspark_schedule(a, ws.ptr, ws.nbytes, 0) == capi.DSPARK_OK


# ---- the asynchronous production mode ----

def _run_async(z, zp, tau, sps, anchor, tokens):
    B, G = z.shape
    ws = workspace_for(B, G, 1, 0, 0, torch.float32)
    out = T.schedule(ws, to_dev_f32(z), to_dev_f32(tau), sps, to_dev_i32(anchor), to_dev_i32(tokens),
                     S.MODE_ASYNC_TOPK, want_surv=True, conf_logit_prev=to_dev_f32(zp))
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in out.items() if isinstance(v, torch.Tensor) and k != "_sps"}
    check_no_error(ws)
    return g


def _check_async(z, zp, tau, sps, anchor, tokens):
    g = _run_async(z, zp, tau, sps, anchor, tokens)
    o = S.schedule(z, tau, sps, anchor, tokens, mode=S.MODE_ASYNC_TOPK, conf_logit_prev=zp)
    np.testing.assert_array_equal(g["surv"], o["a"])
    if o["cap_margin"] <= 1e-12:  # the capacity's argmax is a near tie: exempt
        return False, g, o
    return compare_schedule(g, o, surv_equal=True), g, o


@pytest.mark.parametrize("seed", range(12))
def test_schedule_async_random_small(seed):
    rng = np.random.default_rng(300 + seed)
    B, G = int(rng.integers(1, 40)), int(rng.integers(1, 9))
    tau = rng.uniform(0.8, 1.5, G).astype(np.float32)
    n = np.arange(B * (1 + G) + 1, dtype=np.float64)
    kind = ["tiny", "exp2048"][seed % 2]
    sps = synth.sps_table(kind, B, G) if seed % 3 != 2 else 100.0 / (1.0 + np.floor(n / 3) * 0.05)
    z = synth.random_conf_logits(B, G, seed)
    zp = synth.random_conf_logits(B, G, seed + 1000)
    compared, g, o = _check_async(z, zp, tau, sps, rng.integers(0, 1000, B), synth.random_tokens(B, G, 1000, seed))
    assert compared


@pytest.mark.parametrize("B,G", [(256, 7), (256, 15), (1024, 7), (64, 32)])
def test_schedule_async_workload_sizes(B, G):
    rng = np.random.default_rng(B * 3 + G)
    tau = rng.uniform(0.8, 1.5, G).astype(np.float32)
    z, _, sps, anchor, tokens = _case(B * 11 + G, B, G)
    zp = synth.random_conf_logits(B, G, B * 13 + G, scale=2.5, shift=0.5)
    compared, g, o = _check_async(z, zp, tau, sps, anchor, tokens)
    assert compared
    assert int(g["ell"].sum()) == o["n_admit"] <= o["K"]


def test_schedule_async_same_confidences_is_the_global_search():
    # earlier = current confidences on a stepped cost table: the admission is the
    # best prefix of the whole path, past the first local maximum
    B, G = 40, 6
    z, tau, _, anchor, tokens = _case(77, B, G)
    n = np.arange(B * (1 + G) + 1, dtype=np.float64)
    sps = 100.0 / (1.0 + np.floor(n / 4) * 0.08)
    compared, g, o = _check_async(z, z, tau, sps, anchor, tokens)
    assert compared
    full = S.prefix_schedule(o["a"], sps, S.MODE_GREEDY, early_stop=False)
    np.testing.assert_array_equal(g["ell"], full["ell"])


def test_schedule_async_unsupported_beyond_shared_memory():
    B, G = 4096, 7
    z, tau, sps, anchor, tokens = _case(5, B, G)
    with pytest.raises(Exception, match="UNSUPPORTED|unsupported|2"):
        _run_async(z, z, tau, sps, anchor, tokens)
