"""dspark_schedule_noalloc — the scheduler for callers that cannot allocate device
memory (a plug-in inside a host whose pool allocator owns all of the GPU's
memory, or a decode loop that must never call cudaMalloc because it can stall
the device).  Its scratch is a fixed array inside the library instead of a
caller-allocated workspace.

Checked through the C ABI against dspark_schedule, the entry point that takes a
workspace: two different batches, one call each, back to back, then the first
batch again (it must not see what the second one left in the shared array).
The outputs are compared bit for bit, the tolerance the scheduler's parity
tests use.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import synth
from draft_sampling_lossless_markov_gb300 import capi
from draft_sampling_lossless_markov_gb300 import torch_api as T
from gpu_common import require_gpu, to_dev_f32, to_dev_i32, workspace_for

pytestmark = pytest.mark.gpu

OUT_KEYS = ("ell", "offsets", "flat_tok", "mark_req", "mark_pos", "n_verify", "theta_best", "surv")


def _case(B, G, seed):
    rng = np.random.default_rng(seed)
    z = synth.random_conf_logits(B, G, seed)
    return dict(B=B, G=G,
                conf_logit=to_dev_f32(z),
                sts=to_dev_f32(rng.uniform(0.8, 1.5, G)),
                sps=torch.from_numpy(synth.sps_table("exp2048", B, G)).cuda(),
                anchor=to_dev_i32(rng.integers(0, 151936, B)),
                tokens=to_dev_i32(synth.random_tokens(B, G, 151936, seed + 1)))


def _outputs(B, G):
    cap = B * (1 + G)
    i32 = dict(dtype=torch.int32, device="cuda")
    # filled with a sentinel so that an output the call forgot to write shows up
    return dict(ell=torch.full((B,), -7, **i32), offsets=torch.full((B + 1,), -7, **i32),
                flat_tok=torch.full((cap,), -7, **i32), mark_req=torch.full((cap,), -7, **i32),
                mark_pos=torch.full((cap,), -7, **i32), n_verify=torch.full((1,), -7, **i32),
                theta_best=torch.full((1,), -7.0, dtype=torch.float64, device="cuda"),
                surv=torch.full((B, G), -7.0, dtype=torch.float32, device="cuda"))


def _args(c, out):
    a = capi.dspark_sched_args()
    a.B, a.gamma, a.mode = c["B"], c["G"], c.get("mode", capi.DSPARK_SCHED_GREEDY)
    a.conf_logit_prev = c["prev"].data_ptr() if "prev" in c else None
    a.conf_logit, a.sts_temp, a.sps = c["conf_logit"].data_ptr(), c["sts"].data_ptr(), c["sps"].data_ptr()
    a.anchor, a.tokens = c["anchor"].data_ptr(), c["tokens"].data_ptr()
    for k in ("ell", "offsets", "flat_tok", "mark_req", "mark_pos", "n_verify", "theta_best", "surv"):
        setattr(a, k, out[k].data_ptr())
    a.n_verify_host = None
    return a


def _with_workspace(c):
    out = _outputs(c["B"], c["G"])
    ws = workspace_for(c["B"], c["G"], 1, 0, 0, torch.float32)
    st = capi.dspark_schedule(_args(c, out), ws.ptr, ws.nbytes, torch.cuda.current_stream().cuda_stream)
    assert st == capi.DSPARK_OK, capi.dspark_status_string(st)
    torch.cuda.synchronize()
    return out


def _without_workspace(c):
    out = _outputs(c["B"], c["G"])
    st = capi.dspark_schedule_noalloc(_args(c, out), torch.cuda.current_stream().cuda_stream)
    assert st == capi.DSPARK_OK, capi.dspark_status_string(st)
    return out


def _same(a, b):
    for k in OUT_KEYS:
        assert torch.equal(a[k], b[k]), k


def test_noalloc_schedule_matches_workspace_schedule():
    require_gpu()
    c1 = _case(256, 7, 21)      # the benchmark's batch shape
    c2 = _case(4096, 16, 22)    # the largest batch the fixed array holds (65536 candidates)
    ref1, ref2 = _with_workspace(c1), _with_workspace(c2)
    # two calls in a row on the shared array, then the first batch again
    got1 = _without_workspace(c1)
    got2 = _without_workspace(c2)
    got1b = _without_workspace(c1)
    torch.cuda.synchronize()
    _same(ref1, got1)
    _same(ref2, got2)
    _same(ref1, got1b)
    assert int(ref1["n_verify"][0]) > c1["B"]  # the scheduler admitted something: a real comparison


def test_noalloc_schedule_allocates_no_device_memory():
    # the property the entry point exists for: once the library's device code is
    # loaded (the first call), further calls leave the device's free memory and
    # torch's caching allocator untouched
    require_gpu()
    c = _case(256, 7, 41)
    _without_workspace(c)
    torch.cuda.synchronize()
    outs = [_outputs(c["B"], c["G"]) for _ in range(3)]  # every tensor allocated before the calls
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    stats0 = torch.cuda.memory_stats()
    for out in outs:
        st = capi.dspark_schedule_noalloc(_args(c, out), torch.cuda.current_stream().cuda_stream)
        assert st == capi.DSPARK_OK, capi.dspark_status_string(st)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    stats1 = torch.cuda.memory_stats()
    assert free1 == free0
    for k in ("allocation.all.allocated", "segment.all.allocated", "allocated_bytes.all.allocated"):
        assert stats1.get(k, 0) == stats0.get(k, 0), k
    _same(outs[0], outs[2])


def test_noalloc_schedule_rejects_batches_beyond_the_array():
    require_gpu()
    a = capi.dspark_sched_args()
    a.B, a.gamma, a.mode = 4097, 16, capi.DSPARK_SCHED_GREEDY  # 65552 candidates > 65536
    assert capi.dspark_schedule_noalloc(a, 0) == capi.DSPARK_UNSUPPORTED


def test_noalloc_schedule_in_the_asynchronous_mode():
    # the production variant through the fixed array: capacity from earlier confidences
    require_gpu()
    c = _case(256, 7, 31)
    c["mode"] = capi.DSPARK_SCHED_ASYNC_TOPK
    c["prev"] = to_dev_f32(synth.random_conf_logits(256, 7, 32))
    ref = _with_workspace(c)
    got = _without_workspace(c)
    torch.cuda.synchronize()
    _same(ref, got)
