#!/usr/bin/env python
"""Benchmark of one DSpark decode step on GB300: draft sample + schedule + verify.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints ONE JSON line (rank 0).  A step is dspark_draft_sample + dspark_schedule
+ dspark_verify over one batch of synthetic inputs (seeded; the shapes and value
model of the DSpark pages' workloads).  The target model's forward on the
flattened verify batch is not part of the path: a gather of synthetic target
rows stands in for it and is excluded from the timed region (CUDA events around
the two timed segments of every step).  Inputs (U alone is B*gamma*V*2 bytes,
545 MB at the headline point) are larger than the 129 MB L2, so no flush is
needed between steps.

metric: request-positions/s = B * gamma / t_step, and the step's % of the HBM
roofline.  --impl reference times the fp64 CPU oracle on the host cores instead
(a bounded sample of the same workload, extrapolated per request).

--workload sts_small | sts_N131072_g7_G128_M15 times dspark_sts_fit instead
(fitting the STS temperatures on a held-out set): metric = sigmoid evaluations
per second (every block x candidate x position), roofline against the fp32
issue rate, L2 flushed between fits.

Multi-GPU (torchrun, one rank per GPU): the path shards by request with no
exchange except the scheduler; this benchmark runs independent replicas (weak
scaling), barrier + max-over-ranks timing.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

os.environ.setdefault("OMP_NUM_THREADS", "1")
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# synth (and with it torch) is imported inside the functions that use it: the
# oracle's worker processes start by re-importing this file and need numpy only

METRIC = "spec-decode request-positions/s (draft+schedule+verify) at V=151936; % HBM peak"
UNIT = "request-positions/s"


# ---------------------------------------------------------------------------
# byte model (algorithmic bytes of one step; every figure counted once)
# ---------------------------------------------------------------------------
def step_bytes(wl: synth.Workload, n_verify_rows: int, pd_rows: bool = True) -> dict:
    """Without p_d rows the draft writes none and the final draw re-reads only the
    target row (p_d is recomputed at a few proposed tokens)."""
    e = 2 if wl.dtype == "bf16" else 4
    B, G, V, r, H = wl.B, wl.gamma, wl.V, wl.r, wl.H
    U = B * G * V * e
    W2_strict = r * V * e
    W2_per_pos = G * r * V * e
    pd = B * G * V * 4 if pd_rows else 0
    target = n_verify_rows * V * e
    resid = B * V * (e + 4) if pd_rows else B * V * e
    small = B * G * (r * e + H * e + 24)
    draft_small = B * G * (r * e + H * e + 16)
    draft_strict = U + W2_strict + pd + draft_small
    return dict(U=U, W2_strict=W2_strict, W2_per_position=W2_per_pos, pd=pd, target=target, resid=resid,
                small=small, step_strict=U + W2_strict + pd + target + resid + small,
                step_per_position=U + W2_per_pos + pd + target + resid + small, draft_strict=draft_strict,
                draft_per_position=U + W2_per_pos + pd + draft_small)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except (FileNotFoundError, OSError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.th.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# multi-rank timing: every rank times its own replica, the slowest one counts
# ---------------------------------------------------------------------------
def max_over_ranks(ms: float, world: int, device) -> float:
    """The largest per-rank step time (the job's step time), then a barrier."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t[0])


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def run_ours(args, rank, world, local_rank):
    import synth
    import torch
    from draft_sampling_lossless_markov_gb300 import build, capi
    from draft_sampling_lossless_markov_gb300 import torch_api as T

    build.build()
    capi.load()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = synth.get_workload(args.workload)
    B, G, V = wl.B, wl.gamma, wl.V
    inp = synth.make_inputs(wl, dev)
    inp["sched_mode"], inp["zprev"] = wl.sched, None
    if args.sched == "async":
        # the production mode: capacity from synthetic confidences of an earlier step
        inp["sched_mode"] = synth.SCHED_ASYNC_TOPK
        inp["zprev"] = torch.from_numpy(synth.random_conf_logits(B, G, wl.seed + 77)).to(dev)
    if args.head == "rnn":
        # the optional RNN sequential head (fp32 recurrent rows, CUDA-core bias product)
        inp["W_rnn"] = synth.rnn_weights(wl.r, wl.H, wl.dtype, wl.seed, dev)
    ws = T.Workspace.create(T.dims(B, G, V, wl.r, wl.H, inp["U"].dtype), device=dev)
    cap = B * (G + 1)
    sps_dev = torch.from_numpy(inp["sps"]).to(dev)
    stream = torch.cuda.Stream(device=dev)
    # outputs (allocated once)
    row_free = args.rows == "none"
    d_out = dict(tokens=torch.empty((B, G), dtype=torch.int32, device=dev),
                 pd_tok=torch.empty((B, G), dtype=torch.float32, device=dev),
                 conf_logit=torch.empty((B, G), dtype=torch.float32, device=dev),
                 conf=torch.empty((B, G), dtype=torch.float32, device=dev))
    if row_free:
        # no p_d rows: the select's (max, sum) per row; verify draws the residual by
        # rejection from p_t, recomputing p_d at the proposed tokens
        d_out["pd_stat"] = torch.empty((B, G, 2), dtype=torch.float32, device=dev)
    else:
        d_out["pd_rows"] = torch.empty((B, G, V), dtype=torch.float32, device=dev)
    rej = (dict(U=inp["U"], W1=inp["W1"], W2=inp["W2"], anchor=inp["anchor"], pd_stat=d_out["pd_stat"])
           if row_free else None)
    s_out = dict(ell=torch.empty(B, dtype=torch.int32, device=dev),
                 offsets=torch.empty(B + 1, dtype=torch.int32, device=dev),
                 flat_tok=torch.empty(cap, dtype=torch.int32, device=dev),
                 mark_req=torch.empty(cap, dtype=torch.int32, device=dev),
                 mark_pos=torch.empty(cap, dtype=torch.int32, device=dev),
                 n_verify=torch.empty(1, dtype=torch.int32, device=dev),
                 theta_best=torch.empty(1, dtype=torch.float64, device=dev))
    v_out = dict(n_accept=torch.empty(B, dtype=torch.int32, device=dev),
                 out_tok=torch.empty((B, G + 1), dtype=torch.int32, device=dev),
                 n_out=torch.empty(B, dtype=torch.int32, device=dev))
    rows = torch.empty((cap, V), dtype=inp["U"].dtype, device=dev)
    tgt_flat = inp["target"].reshape(-1, V)

    overlap = sched_overlaps(wl, args)

    def draft_call(st):
        if overlap:
            # dspark_draft_and_schedule: the scheduler beside the draft's last sweep
            draft_and_sched(T, ws, inp, inp["U"], inp["h"], inp["anchor"], inp["temp"], inp["req_id"], sps_dev,
                            d_out, s_out, st, rows=not row_free)
        else:
            T.draft_sample(ws, inp["U"], inp["W1"], inp["W2"], inp["h"], inp["w"], inp["anchor"], inp["temp"],
                           inp["req_id"], inp["seed"], out=d_out, stream=st, W_rnn=inp.get("W_rnn"))

    def sched_call(st):
        if not overlap:
            sched(T, ws, d_out["conf_logit"], inp, sps_dev, inp["anchor"], d_out["tokens"], out=s_out, stream=st)

    def standin(st):
        # stand-in for the target forward on the flattened batch (not timed): the
        # kept rows of the synthetic target logits, packed by the marker tensor
        T.pack_rows(inp["target"], s_out["mark_req"], s_out["mark_pos"], s_out["n_verify"], rows, ws, stream=st)

    cap_accept = args.verify == "cap_accept"
    if cap_accept:
        # cap-accept: every request's whole block is verified (its gamma+1 rows in
        # place), the scheduler's lengths are the committed windows
        full_offsets = (torch.arange(B + 1, device=dev, dtype=torch.int32) * (G + 1)).contiguous()
        full_ell = torch.full((B,), G, dtype=torch.int32, device=dev)

    def verify_call(st):
        if cap_accept:
            T.verify(ws, tgt_flat, full_offsets, full_ell, d_out["tokens"], d_out.get("pd_rows"), d_out["pd_tok"],
                     inp["temp"], inp["req_id"], inp["seed"], out=v_out, stream=st, commit_cap=s_out["ell"],
                     rejection=rej)
        else:
            T.verify(ws, rows, s_out["offsets"], s_out["ell"], d_out["tokens"], d_out.get("pd_rows"),
                     d_out["pd_tok"], inp["temp"], inp["req_id"], inp["seed"], out=v_out, stream=st, rejection=rej)

    calls = (draft_call, sched_call, verify_call)
    use_graph = not args.no_graph
    n0 = capi.dspark_launch_count()
    with torch.cuda.stream(stream):
        draft_call(stream)
        sched_call(stream)
        standin(stream)
        verify_call(stream)
    stream.synchronize()
    launches_per_step = capi.dspark_launch_count() - n0
    if use_graph:
        # one graph per call, so that CUDA events between the replays time each
        # call live inside the timed region
        runs = []
        for fn in calls:
            if fn is sched_call and overlap:
                runs.append(lambda: None)  # the schedule runs inside the draft call
                continue
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn(torch.cuda.current_stream())
            runs.append(g.replay)
    else:
        runs = [lambda fn=fn: fn(stream) for fn in calls]

    def one_step(ev=None):
        # events: 0 | draft | 1 | schedule | 2 | (stand-in, not timed) | 3 | verify | 4
        with torch.cuda.stream(stream):
            if ev:
                ev[0].record(stream)
            runs[0]()
            if ev:
                ev[1].record(stream)
            runs[1]()
            if ev:
                ev[2].record(stream)
            standin(stream)
            if ev:
                ev[3].record(stream)
            runs[2]()
            if ev:
                ev[4].record(stream)

    for _ in range(args.warmup):
        one_step()
    stream.synchronize()

    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    cvd = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    clocks = ClockSampler(cvd[local_rank] if local_rank < len(cvd) else local_rank)
    clocks.start()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    for k in range(args.steps):
        one_step(evs[k])
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    per = np.array([[e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2]), e[3].elapsed_time(e[4])] for e in evs])
    ms_steps = per.sum(axis=1)
    ms = float(np.median(ms_steps))
    br = {"draft_ms": float(np.median(per[:, 0])), "schedule_ms": float(np.median(per[:, 1])),
          "verify_ms": float(np.median(per[:, 2])),
          "timer": "CUDA events around each call's graph replay inside the timed region; median over the steps"}
    if overlap:
        br["schedule"] = ("inside the draft call (dspark_draft_and_schedule), beside the draft kernel's last "
                          "sweep; draft_ms covers both")
    nv = B * (G + 1) if cap_accept else int(s_out["n_verify"][0])
    ms = max_over_ranks(ms, world, dev)
    code, detail = ws.read_error()
    if code != 0:
        raise RuntimeError(f"device error word {capi.dspark_status_string(code)} ({detail})")

    value = world * B * G / (ms * 1e-3)
    peak, peak_kind = load_peaks()
    bytes_ = step_bytes(wl, nv, not row_free)
    # dominant call: the draft sampler, one launch of fz::k_draft_fused (the
    # library's small-batch form fz::k_draft_narrow for B <= 16 unless
    # DSPARK_DRAFT_FORM=wide); its algorithmic bytes with W2 read once per
    # position (the method's sequential structure), and the strict count (W2
    # once per call) beside them
    draft_ms = br["draft_ms"]
    draft_gbs = bytes_["draft_per_position"] / (draft_ms * 1e-3) / 1e9
    e2e = run_e2e(args, T, capi, wl, inp, ws, dev, stream, sps_dev) if not args.no_e2e else None
    traffic, traffic_why = load_traffic(wl)
    if args.head != "markov" or row_free:
        traffic, traffic_why = None, "captured for the Markov head with p_d rows only"
    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic (seeded; DSpark workload model)",
        "config": workload_config(wl, args, inp["sched_mode"], world),
        "run": {"n_verify_rows": nv, "graph": use_graph, "ms_per_step_mean": float(np.mean(ms_steps)),
                "ms_per_step_min": float(np.min(ms_steps)), "ms_per_step_max": float(np.max(ms_steps)),
                "sched_overlap": overlap},
        "hbm_frac_step": bytes_["step_per_position"] / (ms * 1e-3) / 1e9 / peak,
        "hbm_frac_step_strict": bytes_["step_strict"] / (ms * 1e-3) / 1e9 / peak,
        "step_bytes": {"per_position": bytes_["step_per_position"], "strict": bytes_["step_strict"]},
        "breakdown_ms": br,
        "roofline": {"bound": "hbm",
                     "kernel": draft_call_label(wl, args),
                     "achieved": draft_gbs, "peak": peak, "peak_kind": f"hbm_gbs of {peak_kind}",
                     "unit": "GB/s", "frac": draft_gbs / peak,
                     "traffic": traffic,
                     **({"traffic_null_because": traffic_why} if traffic is None else {}),
                     "algorithmic_bytes": bytes_["draft_per_position"],
                     "algorithmic_bytes_strict": bytes_["draft_strict"],
                     "frac_strict": bytes_["draft_strict"] / (draft_ms * 1e-3) / 1e9 / peak},
        "gpu_launches": int(launches_per_step * args.steps),
        "launches_per_step": int(launches_per_step),
        "clocks": clk,
        "e2e": e2e,
    }
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(wl, inp, args.cpu_sample, d_out["tokens"].cpu().numpy())
    return res


def draft_kernel_name(wl):
    """The kernel that runs the draft call of a Markov-head workload."""
    small = wl.B <= 16 and os.environ.get("DSPARK_DRAFT_FORM") != "wide"
    return "fz::k_draft_narrow" if small else "fz::k_draft_fused"


def sched_overlaps(wl, args):
    """Whether the step runs the draft and the schedule as one call: where the
    library runs the scheduler beside the draft kernel's last sweep (either
    fused tensor-core form with p_d rows).
    Elsewhere the two calls stay apart, so that the draft call's time is the
    draft kernel's."""
    fused = not (args.head == "rnn" and wl.B > 512)  # both fused forms (k_draft_fused, k_draft_narrow)
    return args.sched_overlap == "on" and fused and args.rows != "none"


def draft_call_label(wl, args):
    """What the roofline's dominant call runs (the library's default dispatch)."""
    if args.head == "rnn" and wl.B > 512:
        return "dspark_draft_sample, RNN head (two-pass tensor-core passes, tensor-core recurrent step per position)"
    head = ", RNN head" if args.head == "rnn" else ""
    if sched_overlaps(wl, args):
        return f"dspark_draft_and_schedule{head} ({draft_kernel_name(wl)}, one launch, k_schedule_smem beside its last sweep)"
    return f"dspark_draft_sample{head} ({draft_kernel_name(wl)}, one launch)"


def load_traffic(wl):
    """Per-launch DRAM bytes of the dominant call from a committed ncu summary:
    (bytes, None), or (None, why) when there is no capture for this workload or
    the capture was taken on another version of the kernel's source."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(p))
        src = open(os.path.join(ROOT, d["kernel_source"]), "rb").read()
    except (ValueError, OSError, KeyError):
        return None, "no ncu traffic record"
    if hashlib.sha256(src).hexdigest() != d.get("kernel_source_sha256"):
        return None, "the ncu traffic record was captured on another version of the kernel source"
    b = d.get("per_launch_bytes", {}).get(wl.name)
    return (b, None) if b is not None else (None, "no ncu traffic record for this workload")


def draft_and_sched(T, ws, inp, U, h, anchor, temp, req_id, sps_dev, d_out, s_out, stream, rows=True,
                    n_verify_host=None):
    """dspark_draft_and_schedule in the bench's scheduler mode; returns (draft out, schedule out)."""
    return T.draft_and_schedule(ws, U, inp["W1"], inp["W2"], h, inp["w"], anchor, temp, req_id, inp["seed"],
                                inp["sts"], sps_dev, inp["sched_mode"], out=d_out, sched_out=s_out, stream=stream,
                                W_rnn=inp.get("W_rnn"), rows=rows, conf_logit_prev=inp.get("zprev"),
                                n_verify_host=n_verify_host)


def sched(T, ws, conf_logit, inp, sps_dev, anchor, tokens, **kw):
    """dspark_schedule in the bench's scheduler mode (the workload's, or the
    asynchronous production mode with synthetic earlier confidences)."""
    return T.schedule(ws, conf_logit, inp["sts"], sps_dev, anchor, tokens, inp["sched_mode"],
                      conf_logit_prev=inp.get("zprev"), **kw)


def run_e2e(args, T, capi, wl, inp, ws, dev, stream, sps_dev):
    """Same metric through the public API with HOST buffers.  Every step copies its
    inputs from pinned host memory (U, h and the per-request scalars) into one of
    two device input buffers on a copy stream, runs the draft and the scheduler
    on the compute stream once its copy is done, packs the kept target rows
    straight from the pinned host buffer by the marker tensor (dspark_pack_rows:
    only the N_v kept rows cross the host link), verifies, and reads its result
    back into pinned memory.  The copies of step i + 1 overlap the compute of
    step i, as a serving loop would run them.  With cap-accept every row is
    verified: the whole target buffer is copied as well."""
    import torch
    B, G, V = wl.B, wl.gamma, wl.V
    h_U = inp["U"].cpu().pin_memory()
    h_h = inp["h"].cpu().pin_memory()
    h_small = {k: inp[k].cpu().pin_memory() for k in ("anchor", "temp", "req_id")}
    h_tgt = inp["target"].cpu().pin_memory()  # [B, G+1, V]: the target model's rows live on the host here
    nbuf = 2
    d_U = [torch.empty_like(inp["U"]) for _ in range(nbuf)]
    d_h = [torch.empty_like(inp["h"]) for _ in range(nbuf)]
    d_small = [{k: torch.empty_like(inp[k]) for k in h_small} for _ in range(nbuf)]
    cap_accept = args.verify == "cap_accept"
    # cap-accept verifies every row: the whole target buffer moves to the device
    d_tgt = [torch.empty_like(inp["target"]) for _ in range(nbuf)] if cap_accept else None
    cap = B * (G + 1)
    rows = torch.empty((cap, V), dtype=inp["U"].dtype, device=dev)
    h_nv = [torch.empty(1, dtype=torch.int32).pin_memory() for _ in range(nbuf)]
    h_out = [torch.empty((B, G + 1), dtype=torch.int32).pin_memory() for _ in range(nbuf)]
    h_nout = [torch.empty(B, dtype=torch.int32).pin_memory() for _ in range(nbuf)]
    esz = inp["U"].element_size()
    full_offsets = (torch.arange(B + 1, device=dev, dtype=torch.int32) * (G + 1)).contiguous()
    full_ell = torch.full((B,), G, dtype=torch.int32, device=dev)
    copy_stream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event() for _ in range(nbuf)]
    consumed = [torch.cuda.Event() for _ in range(nbuf)]
    issued = [False] * nbuf

    def step(i):
        k = i % nbuf
        with torch.cuda.stream(copy_stream):
            if issued[k]:
                copy_stream.wait_event(consumed[k])  # the compute of step i - 2 is done with buffer k
            d_U[k].copy_(h_U, non_blocking=True)
            d_h[k].copy_(h_h, non_blocking=True)
            for n in h_small:
                d_small[k][n].copy_(h_small[n], non_blocking=True)
            if cap_accept:
                d_tgt[k].copy_(h_tgt, non_blocking=True)
            copied[k].record(copy_stream)
        issued[k] = True
        sm = d_small[k]
        with torch.cuda.stream(stream):
            stream.wait_event(copied[k])
            if sched_overlaps(wl, args):
                d, s = draft_and_sched(T, ws, inp, d_U[k], d_h[k], sm["anchor"], sm["temp"], sm["req_id"], sps_dev,
                                       None, None, stream, rows=args.rows != "none", n_verify_host=h_nv[k])
            else:
                d = T.draft_sample(ws, d_U[k], inp["W1"], inp["W2"], d_h[k], inp["w"], sm["anchor"], sm["temp"],
                                   sm["req_id"], inp["seed"], stream=stream, W_rnn=inp.get("W_rnn"),
                                   rows=args.rows != "none")
                s = sched(T, ws, d["conf_logit"], inp, sps_dev, sm["anchor"], d["tokens"], stream=stream,
                          n_verify_host=h_nv[k])
            rj = (dict(U=d_U[k], W1=inp["W1"], W2=inp["W2"], anchor=sm["anchor"], pd_stat=d["pd_stat"])
                  if args.rows == "none" else None)
            if cap_accept:
                v = T.verify(ws, d_tgt[k].reshape(-1, V), full_offsets, full_ell, d["tokens"], d.get("pd_rows"),
                             d["pd_tok"], sm["temp"], sm["req_id"], inp["seed"], stream=stream, commit_cap=s["ell"],
                             rejection=rj)
            else:
                # the kept rows in flattened verify order, pulled from the host
                T.pack_rows(h_tgt, s["mark_req"], s["mark_pos"], s["n_verify"], rows, ws, stream=stream)
                v = T.verify(ws, rows, s["offsets"], s["ell"], d["tokens"], d.get("pd_rows"), d["pd_tok"],
                             sm["temp"], sm["req_id"], inp["seed"], stream=stream, rejection=rj)
            h_out[k].copy_(v["out_tok"], non_blocking=True)
            h_nout[k].copy_(v["n_out"], non_blocking=True)
            consumed[k].record(stream)

    nw = max(1, min(args.warmup, 2))
    for i in range(nw):
        step(i)
    torch.cuda.synchronize(dev)
    n_e2e = max(4, min(args.steps, 16))
    t0 = time.perf_counter()
    for i in range(nw, nw + n_e2e):
        step(i)
    torch.cuda.synchronize(dev)
    t1 = time.perf_counter()
    sec = (t1 - t0) / n_e2e
    # the same steps one at a time (each synchronised before the next starts): no overlap
    ser = []
    for i in range(nw + n_e2e, nw + 2 * n_e2e):
        s0 = time.perf_counter()
        step(i)
        torch.cuda.synchronize(dev)
        ser.append(time.perf_counter() - s0)
    # the host link's own rate: one pinned-host -> device copy of U, event-timed
    lk = []
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(copy_stream):
            e0.record(copy_stream)
            d_U[0].copy_(h_U, non_blocking=True)
            e1.record(copy_stream)
        copy_stream.synchronize()
        lk.append(e0.elapsed_time(e1))
    link_gbs = h_U.numel() * h_U.element_size() / (float(np.median(lk)) * 1e-3) / 1e9
    nv_rows = float(np.mean([int(h_nv[k][0]) for k in range(nbuf)]))
    tgt_bytes = h_tgt.numel() * esz if cap_accept else nv_rows * V * esz
    h2d = (h_U.numel() * esz + h_h.numel() * esz + sum(t.numel() * t.element_size() for t in h_small.values())
           + tgt_bytes)
    d2h = 4 + h_out[0].numel() * 4 + h_nout[0].numel() * 4
    return {"value": B * G / sec, "unit": UNIT, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "steps": n_e2e, "ms_per_step": sec * 1e3, "h2d_gbs": h2d / sec / 1e9,
            "serial_ms_per_step": float(np.median(ser)) * 1e3,
            "link_gbs": link_gbs, "link_floor_ms": h2d / link_gbs / 1e6,
            "timer": "host wall clock around n pipelined steps (two input buffers; step i + 1's copies overlap "
                     "step i's compute), synchronised at both ends"}


# ---------------------------------------------------------------------------
# CPU oracle (the baseline leg and --impl reference): one worker process per
# host core, each holding a disjoint subset of the sampled requests
# ---------------------------------------------------------------------------
def host_cores() -> int:
    """Cores this process may run on (its affinity mask), else the machine's count."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def _oracle_worker(conn, shm_names, shapes, data):
    """One worker of the oracle pool: drafts and verifies its own requests, on
    command, with NumPy's BLAS pinned to one thread (set in the environment
    before this process started)."""
    from multiprocessing import shared_memory
    from oracle.draft import draft as o_draft
    from oracle import schedule as S
    from oracle.verify import verify as o_verify
    shms = [shared_memory.SharedMemory(name=n) for n in shm_names]
    W1, W2 = (np.ndarray(s, dtype=np.float64, buffer=m.buf) for s, m in zip(shapes, shms))
    d = None
    try:
        while True:
            msg = conn.recv()
            if msg[0] == "draft":
                t0 = time.perf_counter()
                d = o_draft(data["U"], W1, W2, data["h"], data["w"], data["anchor"], data["temp"], data["seed"],
                            data["req_id"], W_rnn=data.get("W_rnn"), rnn_row_dtype=data.get("rnn_row_dtype"))
                conn.send((d["conf_logit"], d["tokens"], d["margin"], time.perf_counter() - t0))
            elif msg[0] == "verify":
                t0 = time.perf_counter()
                ell = msg[1]
                fl = S.flatten(ell, data["anchor"], d["tokens"])
                rows = data["target"][fl["mark_req"], fl["mark_pos"]]
                o_verify(rows, fl["offsets"], ell, d["tokens"], d["pd"], d["pd_tok"], data["temp"], data["seed"],
                         data["req_id"])
                conn.send(time.perf_counter() - t0)
            else:
                break
    finally:
        del W1, W2
        for m in shms:
            m.close()
        conn.close()


class OraclePool:
    """The fp64 oracle over the first n_req requests of a workload, split into
    disjoint contiguous subsets, one per worker process (one process per host
    core, at most one per request).  A step drafts every subset in parallel,
    runs the scheduler on the whole batch in this process (the sampled
    requests' confidences tiled over the batch), then verifies every subset in
    parallel with the scheduler's lengths.  W1 and W2 are shared with the
    workers through shared memory; the per-request rows travel once, at start.
    Workers are started with spawn, so that a pool made after the GPU is in use
    does not fork a CUDA context."""

    def __init__(self, wl, inp, n_req, cores=None):
        import multiprocessing as mp
        from multiprocessing import shared_memory
        import torch
        self.wl, self.n_req = wl, max(1, min(n_req, wl.B))
        self.cores = max(1, min(cores or host_cores(), self.n_req))
        f = lambda x: x.detach().to("cpu", torch.float64).numpy()  # noqa: E731
        sub = slice(0, self.n_req)
        self.anchor_all = inp["anchor"].cpu().numpy().astype(np.int64)
        self.sts = inp["sts"].cpu().numpy()
        self.sps = inp["sps"]
        self.sched_mode = inp["sched_mode"]
        self.zprev = inp["zprev"].cpu().numpy() if inp.get("zprev") is not None else None
        self.shms, shapes = [], []
        for name in ("W1", "W2"):
            a = f(inp[name])
            m = shared_memory.SharedMemory(create=True, size=max(1, a.nbytes))
            np.ndarray(a.shape, dtype=np.float64, buffer=m.buf)[...] = a
            self.shms.append(m)
            shapes.append(a.shape)
            del a
        U, h, tgt = f(inp["U"][sub]), f(inp["h"][sub]), f(inp["target"][sub])
        temp = inp["temp"].cpu().numpy().astype(np.float64)
        req = inp["req_id"].cpu().numpy().astype(np.int64)
        w = f(inp["w"])
        W_rnn = f(inp["W_rnn"]) if inp.get("W_rnn") is not None else None
        self.bounds = np.linspace(0, self.n_req, self.cores + 1).round().astype(int)
        ctx = mp.get_context("spawn")
        self.conns, self.procs = [], []
        for c in range(self.cores):
            lo, hi = int(self.bounds[c]), int(self.bounds[c + 1])
            data = dict(U=U[lo:hi], h=h[lo:hi], target=tgt[lo:hi], w=w, anchor=self.anchor_all[lo:hi],
                        temp=temp[lo:hi], req_id=req[lo:hi], seed=inp["seed"], W_rnn=W_rnn,
                        rnn_row_dtype=wl.dtype if W_rnn is not None else None)
            pc, cc = ctx.Pipe()
            pr = ctx.Process(target=_oracle_worker, args=(cc, [m.name for m in self.shms], shapes, data), daemon=True)
            pr.start()
            cc.close()
            self.conns.append(pc)
            self.procs.append(pr)
        self.tokens = None

    def step(self) -> dict:
        """One oracle step over the sample; wall seconds and the parts' times."""
        from oracle import schedule as S
        B, G, n = self.wl.B, self.wl.gamma, self.n_req
        t0 = time.perf_counter()
        for c in self.conns:
            c.send(("draft",))
        res = [c.recv() for c in self.conns]
        t1 = time.perf_counter()
        zl = np.concatenate([r[0] for r in res])
        self.tokens = np.concatenate([r[1] for r in res])
        self.margin = np.concatenate([r[2] for r in res])
        tile = np.arange(B) % n
        sch = S.schedule(zl[tile].astype(np.float32), self.sts, self.sps, self.anchor_all[tile], self.tokens[tile],
                         mode=self.sched_mode, conf_logit_prev=self.zprev)
        t2 = time.perf_counter()
        for c, lo, hi in zip(self.conns, self.bounds[:-1], self.bounds[1:]):
            c.send(("verify", sch["ell"][lo:hi]))
        vt = [c.recv() for c in self.conns]
        t3 = time.perf_counter()
        return dict(step_s=t3 - t0, draft_s=t1 - t0, schedule_s=t2 - t1, verify_s=t3 - t2,
                    worker_draft_s=float(max(r[3] for r in res)), worker_verify_s=float(max(vt)))

    def close(self):
        for c in self.conns:
            try:
                c.send(("stop",))
            except (BrokenPipeError, OSError):
                pass
        for p in self.procs:
            p.join(timeout=10)
            if p.is_alive():
                p.terminate()
        for m in self.shms:
            m.close()
            m.unlink()

    def describe(self) -> str:
        return (f"fp64 oracle: draft + verify of requests 0..{self.n_req - 1} of {self.wl.B} (all "
                f"{self.wl.gamma} positions each), split over {self.cores} worker processes (one per host core, "
                f"BLAS one thread each); the scheduler on the whole batch (the sample's confidences tiled) in "
                f"the parent; value = sampled request-positions / step wall time, nothing extrapolated")


def default_oracle_requests(wl, cores: int) -> int:
    """Requests per oracle step: two per core, within the batch."""
    return max(1, min(wl.B, 2 * cores))


def cpu_baseline(wl, inp, n_req, gpu_tokens=None, steps=2):
    """The oracle on the host cores, timed on a bounded sample (one untimed
    step, then `steps` timed steps, median)."""
    cores = host_cores()
    n_req = n_req or default_oracle_requests(wl, cores)
    pool = OraclePool(wl, inp, n_req, cores)
    try:
        pool.step()
        runs = [pool.step() for _ in range(steps)]
    finally:
        pool.close()
    sec = float(np.median([r["step_s"] for r in runs]))
    res = {"value": pool.n_req * wl.gamma / sec, "unit": UNIT, "cores": pool.cores, "kind": "oracle",
           "sample": pool.describe() + f"; {steps} timed steps after one untimed, median",
           "host_cores": cores, "step_s": sec,
           "parts_s": {k: float(np.median([r[k] for r in runs])) for k in runs[0] if k != "step_s"}}
    if gpu_tokens is not None:
        # the sampled requests' draft tokens against the oracle's, position by position up
        # to the first draw inside the margin (later positions depend on that draw)
        g = np.asarray(gpu_tokens)[:pool.n_req]
        agree = {}
        for name, mg in (("margin_1e-5", 1e-5), ("margin_1e-7", 1e-7)):
            n_cmp = n_ok = 0
            for r in range(pool.n_req):
                for k in range(wl.gamma):
                    if pool.margin[r, k] < mg:
                        break
                    n_cmp += 1
                    n_ok += int(g[r, k] == pool.tokens[r, k])
            agree[name] = {"compared": n_cmp, "equal": n_ok}
        res["token_agreement"] = agree
    return res


def run_reference(args):
    """The oracle as the reference arm: every step a bounded sample of the
    workload (two requests per host core by default), all host cores."""
    import synth
    import torch
    wl = synth.get_workload(args.workload)
    inp = synth.make_inputs(wl, "cpu")
    inp["sched_mode"], inp["zprev"] = wl.sched, None
    if args.sched == "async":
        inp["sched_mode"] = synth.SCHED_ASYNC_TOPK
        inp["zprev"] = torch.from_numpy(synth.random_conf_logits(wl.B, wl.gamma, wl.seed + 77))
    if args.head == "rnn":
        inp["W_rnn"] = synth.rnn_weights(wl.r, wl.H, wl.dtype, wl.seed, "cpu")
    cores = host_cores()
    n_req = args.cpu_sample or default_oracle_requests(wl, cores)
    pool = OraclePool(wl, inp, n_req, cores)
    try:
        for _ in range(args.warmup):
            pool.step()
        t0 = time.perf_counter()
        runs = [pool.step() for _ in range(args.steps)]
        timed = time.perf_counter() - t0
    finally:
        pool.close()
    sec = float(np.median([r["step_s"] for r in runs]))
    value = pool.n_req * wl.gamma / sec
    sample = pool.describe() + f"; median of {args.steps} steps after {args.warmup} untimed"
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; DSpark workload model)",
            "config": workload_config(wl, args, inp["sched_mode"], 1),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": pool.cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "timed_region_s": timed, "requests_per_step": pool.n_req, "host_cores": cores,
            "parts_s": {k: float(np.median([r[k] for r in runs])) for k in runs[0] if k != "step_s"}}


def workload_config(wl, args, sched_mode, world) -> dict:
    """The `config` object of both arms: the workload and the modes, nothing
    that depends on the run."""
    u_mb = wl.B * wl.gamma * wl.V * (2 if wl.dtype == "bf16" else 4) / 1e6
    return {"workload": wl.name, "B": wl.B, "gamma": wl.gamma, "V": wl.V, "r": wl.r, "H": wl.H, "temp": wl.temp,
            "scheduler": {0: "off", 1: "greedy_early_stop", 2: "async_topk"}[sched_mode],
            "head": args.head, "verify": args.verify, "pd_rows": args.rows,
            "l2": (("inputs larger than L2 (U alone %.0f MB per step), no flush" if u_mb > 129 else
                    "inputs within the 129 MB L2 (U %.1f MB per step), no flush") % u_mb),
            "parallelism": "replicas" if world > 1 else "1gpu"}


# ---------------------------------------------------------------------------
# STS temperature fitting (dspark_sts_fit) on a held-out set
# ---------------------------------------------------------------------------
STS_METRIC = "STS fit (block, candidate, position) sigmoid evaluations/s"
STS_UNIT = "evaluations/s"
# fp32 arithmetic operations of one calibrated confidence c' in the fit (the
# double-float sigmoid as written: 63 for t >= 0, 67 for t < 0; the reciprocal
# counted as one)
STS_FP32_OPS_PER_EVAL = 65
# fp32 issue rate: 128 lanes per SM, 152 SMs, 2070 MHz
FP32_OPS_PEAK = 152 * 128 * 2.07e9


def sts_evals(wl) -> int:
    # every (block, candidate, position), plus the chosen candidate's products
    return wl.N * wl.gamma * wl.n_grid + wl.N * (wl.gamma - 1)


def run_sts_ours(args, rank, world, local_rank):
    import synth
    import torch
    from draft_sampling_lossless_markov_gb300 import build, capi
    from draft_sampling_lossless_markov_gb300 import torch_api as T

    build.build()
    capi.load()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = synth.STS_WORKLOADS[args.workload]
    inp = synth.sts_inputs(replace_seed(wl, wl.seed + rank))
    z = torch.from_numpy(inp["conf_logit"]).to(dev)
    L = torch.from_numpy(inp["accept_len"]).to(dev)
    grid = torch.from_numpy(inp["grid"]).to(dev)
    stream = torch.cuda.Stream(device=dev)
    ws = T.sts_fit_workspace(wl.N, wl.gamma, wl.n_grid, wl.n_bins, device=dev)
    out = dict(sts_temp=torch.empty(wl.gamma, dtype=torch.float32, device=dev),
               grid_index=torch.empty(wl.gamma, dtype=torch.int32, device=dev),
               ece=torch.empty((wl.gamma, wl.n_grid), dtype=torch.float64, device=dev))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # twice the L2

    def fit():
        T.sts_fit(ws, z, L, grid, wl.n_bins, out=out, stream=stream)

    n0 = capi.dspark_launch_count()
    with torch.cuda.stream(stream):
        fit()
    stream.synchronize()
    launches_per_fit = capi.dspark_launch_count() - n0
    for _ in range(args.warmup):
        with torch.cuda.stream(stream):
            fit()
    stream.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    cvd = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    clocks = ClockSampler(cvd[local_rank] if local_rank < len(cvd) else local_rank)
    clocks.start()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for k in range(args.steps):
        with torch.cuda.stream(stream):
            flush.fill_(k & 0xFF)  # L2 flushed between fits, outside the events
            evs[k][0].record(stream)
            fit()
            evs[k][1].record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    ms = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
    ms = max_over_ranks(ms, world, dev)
    code, detail = ws.read_error()
    if code != 0:
        raise RuntimeError(f"device error word {capi.dspark_status_string(code)} ({detail})")

    evals = sts_evals(wl)
    value = world * evals / (ms * 1e-3)
    achieved = evals * STS_FP32_OPS_PER_EVAL / (ms * 1e-3) / 1e9
    peak = FP32_OPS_PEAK / 1e9

    # end to end through the public call: pinned host inputs in, temperatures and ECE table out
    h_z = torch.from_numpy(inp["conf_logit"]).pin_memory()
    h_L = torch.from_numpy(inp["accept_len"]).pin_memory()
    h_grid = torch.from_numpy(inp["grid"]).pin_memory()
    h_temp = torch.empty(wl.gamma, dtype=torch.float32).pin_memory()
    h_ece = torch.empty((wl.gamma, wl.n_grid), dtype=torch.float64).pin_memory()
    e2e_ms = []
    for k in range(max(3, min(args.steps, 10))):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            z.copy_(h_z, non_blocking=True)
            L.copy_(h_L, non_blocking=True)
            grid.copy_(h_grid, non_blocking=True)
            fit()
            h_temp.copy_(out["sts_temp"], non_blocking=True)
            h_ece.copy_(out["ece"], non_blocking=True)
        stream.synchronize()
        e2e_ms.append((time.perf_counter() - t0) * 1e3)
    e2e_t = float(np.median(e2e_ms[1:]))
    h2d = h_z.numel() * 4 + h_L.numel() * 4 + h_grid.numel() * 4
    d2h = h_temp.numel() * 4 + h_ece.numel() * 8

    res = {
        "metric": STS_METRIC, "value": value, "unit": STS_UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic held-out blocks (seeded logistic acceptance model)",
        "config": {"workload": wl.name, "N": wl.N, "gamma": wl.gamma, "n_grid": wl.n_grid, "n_bins": wl.n_bins,
                   "l2": "flushed between fits (256 MB write outside the timed events)",
                   "parallelism": "replicas" if world > 1 else "1gpu"},
        "roofline": {"bound": "alu", "kernel": "dspark_sts_fit (k_sts_hist + k_sts_select per position)",
                     "achieved": achieved, "peak": peak,
                     "peak_kind": "fp32 issue rate from the unit counts (128 lanes x 152 SMs x 2070 MHz)",
                     "unit": "G fp32-op/s", "frac": achieved / peak, "traffic": None,
                     "algorithmic_ops": evals * STS_FP32_OPS_PER_EVAL},
        "gpu_launches": int(launches_per_fit * args.steps),
        "launches_per_step": int(launches_per_fit),
        "clocks": clk,
        "e2e": {"value": world * evals / (e2e_t * 1e-3), "unit": STS_UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "steps": len(e2e_ms) - 1,
                "timer": "host wall clock around each full fit (synchronised)"},
        "result": {"sts_temp": [float(x) for x in out["sts_temp"].cpu()],
                   "ece_best": [float(out["ece"][k, int(out["grid_index"][k])]) for k in range(wl.gamma)]},
    }
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = sts_cpu_baseline(wl, inp)
    return res


def replace_seed(wl, seed):
    from dataclasses import replace
    return replace(wl, seed=seed)


def sts_oracle_time(wl, inp) -> float:
    from oracle.sts_fit import sts_fit
    t0 = time.perf_counter()
    sts_fit(inp["conf_logit"], inp["accept_len"], inp["grid"], wl.n_bins)
    return time.perf_counter() - t0


def sts_cpu_baseline(wl, inp):
    sec = sts_oracle_time(wl, inp)
    return {"value": sts_evals(wl) / sec, "unit": STS_UNIT, "cores": 1, "kind": "oracle",
            "sample": f"the whole fit ({wl.N} blocks x {wl.n_grid} candidates x {wl.gamma} positions), "
                      "vectorised NumPy fp64, one host thread"}


def run_sts_reference(args):
    import synth
    wl = synth.STS_WORKLOADS[args.workload]
    inp = synth.sts_inputs(wl)
    for _ in range(min(args.warmup, 1)):
        sts_oracle_time(wl, inp)
    secs = [sts_oracle_time(wl, inp) for _ in range(args.steps)]
    sec = float(np.mean(secs))
    value = sts_evals(wl) / sec
    sample = (f"fp64 oracle per step: the whole fit ({wl.N} blocks x {wl.n_grid} candidates x {wl.gamma} "
              "positions), vectorised NumPy, one host thread")
    return {"impl": "reference", "metric": STS_METRIC, "value": value, "unit": STS_UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic held-out blocks (seeded logistic acceptance model)",
            "config": {"workload": wl.name, "N": wl.N, "gamma": wl.gamma, "n_grid": wl.n_grid, "n_bins": wl.n_bins},
            "cpu_baseline": {"value": value, "unit": STS_UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": STS_UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# every point of the batch/gamma sweep, then the named full-size configs
SWEEP_ALL = ([f"sweep_B{b}_g{g}" for b in (1, 8, 64, 256, 1024, 4096) for g in (4, 7, 15, 16)]
             + ["qwen3_4b", "qwen3_8b_sched", "deepseek_vocab"])


def main():
    import synth
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=synth.HEADLINE.name)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--sched", default="workload", choices=["workload", "async"],
                    help="the workload's scheduler mode, or the asynchronous production mode")
    ap.add_argument("--head", default="markov", choices=["markov", "rnn"],
                    help="the Markov head (default), or the optional RNN sequential head")
    ap.add_argument("--verify", default="compact", choices=["compact", "cap_accept"],
                    help="verify the scheduled prefixes (compact), or the full blocks committing the scheduled "
                         "windows (cap_accept)")
    ap.add_argument("--rows", default="full", choices=["full", "none"],
                    help="write the p_d rows (full), or draft without them and draw the residual by rejection "
                         "from p_t (none)")
    ap.add_argument("--sweep", default=None,
                    help="comma-separated workloads (or 'all': the batch/gamma sweep and the named configs): one "
                         "JSON line per workload, device-timed only (no end-to-end leg, no oracle baseline)")
    ap.add_argument("--sched-overlap", default="on", choices=["on", "off"],
                    help="on: where the scheduler can run beside the draft kernel's last sweep, the step's draft "
                         "and schedule are one dspark_draft_and_schedule call; off: always two calls")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample", type=int, default=0,
                    help="requests the oracle runs per step (default: two per host core)")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    sts = args.workload in synth.STS_WORKLOADS
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_sts_reference(args) if sts else run_reference(args)), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    if args.sweep:
        import torch
        names = (SWEEP_ALL if args.sweep == "all" else args.sweep.split(","))
        args.no_e2e = args.no_cpu_baseline = True
        for name in names:
            args.workload = name
            res = run_ours(args, rank, world, local_rank)
            if rank == 0:
                print(json.dumps(res), flush=True)
            torch.cuda.empty_cache()
    else:
        res = run_sts_ours(args, rank, world, local_rank) if sts else run_ours(args, rank, world, local_rank)
        if rank == 0:
            print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
