"""The N > 1 path on the CPU: two gloo ranks.

The hot path shards by request: draft sampling and verification are
independent per request (their random numbers are keyed by the global
request id), and the only step that needs every request is the scheduler's
sort, whose inputs a multi-rank run all-gathers (B gamma fp32 confidences).
These tests run that sharded step with the oracle on two gloo ranks and
compare it with the single-process step, check the bench's max-over-ranks
timing, and check that the reference arm prints on rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _oracle_step(inp, sl, conf_all=None):
    """Draft and verify the requests in slice sl; the scheduler sees every
    request's confidences (conf_all, else the slice's own)."""
    sys.path.insert(0, ROOT)
    from oracle.draft import draft
    from oracle import schedule as S
    from oracle.verify import verify
    f = lambda t: t.detach().to(torch.float64).numpy()  # noqa: E731
    d = draft(f(inp["U"][sl]), f(inp["W1"]), f(inp["W2"]), f(inp["h"][sl]), f(inp["w"]),
              inp["anchor"][sl].numpy(), inp["temp"][sl].numpy(), inp["seed"], inp["req_id"][sl].numpy())
    z = d["conf_logit"].astype(np.float32) if conf_all is None else conf_all(d["conf_logit"].astype(np.float32))
    sch = S.schedule(z, inp["sts"].numpy(), inp["sps"], np.zeros(z.shape[0], np.int64),
                     np.zeros(z.shape, np.int64), mode=inp["sched"])
    ell = sch["ell"][sl] if conf_all is not None else sch["ell"]
    fl = S.flatten(ell, inp["anchor"][sl].numpy(), d["tokens"])
    rows = f(inp["target"][sl])[fl["mark_req"], fl["mark_pos"]]
    v = verify(rows, fl["offsets"], ell, d["tokens"], d["pd"], d["pd_tok"], inp["temp"][sl].numpy(), inp["seed"],
               inp["req_id"][sl].numpy())
    return dict(tokens=d["tokens"], pd_tok=d["pd_tok"], margin=d["margin"], ell=ell, n_accept=v["n_accept"],
                out_tok=v["out_tok"])


def _sharded_worker(rank, world, port, q):
    try:
        sys.path.insert(0, ROOT)
        import synth
        _init(rank, world, port)
        wl = synth.WORKLOADS["tiny"]
        inp = synth.make_inputs(wl, "cpu")
        per = wl.B // world
        sl = slice(rank * per, (rank + 1) * per)

        def gather_conf(z_local):
            parts = [torch.empty_like(torch.from_numpy(z_local)) for _ in range(world)]
            dist.all_gather(parts, torch.from_numpy(z_local))
            return torch.cat(parts).numpy()

        out = _oracle_step(inp, sl, gather_conf)
        gathered = [None] * world
        dist.all_gather_object(gathered, out)
        if rank == 0:
            full = _oracle_step(inp, slice(0, wl.B))
            merged = {k: np.concatenate([g[k] for g in gathered]) for k in out}
            ok = (full["margin"] >= 1e-12).all(axis=1)  # batch composition may move BLAS rounding
            assert ok.sum() >= wl.B // 2
            for k in ("tokens", "ell", "n_accept", "out_tok"):
                np.testing.assert_array_equal(merged[k][ok], full[k][ok], err_msg=k)
            np.testing.assert_allclose(merged["pd_tok"][ok], full["pd_tok"][ok], rtol=1e-12)
        dist.barrier()
        dist.destroy_process_group()
        q.put((rank, "ok"))
    except BaseException as e:  # noqa: BLE001
        q.put((rank, f"{type(e).__name__}: {e}"))


def _timing_worker(rank, world, port, q):
    try:
        sys.path.insert(0, ROOT)
        sys.argv = ["bench.py"]
        import bench
        _init(rank, world, port)
        ms = bench.max_over_ranks(1.5 + rank, world, "cpu")
        dist.destroy_process_group()
        q.put((rank, ms))
    except BaseException as e:  # noqa: BLE001
        q.put((rank, f"{type(e).__name__}: {e}"))


def _run(worker, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=300) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
    return res


def test_request_sharded_step_matches_the_single_process_step():
    res = _run(_sharded_worker)
    assert res == {0: "ok", 1: "ok"}, res


def test_bench_takes_the_slowest_rank():
    res = _run(_timing_worker)
    assert res == {0: 2.5, 1: 2.5}, res


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_prints_on_rank_zero_only(rank):
    env = {**os.environ, "RANK": str(rank), "WORLD_SIZE": "2", "LOCAL_RANK": str(rank)}
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "1",
                          "--warmup", "0", "--cpu-sample", "2"], cwd=ROOT, env=env, capture_output=True, text=True,
                         timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.strip()]
    if rank == 0:
        assert len(lines) == 1 and json.loads(lines[0])["impl"] == "reference"
    else:
        assert lines == []
