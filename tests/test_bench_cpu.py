"""bench.py host logic: the ncu traffic figure is reported only for the kernel
source it was captured on."""
import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(monkeypatch, root):
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setattr(bench, "ROOT", str(root))
    return bench


class _Wl:
    name = "sweep_B256_g7"


def _layout(tmp_path, src: bytes, recorded: bytes):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "k.cu").write_bytes(src)
    rec = {"kernel_source": "k.cu", "kernel_source_sha256": hashlib.sha256(recorded).hexdigest(),
           "per_launch_bytes": {"sweep_B256_g7": 123.0}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))


def test_traffic_reported_for_the_captured_source(tmp_path, monkeypatch):
    _layout(tmp_path, b"kernel v1", b"kernel v1")
    b = _bench(monkeypatch, tmp_path)
    assert b.load_traffic(_Wl()) == (123.0, None)


def test_traffic_null_once_the_source_changed(tmp_path, monkeypatch):
    _layout(tmp_path, b"kernel v2", b"kernel v1")
    b = _bench(monkeypatch, tmp_path)
    t, why = b.load_traffic(_Wl())
    assert t is None and "another version" in why


def test_traffic_null_without_a_record(tmp_path, monkeypatch):
    b = _bench(monkeypatch, tmp_path)
    assert b.load_traffic(_Wl())[0] is None


def test_oracle_pool_splits_requests_without_changing_results(monkeypatch):
    # the baseline's worker processes each draft a disjoint subset of the sampled
    # requests; put together, their tokens are the single-process oracle's
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    import synth
    from oracle.draft import draft as o_draft
    wl = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(wl, "cpu")
    inp["sched_mode"], inp["zprev"] = wl.sched, None
    pool = bench.OraclePool(wl, inp, wl.B, cores=3)
    try:
        st = pool.step()
        toks = pool.tokens.copy()
    finally:
        pool.close()
    assert pool.cores == 3 and st["step_s"] > 0
    f = lambda t: t.double().numpy()  # noqa: E731
    o = o_draft(f(inp["U"]), f(inp["W1"]), f(inp["W2"]), f(inp["h"]), f(inp["w"]), inp["anchor"].numpy(),
                inp["temp"].numpy(), inp["seed"], inp["req_id"].numpy())
    np.testing.assert_array_equal(toks, o["tokens"])


def test_reference_arm_reports_what_it_ran(tmp_path):
    # the reference line: steps and warm-up as run, the same config keys as the GPU
    # arm, and a step time that is the measured one (no extrapolation)
    import subprocess
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "3",
                          "--warmup", "2"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr
    d = json.loads(res.stdout.strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["steps"] == 3 and d["warmup"] == 2
    assert d["cpu_baseline"]["cores"] >= 1
    assert abs(d["value"] - d["requests_per_step"] * 4 / (d["ms_per_step"] * 1e-3)) < 1e-6 * d["value"]
    assert d["timed_region_s"] >= 0.5 * 3 * d["ms_per_step"] * 1e-3
    sys.path.insert(0, ROOT)
    import bench
    import synth

    class A:
        head, verify, rows = "markov", "compact", "full"
    assert set(d["config"]) == set(bench.workload_config(synth.WORKLOADS["tiny"], A, 1, 1))
