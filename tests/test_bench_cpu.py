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
