"""CPU checks of bench.py's host-side helpers: the DRAM-traffic record is used only while it was
measured on the current GEMV source, and the host facts the CPU baseline reports."""

import hashlib
import json

import bench


def _record(tmp_path, source_bytes, sha=None):
    src = tmp_path / "lb_gemv.cu"
    src.write_bytes(source_bytes)
    rec = tmp_path / "gemv_traffic.json"
    rec.write_text(json.dumps({"gemv_source_sha256": sha or hashlib.sha256(source_bytes).hexdigest(),
                               "dram_bytes_per_launch": 1234, "basis": "test capture"}))
    return src, rec


def test_traffic_used_while_the_source_matches(tmp_path, monkeypatch):
    src, rec = _record(tmp_path, b"kernel v1")
    monkeypatch.setattr(bench, "GEMV_SOURCE", str(src))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(rec))
    assert bench._traffic_per_launch() == (1234, "test capture")


def test_traffic_dropped_once_the_source_changes(tmp_path, monkeypatch):
    src, rec = _record(tmp_path, b"kernel v1")
    src.write_bytes(b"kernel v2")
    monkeypatch.setattr(bench, "GEMV_SOURCE", str(src))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(rec))
    value, why = bench._traffic_per_launch()
    assert value is None and "changed" in why


def test_traffic_without_a_record(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "missing.json"))
    value, why = bench._traffic_per_launch()
    assert value is None and why


def test_committed_record_is_well_formed():
    rec = json.load(open(bench.TRAFFIC_FILE))
    assert len(rec["gemv_source_sha256"]) == 64
    assert len(rec["per_launch_bytes"]) == 4                      # q, o, [gate, up], down
    assert rec["dram_bytes_per_launch"] == round(sum(rec["per_launch_bytes"]) / 4)


def test_host_facts():
    assert bench.host_cores() >= 1
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()
