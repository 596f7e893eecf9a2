"""Host logic of bench.py that decides which evidence a bench line carries:
the DRAM traffic of a committed ncu capture is reported only while the
kernel sources still hash to the recorded value, and the roofline peaks come
from the measured file when it exists."""
import hashlib
import json
import os
import shutil

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join("quantized_sparse_moe_gb300", "csrc")


def _copy_tree(tmp_path):
    shutil.copytree(os.path.join(ROOT, "profiles"), tmp_path / "profiles")
    shutil.copytree(os.path.join(ROOT, CSRC), tmp_path / CSRC)
    return tmp_path / "profiles" / "ffn_dram_traffic.json"


def _sha(tmp_path, sources):
    m = hashlib.sha256()
    for f in sources:
        m.update((tmp_path / CSRC / f).read_bytes())
    return m.hexdigest()


def test_traffic_reported_only_for_the_captured_sources(tmp_path, monkeypatch):
    rec = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    table = json.loads(rec.read_text())
    names = [n for n in table if n != "about"]
    assert names, "no capture entries"
    for name in names:
        ent = table[name]
        # the record matches the sources: the capture's bytes are reported
        ent["sources_sha256"] = _sha(tmp_path, ent["sources"])
        rec.write_text(json.dumps(table))
        assert bench.measured_traffic(name) == ent["bytes_per_launch"]
    for name in names:
        # any change to one of the listed sources makes the capture stale
        src = tmp_path / CSRC / table[name]["sources"][0]
        keep = src.read_bytes()
        src.write_bytes(keep + b"\n// changed\n")
        assert bench.measured_traffic(name) is None
        src.write_bytes(keep)
        assert bench.measured_traffic(name) == table[name]["bytes_per_launch"]
    assert bench.measured_traffic("no_such_workload") is None


def test_peaks_measured_or_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.peaks() == (6800.0, 1900.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(
        json.dumps({"hbm_gbs": 6792.4, "bf16_tflops": 1898.5}))
    assert bench.peaks() == (6792.4, 1898.5, "measured")
