"""Host-side pieces of bench.py that need no GPU: the roofline traffic
record is used only while the kernel sources still match the capture."""
import json
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_traffic_record_matches_the_committed_sources():
    rec = json.load(open(os.path.join(ROOT, "profiles", "roofline_traffic.json")))["gate_up_q4"]
    assert rec["traffic_bytes"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
    assert bench.roofline_traffic("gate_up_q4") == rec["traffic_bytes"]
    # traffic well above the algorithmic bytes would mean re-reads
    assert rec["traffic_bytes"] < 1.05 * 56_688_640


def test_traffic_is_null_once_a_source_changes(tmp_path, monkeypatch):
    rec = json.load(open(os.path.join(ROOT, "profiles", "roofline_traffic.json")))["gate_up_q4"]
    fake = tmp_path / "repo"
    for rel in rec["sources"] + ["profiles/roofline_traffic.json"]:
        dst = fake / rel
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(os.path.join(ROOT, rel), dst)
    monkeypatch.setattr(bench, "ROOT", str(fake))
    assert bench.roofline_traffic("gate_up_q4") == rec["traffic_bytes"]
    src = fake / rec["sources"][0]
    src.write_text(src.read_text() + "\n// changed\n")
    assert bench.roofline_traffic("gate_up_q4") is None
    assert bench.roofline_traffic("no_such_kernel") is None
