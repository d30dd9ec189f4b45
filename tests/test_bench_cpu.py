"""bench.py's bookkeeping that needs no GPU: the DRAM traffic it reports comes
from the committed ncu figures only while the kernel sources still hash to
the captured ones, and it is scaled to a launch by the algorithmic bytes."""
import json
import os
import shutil

import bench


def _entry(kernel):
    with open(bench.TRAFFIC_FILE) as f:
        return json.load(f)["kernels"][kernel]


def test_committed_traffic_matches_the_current_sources():
    for kernel in ("a2a_runs_kernel", "a2a_pc_kernel"):
        e = _entry(kernel)
        assert e["sources_hash"] == bench._kernel_sources_hash(e["sources"]), kernel
        # one captured launch scales to itself, a launch twice as large to twice the bytes
        assert bench._traffic(kernel, e["algorithmic_bytes"]) == e["dram_bytes"]
        assert bench._traffic(kernel, 2 * e["algorithmic_bytes"]) == 2 * e["dram_bytes"]


def test_traffic_is_withheld_once_a_source_changes(tmp_path, monkeypatch):
    csrc = os.path.join(bench.ROOT, "symmetric_memory_moe_gb300", "csrc")
    fake_root = tmp_path / "root"
    shutil.copytree(csrc, fake_root / "symmetric_memory_moe_gb300" / "csrc")
    prof = fake_root / "profiles"
    prof.mkdir()
    shutil.copy(bench.TRAFFIC_FILE, prof / "traffic.json")
    monkeypatch.setattr(bench, "ROOT", str(fake_root))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(prof / "traffic.json"))
    e = _entry("a2a_runs_kernel")
    assert bench._traffic("a2a_runs_kernel", e["algorithmic_bytes"]) == e["dram_bytes"]
    with open(fake_root / "symmetric_memory_moe_gb300" / "csrc" / "a2a.cu", "a") as f:
        f.write("\n// edited\n")
    assert bench._traffic("a2a_runs_kernel", e["algorithmic_bytes"]) is None
    assert bench._traffic("no_such_kernel", 1) is None
