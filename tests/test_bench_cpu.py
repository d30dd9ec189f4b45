"""bench.py's bookkeeping that needs no GPU: the DRAM traffic it reports comes
from the committed ncu figures only while the kernel sources still hash to
the captured ones, and it is the slope of two captures of different sizes
(DRAM bytes per algorithmic byte) times the launch's algorithmic bytes; the
reference arm reports the same workload config as the GPU arm; the oracle's
OpenMP build that the CPU baseline times computes what the plain build does."""
import json
import os
import shutil

import bench


def _entry(kernel):
    with open(bench.TRAFFIC_FILE) as f:
        return json.load(f)["kernels"][kernel]


def test_committed_traffic_matches_the_current_sources():
    for kernel in ("a2a_runs_kernel", "a2a_pc_rel_kernel"):
        e = _entry(kernel)
        assert e["sources_hash"] == bench._kernel_sources_hash(e["sources"]), kernel
        (a0, d0), (a1, d1) = [(c["algorithmic_bytes"], c["dram_bytes"]) for c in e["captures"]]
        assert a1 > a0
        # the difference of the two captures is one slope's worth of its bytes
        assert abs(bench._traffic(kernel, a1 - a0) - (d1 - d0)) <= 1
        # a launch twice as large moves twice the bytes
        t = bench._traffic(kernel, 10**9)
        assert abs(bench._traffic(kernel, 2 * 10**9) - 2 * t) <= 1
        # a copy reads and writes every byte at least once: at least the algorithmic bytes
        assert t >= 0.98 * 10**9


def test_traffic_is_withheld_once_a_source_changes(tmp_path, monkeypatch):
    csrc = os.path.join(bench.ROOT, "symmetric_memory_moe_gb300", "csrc")
    fake_root = tmp_path / "root"
    shutil.copytree(csrc, fake_root / "symmetric_memory_moe_gb300" / "csrc")
    prof = fake_root / "profiles"
    prof.mkdir()
    shutil.copy(bench.TRAFFIC_FILE, prof / "traffic.json")
    monkeypatch.setattr(bench, "ROOT", str(fake_root))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(prof / "traffic.json"))
    assert bench._traffic("a2a_runs_kernel", 10**9) is not None
    with open(fake_root / "symmetric_memory_moe_gb300" / "csrc" / "a2a.cu", "a") as f:
        f.write("\n// edited\n")
    assert bench._traffic("a2a_runs_kernel", 10**9) is None
    assert bench._traffic("no_such_kernel", 1) is None


def test_both_arms_report_one_config():
    for variant in ("direct", "pc"):
        c = bench.bench_config(1, variant)
        assert c == bench.bench_config(1, variant)
        assert (c["W"], c["S"], c["H"], c["D"]) == (8, 2048, 1, 7168)
        assert c["bytes_per_step"] == 2 * 8 * 2048 * 8 * 7168 * 2


def test_openmp_oracle_build_matches_the_plain_build(monkeypatch):
    """The CPU baseline times the oracle's OpenMP build (its loops over
    destination and row split across threads): it must compute the same
    combine as the plain build, also with more threads than destinations."""
    import numpy as np

    import oracle

    monkeypatch.setenv("OMP_NUM_THREADS", "5")
    x = np.random.default_rng(3).integers(-2**15, 2**15, (4, 4 * 13, 3, 7), dtype=np.int16)
    want = oracle.load().combine(x, 4, 13, 3, 7)
    assert np.array_equal(oracle.load_openmp().combine(x, 4, 13, 3, 7), want)
