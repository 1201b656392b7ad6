"""The benchmark's DRAM-traffic figures come from committed ncu counters that
are locked to the kernel sources they were taken on (host logic, no GPU)."""
import json
import os
import shutil

import bench


def test_every_workload_names_recorded_kernels():
    with open(os.path.join(bench.ROOT, "profiles", "counters.json")) as f:
        recs = json.load(f)
    keys = [k for ks in bench.TRAFFIC_KEYS.values() for k in ks] + ["w4a16_dequant_kernel"]
    for key in keys:
        rec = recs[key]
        assert rec["dram_read_bytes"] > 0 and rec["dram_write_bytes"] >= 0
        assert rec["command"].startswith("ncu ") and "--clock-control none" in rec["command"]
        for src in rec["sources"]:
            assert os.path.isfile(os.path.join(bench.ROOT, "paged_kv_cache_241_gb300", src)), src


def test_traffic_is_withheld_once_a_source_changes(tmp_path, monkeypatch):
    # A copy of the tree with the counters and the sources they name.
    root = tmp_path / "repo"
    shutil.copytree(os.path.join(bench.ROOT, "profiles"), root / "profiles")
    shutil.copytree(os.path.join(bench.ROOT, "paged_kv_cache_241_gb300", "csrc"),
                    root / "paged_kv_cache_241_gb300" / "csrc")
    monkeypatch.setattr(bench, "ROOT", str(root))
    key = "w4a16_dequant_kernel"
    with open(root / "profiles" / "counters.json") as f:
        rec = json.load(f)[key]
    before = bench.ncu_traffic(key)
    if before is not None:  # counters taken on these very sources
        assert before == rec["dram_read_bytes"] + rec["dram_write_bytes"]
    src = root / "paged_kv_cache_241_gb300" / rec["sources"][0]
    src.write_text(src.read_text() + "\n// edited\n")
    assert bench.ncu_traffic(key) is None
    assert bench.ncu_traffic("no_such_kernel") is None
