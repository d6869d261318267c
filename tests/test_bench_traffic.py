"""bench.py reports a kernel's ncu DRAM traffic only while the kernel's sources
hash as they did when the counters were taken (CPU only)."""
import json
import os
import shutil

import bench


def _write_traffic(root, entries):
    os.makedirs(os.path.join(root, "profiles"), exist_ok=True)
    with open(os.path.join(root, "profiles", "ncu_traffic.json"), "w") as f:
        json.dump(entries, f)


def test_traffic_only_while_sources_match(tmp_path, monkeypatch):
    _write_traffic(str(tmp_path), {"fa_fwd_kernel": {"w": {"dram_bytes_per_launch": 123, "source_hash": "abc"}}})
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: "abc")
    assert bench.ncu_traffic("fa_fwd_kernel", "w") == 123.0
    assert bench.ncu_traffic("fa_fwd_kernel", "another_workload") is None
    assert bench.ncu_traffic("fa_bwd_dkdv_kernel", "w") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: "changed")
    assert bench.ncu_traffic("fa_fwd_kernel", "w") is None


def test_missing_traffic_table_gives_none(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: "abc")
    assert bench.ncu_traffic("fa_fwd_kernel", "w") is None


def test_source_hash_follows_every_listed_file(tmp_path, monkeypatch):
    src = os.path.join(os.path.dirname(bench.__file__), "exact_io_aware_flashattention_gb300", "csrc")
    dst = tmp_path / "exact_io_aware_flashattention_gb300" / "csrc"
    shutil.copytree(src, dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    for kernel, files in bench.KERNEL_SOURCES.items():
        assert any(f.endswith(".cu") for f in files), kernel
        before = bench.kernel_source_hash(kernel)
        for name in files:
            p = dst / name
            text = p.read_bytes()
            p.write_bytes(text + b"\n")
            assert bench.kernel_source_hash(kernel) != before, (kernel, name)
            p.write_bytes(text)
        assert bench.kernel_source_hash(kernel) == before


def test_committed_traffic_entries_name_their_summary():
    with open(os.path.join(os.path.dirname(bench.__file__), "profiles", "ncu_traffic.json")) as f:
        table = json.load(f)
    root = os.path.dirname(bench.__file__)
    for kernel, per_workload in table.items():
        assert kernel in bench.KERNEL_SOURCES
        for workload, e in per_workload.items():
            assert e["dram_bytes_per_launch"] > 0
            assert len(e["source_hash"]) == 16
            assert os.path.exists(os.path.join(root, e["from"])), e["from"]
