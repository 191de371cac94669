"""bench.py's `traffic` figures come from committed ncu records keyed by the
hash of the kernel sources they were taken on (CPU). A record is used only
while the sources hash the same; every committed record is well formed
(read + write = the bytes reported) and names the capture that made it."""
import json
import os

import pytest

import bench


def _records():
    out = []
    for kind, (fname, files) in bench.TRAFFIC_RECORDS.items():
        path = os.path.join(bench.ROOT, "profiles", fname)
        if os.path.exists(path):
            with open(path) as f:
                for key, entry in json.load(f).items():
                    out.append((kind, key, entry))
    return out


@pytest.mark.parametrize("kind,key,entry", _records(), ids=lambda x: x if isinstance(x, str) else "")
def test_committed_records_are_well_formed(kind, key, entry):
    total = entry.get("bytes_per_launch", entry.get("bytes_per_step"))
    assert total == entry["dram_bytes_read"] + entry["dram_bytes_write"]
    assert len(entry["source_sha1"]) == 40
    cap = entry["capture"]
    assert cap.startswith("ncu ") and "--clock-control none" in cap and "python bench.py" in cap


def test_record_used_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    files = ("relayout.cu",)
    sha = bench.kernel_source_sha1(files)
    (tmp_path / "profiles").mkdir()
    rec = {"same": {"source_sha1": sha, "bytes_per_step": 30, "dram_bytes_read": 20, "dram_bytes_write": 10},
           "other": {"source_sha1": "0" * 40, "bytes_per_step": 30, "dram_bytes_read": 20, "dram_bytes_write": 10}}
    (tmp_path / "profiles" / "t.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setitem(bench.TRAFFIC_RECORDS, "probe", ("t.json", files))
    # the sources are read from the package, not from ROOT: hash them where they are
    monkeypatch.setattr(bench, "kernel_source_sha1", lambda f: sha)
    assert bench.recorded_traffic("same", "probe") == 30
    assert bench.recorded_traffic("other", "probe") is None
    assert bench.recorded_traffic("missing", "probe") is None


def test_source_hash_follows_the_kernel_text():
    a = bench.kernel_source_sha1(("relayout.cu",))
    b = bench.kernel_source_sha1(("relayout.cu", "merge.cu"))
    assert a != b and len(a) == 40
    assert a == bench.kernel_source_sha1(("relayout.cu",))
