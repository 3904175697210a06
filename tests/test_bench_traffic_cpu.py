"""bench.py's committed DRAM counts: each entry names its kernel's source files and the hash
they had when ncu took the counts; a count is reported only while that hash still holds."""
from __future__ import annotations

import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_every_traffic_entry_names_its_kernel_files_and_summary():
    d = json.load(open(os.path.join(ROOT, "profiles", "dram_traffic.json")))
    assert d, "no committed DRAM counts"
    for name, e in d.items():
        assert e["kernel_files"] in bench.KERNEL_FILES, name
        assert e["traffic_bytes_per_launch"] == e["dram_bytes_read"] + e["dram_bytes_write"], name
        assert os.path.exists(os.path.join(ROOT, e["summary"])), name


def test_a_count_is_reported_only_for_unchanged_kernel_sources(tmp_path, monkeypatch):
    files = bench.KERNEL_FILES["decode"]
    good = bench.kernel_source_hash(files)
    prof = tmp_path / "profiles"
    prof.mkdir()
    entry = {"kernel_files": "decode", "kernel_source_hash": good, "dram_bytes_read": 5, "dram_bytes_write": 7,
             "traffic_bytes_per_launch": 12, "summary": "x"}
    (prof / "dram_traffic.json").write_text(json.dumps({"w": entry, "stale": dict(entry, kernel_source_hash="0" * 16),
                                                        "unnamed": dict(entry, kernel_files="nope")}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # kernel_source_hash reads the sources under ROOT: point it back at the repository's
    real = bench.kernel_source_hash
    monkeypatch.setattr(bench, "kernel_source_hash", lambda f=None: good if f == files else real(f))
    assert bench.measured_traffic("w") == 12
    assert bench.measured_traffic("stale") is None
    assert bench.measured_traffic("unnamed") is None
    assert bench.measured_traffic("missing") is None


def test_the_source_hash_ignores_comments_but_not_code():
    a = 'int f() { return 1; }  // one\n/* block\n */\nconst char* s = "x//y";\n'
    b = '// header\nint f() { return 1; }\n\nconst char* s = "x//y";   /* trailing */\n'
    c = 'int f() { return 2; }\nconst char* s = "x//y";\n'
    assert bench.strip_comments(a) == bench.strip_comments(b)
    assert bench.strip_comments(a) != bench.strip_comments(c)
    assert '"x//y"' in bench.strip_comments(a)
