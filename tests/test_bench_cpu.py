"""Host logic of the benchmark that decides which evidence a bench line may
carry: the kernel-source hash (a comment-only edit keeps it, a code edit
changes it) and the DRAM-traffic lookup (only a capture taken on the current
kernel source is reported; anything else gives null)."""
import json
import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_only_ignores_comments_and_layout():
    a = "int x = 1; // one\n/* block\n comment */ int   y=2;\n"
    b = "int x = 1;\nint y=2;"
    assert bench._code_only(a) == bench._code_only(b) == "int x = 1; int y=2;"
    assert bench._code_only("a /* x */ b") == "a b"
    assert bench._code_only("a // x\nb") == "a b"


@pytest.fixture
def source_copy(tmp_path, monkeypatch):
    """A copy of the hashed kernel sources under a temporary root."""
    for f in bench.KERNEL_SOURCES:
        dst = tmp_path / f
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(os.path.join(ROOT, f), dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def test_kernel_sha_keeps_comment_edits_and_tracks_code_edits(source_copy):
    base = bench.kernel_sha()
    assert len(base) == 16 and int(base, 16) >= 0
    f = source_copy / bench.KERNEL_SOURCES[0]
    text = f.read_text(encoding="utf-8")
    f.write_text("// a new comment line\n" + text.replace("\n", "\n   ", 3), encoding="utf-8")
    assert bench.kernel_sha() == base
    f.write_text(text + "\nstatic int ra_hash_probe = 0;\n", encoding="utf-8")
    assert bench.kernel_sha() != base


def test_traffic_is_reported_only_for_the_current_source(tmp_path, monkeypatch):
    path = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(path))
    assert bench.traffic_for("gqa_s16384") is None  # no file
    path.write_text("not json")
    assert bench.traffic_for("gqa_s16384") is None
    entry = {"kernel_sha": bench.kernel_sha(), "dram_bytes_per_launch": 123}
    path.write_text(json.dumps({"gqa_s16384": entry}))
    assert bench.traffic_for("gqa_s16384") == 123
    assert bench.traffic_for("long_s65536") is None  # another workload
    entry["kernel_sha"] = "0" * 16
    path.write_text(json.dumps({"gqa_s16384": entry}))
    assert bench.traffic_for("gqa_s16384") is None  # captured on other code


def test_committed_traffic_record_names_its_source():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    for name, e in d.items():
        assert len(e["kernel_sha"]) == 16
        assert e["dram_bytes_per_launch"] == e["dram_bytes_read"] + e["dram_bytes_write"]
        assert os.path.exists(os.path.join(ROOT, e["source"]))
