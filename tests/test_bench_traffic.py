"""bench.py's DRAM-traffic bookkeeping on CPU: the committed capture is used
only while the captured kernel's own source files are unchanged."""
import json
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _copy_tree(tmp_path):
    src = os.path.join(ROOT, "block_scaled_fp4_softmax_gb300", "csrc")
    dst = tmp_path / "block_scaled_fp4_softmax_gb300" / "csrc"
    shutil.copytree(src, dst)
    shutil.copytree(os.path.join(ROOT, "profiles"), tmp_path / "profiles")
    return dst


def test_hashed_files_exist_and_match_the_record():
    d = os.path.join(ROOT, "block_scaled_fp4_softmax_gb300", "csrc")
    for n in bench.ONESHOT_SOURCES:
        assert os.path.isfile(os.path.join(d, n)), n
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))["moe_decode_layer"]
    assert [os.path.basename(p) for p in rec["hashed_files"]] == list(bench.ONESHOT_SOURCES)
    assert rec["bytes_per_launch"] > 0


def test_capture_used_only_while_its_kernel_sources_are_unchanged(tmp_path, monkeypatch):
    csrc = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # record the copy's own hash, as a fresh capture would
    p = tmp_path / "profiles" / "traffic.json"
    rec = json.load(open(p))
    rec["moe_decode_layer"]["sources"] = bench._hash_sources()
    p.write_text(json.dumps(rec))
    want = rec["moe_decode_layer"]["bytes_per_launch"]
    assert bench._traffic_from_profiles("moe_decode_layer") == want
    # a file of another kernel changes: the capture still stands
    with open(csrc / "grouped.cu", "a") as f:
        f.write("\n// edit\n")
    assert bench._traffic_from_profiles("moe_decode_layer") == want
    # a file the captured kernel is built from changes: no traffic figure
    with open(csrc / "decode_oneshot.cu", "a") as f:
        f.write("\n// edit\n")
    assert bench._traffic_from_profiles("moe_decode_layer") is None
